// ring_attend_static: the attention of ring_attend for callers that cannot allocate.
//
// Some callers of this library cannot call cudaMalloc at all -- code that runs under a
// host framework that owns every device allocation, or inside a region (a memory-budgeted
// service, a stream that is being captured) where a runtime allocation is not allowed.
// They hold the ring's buffers themselves and need the attention step without a ring
// handle, whose creation allocates.  This entry point takes every input and output from
// the caller and keeps its own scratch (per-tile flags and visibility bits, the RoPE table
// of the noise positions, split partials for the combine pass) in one fixed file-scope
// device array, so it allocates nothing.  The computation is the one ring_attend launches:
// the same attention and combine kernels run, pointed at this scratch.
#include "dflash_ring.h"
#include "ring_internal.h"

#include <algorithm>
#include <cstdarg>
#include <cmath>
#include <cstdio>
#include <mutex>

namespace dflash {
namespace {

// Scratch of ring_attend_static, shared by every call on a device.  Every GPU that loads
// the library holds it until the process exits.
constexpr size_t kStaticScratchBytes = 16u << 20;   // 16 MiB
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxStaticSeqs = 256;
constexpr int kMaxDevices = 64;

struct StaticParams {
    int64_t committed[kMaxStaticSeqs];
    double inv_freq[kHeadDim / 2];
};

std::mutex g_setup_mu;
void *g_scratch_addr[kMaxDevices] = {};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Tile flags, per-row visibility bits and the RoPE table, from the caller's F32 mask and
// committed counts.  Grid (n_tiles + 1, n_seq), 128 threads: block t < n_tiles handles tile
// t (threads 0-63 one slot each), the last block the cos/sin of committed + i.
__global__ void __launch_bounds__(128)
k_static_prepare(RingDims d, RingDev m, const float *__restrict__ mask, StaticParams prm) {
    const int b = blockIdx.x, s = blockIdx.y;
    const int half = d.head_dim / 2;
    if (b == d.n_tiles) {
        for (int idx = threadIdx.x; idx < d.q_len * half; idx += blockDim.x) {
            const int i = idx / half, j = idx - i * half;
            m.rope32[((int64_t)s * d.q_len + i) * half + j] =
                rope_angle_cs(prm.committed[s] + i, prm.inv_freq[j]);
        }
        return;
    }
    const int slot = b * kTile + (int)threadIdx.x;
    const bool active = threadIdx.x < kTile;
    const bool in_range = active && slot < d.kv_total;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qw = (d.q_len + 1) & ~1;
    const int64_t fi = (int64_t)s * d.n_tiles + b;
    uint32_t *bits = reinterpret_cast<uint32_t *>(m.maskbits + fi * qw);
    bool all_rows = true, any_row = false;
    for (int i = 0; i < qw; ++i) {
        bool vis = false;
        if (in_range && i < d.q_len)
            vis = mask[((int64_t)s * d.q_len + i) * d.kv_total + slot] == 0.f;
        if (warp < 2) {
            const uint32_t w = __ballot_sync(0xffffffffu, vis);
            if (lane == 0) bits[2 * i + warp] = w;
        }
        if (i < d.q_len) {
            all_rows = all_rows && vis;
            any_row = any_row || vis;
        }
    }
    const int all = __syncthreads_and(!active || all_rows);
    const int any = __syncthreads_or(active && any_row);
    if (threadIdx.x == 0) m.flags[fi] = any ? (all ? 1 : 2) : 0;
}

// Carve the scratch for this shape; false when it does not fit.
bool carve(unsigned char *base, const RingDims &d, RingDev &m) {
    size_t off = 0;
    auto take = [&](size_t bytes) {
        unsigned char *p = base + off;
        off += align256(bytes);
        return p;
    };
    const int qw = (d.q_len + 1) & ~1;
    m.err = reinterpret_cast<uint32_t *>(take(4));
    m.rope32 = reinterpret_cast<float2 *>(take(sizeof(float2) * d.n_seq * d.q_len * (d.head_dim / 2)));
    m.flags = take((size_t)d.n_seq * d.n_tiles);
    m.maskbits = reinterpret_cast<uint64_t *>(take(sizeof(uint64_t) * d.n_seq * d.n_tiles * qw));
    // split partials only when several CTAs share a (sequence, kv head): with one group the
    // attention kernel writes O itself
    m.part_acc = nullptr;
    m.part_ml = nullptr;
    if (d.groups > 1) {
        m.part_acc = reinterpret_cast<float *>(
            take(sizeof(float) * d.n_seq * d.n_head_kv * d.groups * kRows * kHeadDim));
        m.part_ml = reinterpret_cast<float2 *>(take(sizeof(float2) * d.n_seq * d.n_head_kv * d.groups * kRows));
    }
    return off <= kStaticScratchBytes;
}

int fail_static(int code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    set_global_error(buf);
    return code;
}

// Set-up, once per device (with that device current): the device address of the scratch
// array -- in host code its name is only a host-side stand-in -- and the attention
// kernels' attributes.
int scratch_base(const char *who, unsigned char **base, int *dev_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return fail_static(RING_ECUDA, "%s: cudaGetDevice failed", who);
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_static_scratch);
        if (e != cudaSuccess)
            return fail_static(RING_ECUDA, "%s: cudaGetSymbolAddress: %s", who, cudaGetErrorString(e));
        e = attend_kernels_init();
        if (e != cudaSuccess)
            return fail_static(RING_ECUDA, "%s: kernel attributes: %s", who, cudaGetErrorString(e));
        g_scratch_addr[dev] = ptr;
    }
    *base = static_cast<unsigned char *>(g_scratch_addr[dev]);
    *dev_out = dev;
    return RING_OK;
}

}  // namespace
}  // namespace dflash

using namespace dflash;

extern "C" int ring_attend_static(const ring_attend_static_args *a, void *stream) {
    if (!a) return fail_static(RING_EINVAL, "ring_attend_static: args is NULL");
    if (a->cap <= 0 || a->q_len <= 0 || a->n_head_kv <= 0 || a->n_head <= 0 || a->n_seq <= 0 ||
        !(a->rope_theta > 0.f))
        return fail_static(RING_EINVAL, "ring_attend_static: every dimension must be positive");
    if (a->head_dim != kHeadDim || a->n_head % a->n_head_kv)
        return fail_static(RING_EINVAL, "ring_attend_static: head_dim must be %d and n_head a "
                                        "multiple of n_head_kv", kHeadDim);
    const int group = a->n_head / a->n_head_kv;
    if ((int64_t)group * a->q_len > kRows || a->q_len > kMaxQWords)
        return fail_static(RING_EINVAL, "ring_attend_static: (n_head/n_head_kv)*q_len exceeds %d", kRows);
    if (a->n_seq > kMaxStaticSeqs)
        return fail_static(RING_ERANGE, "ring_attend_static: n_seq %d above the maximum %d",
                           a->n_seq, kMaxStaticSeqs);
    if ((int64_t)a->cap + a->q_len + 32 > (int64_t)INT32_MAX / 2)
        return fail_static(RING_EINVAL, "ring_attend_static: cap too large");
    if (!a->committed || !a->k || !a->v || !a->mask || !a->q || !a->k_noise || !a->v_noise || !a->o)
        return fail_static(RING_EINVAL, "ring_attend_static: NULL pointer argument");
    const uintptr_t align = reinterpret_cast<uintptr_t>(a->k) | reinterpret_cast<uintptr_t>(a->v) |
                            reinterpret_cast<uintptr_t>(a->q) | reinterpret_cast<uintptr_t>(a->o) |
                            reinterpret_cast<uintptr_t>(a->k_noise) | reinterpret_cast<uintptr_t>(a->v_noise);
    if (align & 15) return fail_static(RING_EINVAL, "ring_attend_static: buffers must be 16-byte aligned");
    const int64_t pos_limit = (int64_t)INT32_MAX - a->q_len - 1;
    StaticParams prm;
    for (int s = 0; s < a->n_seq; ++s) {
        if (a->committed[s] < 0 || a->committed[s] > pos_limit)
            return fail_static(RING_ERANGE, "ring_attend_static: committed[%d] out of range", s);
        prm.committed[s] = a->committed[s];
    }
    for (int j = 0; j < kHeadDim / 2; ++j)
        prm.inv_freq[j] = std::pow((double)a->rope_theta, -2.0 * j / kHeadDim);

    unsigned char *base = nullptr;
    int dev = 0;
    int rc = scratch_base("ring_attend_static", &base, &dev);
    if (rc != RING_OK) return rc;
    cudaError_t e = cudaSuccess;

    RingDims d{};
    d.cap = a->cap;
    d.q_len = a->q_len;
    d.head_dim = a->head_dim;
    d.n_head_kv = a->n_head_kv;
    d.n_head = a->n_head;
    d.n_layer = 1;
    d.n_seq = a->n_seq;
    d.a_step = 2 * a->q_len + 2;
    d.trash_slot = a->cap + a->q_len;
    d.kv_total = (a->cap + a->q_len + 1 + 31) / 32 * 32;
    d.kv_row = a->head_dim * a->n_head_kv;
    d.group = group;
    d.rows = group * a->q_len;
    d.n_tiles = (d.kv_total + kTile - 1) / kTile;
    d.n_kinds = 1;
    d.bulk_chunk = 1024;
    d.cluster = 1;
    // independent CTAs, about four waves of two per SM; fewer, longer splits when the
    // partials would not fit the scratch
    int sms = 1;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t pairs = (int64_t)d.n_seq * d.n_head_kv;
    const int64_t slots = 2LL * std::max(sms, 1);
    int64_t tps = (pairs * d.n_tiles + 4 * slots - 1) / (4 * slots);
    tps = std::max<int64_t>(2, std::min<int64_t>(64, tps));
    tps = std::min<int64_t>(tps, d.n_tiles);
    d.groups = (int)((d.n_tiles + tps - 1) / tps);
    RingDev m{};
    while (true) {
        d.tiles_per_split = (d.n_tiles + d.groups - 1) / d.groups;
        d.groups = (d.n_tiles + d.tiles_per_split - 1) / d.tiles_per_split;
        d.n_splits = d.groups;
        if (carve(base, d, m)) break;
        if (d.groups == 1)
            return fail_static(RING_ERANGE, "ring_attend_static: this shape needs more than the "
                                            "%zu bytes of static scratch", kStaticScratchBytes);
        d.groups = std::max(1, d.groups / 2);
    }
    d.single_wave = pairs * d.n_splits <= slots ? 1 : 0;
    m.k = static_cast<uint16_t *>(a->k);
    m.v = static_cast<uint16_t *>(a->v);

    CUtensorMap tm_k, tm_v;
    if (!encode_kv_tensor_map(&tm_k, a->k, d) || !encode_kv_tensor_map(&tm_v, a->v, d))
        return fail_static(RING_ECUDA, "ring_attend_static: cuTensorMapEncodeTiled failed");

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the error word (first word of the scratch) keeps its bits until
    // ring_attend_static_device_error reads and clears it
    k_static_prepare<<<dim3(d.n_tiles + 1, d.n_seq), 128, 0, st>>>(d, m, a->mask, prm);
    e = cudaGetLastError();
    const float scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)a->head_dim));
    if (e == cudaSuccess)
        e = launch_attend(d, m, &tm_k, &tm_v, 0, 0, scale_log2, a->q,
                          static_cast<const uint16_t *>(a->k_noise),
                          static_cast<const uint16_t *>(a->v_noise), a->o, false, 0, st);
    if (e == cudaSuccess && d.groups > 1) e = launch_attend_combine(d, m, a->o, st);
    if (e != cudaSuccess)
        return fail_static(RING_ECUDA, "ring_attend_static: launch: %s", cudaGetErrorString(e));
    return RING_OK;
}

extern "C" int ring_attend_static_device_error(uint32_t *bits) {
    unsigned char *base = nullptr;
    int dev = 0;
    int rc = scratch_base("ring_attend_static_device_error", &base, &dev);
    if (rc != RING_OK) return rc;
    // the error word is the first word of the scratch (see carve)
    uint32_t w = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(&w, base, 4, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && w) e = cudaMemset(base, 0, 4);
    if (e != cudaSuccess)
        return fail_static(RING_ECUDA, "ring_attend_static_device_error: %s", cudaGetErrorString(e));
    if (bits) *bits = w;
    if (w) return fail_static(RING_EDEVICE, "ring_attend_static: device error word 0x%x", w);
    return RING_OK;
}
