// Host side of the C ABI declared in include/dflash_ring.h.
//
// Owns the ring's device buffers (allocated and zeroed once, like the persistent buffer
// of the page "DFLASH2_RING_PORT.md", section 1.1), validates every argument before
// launching anything, performs the per-sequence window arithmetic of section 1.3 on the
// host (it needs only integers the caller already holds), stages those few bytes to the
// device through pinned memory and enqueues the kernels.  Nothing here blocks on the GPU
// except the read-back calls, destroy, and the rare reuse of a still-busy staging slot.
#include "dflash_ring.h"
#include "ring_internal.h"

#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

using namespace dflash;

namespace {

constexpr int kStagingSlots = 8;
constexpr int kKinds = 6;

struct EventRec {
    int cls;
    cudaEvent_t a, b;
};

struct GraphKey {
    const void *k_rows = nullptr, *v_rows = nullptr;
    int64_t n_rows = -1;
    int kind = -1;
    std::vector<const void *> ptrs;
    bool clock = false;
    bool operator==(const GraphKey &o) const {
        return k_rows == o.k_rows && v_rows == o.v_rows && n_rows == o.n_rows && kind == o.kind &&
               ptrs == o.ptrs && clock == o.clock;
    }
};

thread_local std::string g_init_error = "no error";

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

}  // namespace

struct dflash_ring {
    RingDims d{};
    RingDev m{};
    float rope_theta = 0.f;
    float scale_log2 = 0.f;
    int device = 0;
    std::vector<int64_t> next_pos, committed;
    bool have_step = false;
    CUtensorMap tm_k{}, tm_v{};
    SeqStep *h_steps = nullptr;            // pinned [kStagingSlots][n_seq]
    cudaEvent_t slot_ev[kStagingSlots] = {};
    bool slot_used[kStagingSlots] = {};
    int slot_next = 0;
    int64_t launches = 0;
    int64_t device_bytes = 0;
    bool profiling = false;
    std::vector<EventRec> recs;
    std::vector<cudaEvent_t> ev_pool;
    std::string err = "no error";
    std::vector<void *> allocs;
    cudaStream_t cap_stream = nullptr;
    // one replayable step graph per staging slot: its begin-step kernel reads that slot
    cudaGraphExec_t graph_exec[kStagingSlots] = {};
    GraphKey graph_key;
    int64_t graph_kernels = 0;
    bool last_was_begin = false;   // the ring's last kernel launch was the begin-step kernel
    // whole-step attention kernel inside ring_step: CTAs per (sequence, kv head), 0 = the
    // layers are launched one by one; step_pdl: it may overlap the begin-step kernel
    int step_split = 0;
    bool step_pdl = true;
    unsigned long long *clock_buf = nullptr;   // kernel clock words (ring_clock_enable)
    bool clock_on = false;
    // context-row producer (ring_set_producer): weights repacked into ring-owned tiles
    bool has_producer = false;
    int hidden = 0;
    float eps = 0.f;
    uint16_t *w_packed = nullptr;
    float *k_norm = nullptr;             // ring-owned copy [n_layer][head_dim]
    float *q_norm = nullptr;             // [n_layer][head_dim] when W_q is given
    int out_heads = 0;                   // heads per layer in the packed weights
    float *noise_q = nullptr;            // draft-step noise rows, [n_layer][n_seq][q_len][...]
    uint16_t *noise_k = nullptr, *noise_v = nullptr;
    CUtensorMap tm_w{};
    int sms = 0;
    int prod_slots[kProduceMaxSplit + 1] = {};   // resident producer CTAs per cluster size
};

namespace {

int fail(ring_t *r, int code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    if (r)
        r->err = buf;
    else
        g_init_error = buf;
    return code;
}

int cuda_fail(ring_t *r, cudaError_t e, const char *what) {
    return fail(r, e == cudaErrorMemoryAllocation ? RING_ENOMEM : RING_ECUDA, "%s: %s", what,
                cudaGetErrorString(e));
}

cudaEvent_t pool_event(ring_t *r) {
    if (!r->ev_pool.empty()) {
        cudaEvent_t e = r->ev_pool.back();
        r->ev_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

// Launch wrapper: counts the launch and, while profiling, brackets it with events.
template <typename F>
cudaError_t timed(ring_t *r, int cls, cudaStream_t st, F &&launch) {
    EventRec rec{cls, nullptr, nullptr};
    if (r->profiling) {
        rec.a = pool_event(r);
        rec.b = pool_event(r);
        cudaEventRecord(rec.a, st);
    }
    cudaError_t e = launch();
    if (r->profiling) {
        cudaEventRecord(rec.b, st);
        r->recs.push_back(rec);
    }
    if (e == cudaSuccess) ++r->launches;
    return e;
}

void *dalloc(ring_t *r, size_t bytes, cudaError_t *err) {
    void *p = nullptr;
    *err = cudaMalloc(&p, bytes);
    if (*err != cudaSuccess) return nullptr;
    r->allocs.push_back(p);
    r->device_bytes += (int64_t)bytes;
    return p;
}

void release(ring_t *r) {
    if (!r) return;
    cudaDeviceSynchronize();
    for (void *p : r->allocs) cudaFree(p);
    r->allocs.clear();
    if (r->h_steps) cudaFreeHost(r->h_steps);
    for (auto &e : r->slot_ev)
        if (e) cudaEventDestroy(e);
    for (auto &rec : r->recs) {
        cudaEventDestroy(rec.a);
        cudaEventDestroy(rec.b);
    }
    for (auto e : r->ev_pool) cudaEventDestroy(e);
    for (void *p : {(void *)r->w_packed, (void *)r->k_norm, (void *)r->q_norm, (void *)r->noise_q,
                    (void *)r->noise_k, (void *)r->noise_v})
        if (p) cudaFree(p);
    for (auto &ge : r->graph_exec)
        if (ge) cudaGraphExecDestroy(ge);
    if (r->cap_stream) cudaStreamDestroy(r->cap_stream);
    delete r;
}

bool encode_kv_map(CUtensorMap *tm, void *base, const RingDims &d) {
    auto fn = get_encode_fn();
    if (!fn) return false;
    // dims (innermost first): head_dim, kv_total slots, (seq, layer, kv head) planes; F16
    // slots in 64 x 64 boxes, q8_0 codes (one byte each) in 128 x 64 boxes -- 128 bytes wide
    const cuuint64_t esz = d.kv_q8 ? 1 : 2;
    cuuint64_t dims[3] = {(cuuint64_t)d.head_dim, (cuuint64_t)d.kv_total,
                          (cuuint64_t)d.n_seq * d.n_layer * d.n_head_kv};
    cuuint64_t strides[2] = {(cuuint64_t)d.head_dim * esz, (cuuint64_t)d.kv_total * d.head_dim * esz};
    cuuint32_t box[3] = {(cuuint32_t)(128 / esz), (cuuint32_t)kTile, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult res = fn(tm, d.kv_q8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                      3, base, dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return res == CUDA_SUCCESS;
}

// 2-D TMA map over F16 rows [rows][hidden]: 64 x box_rows boxes, 128-byte swizzle.
bool encode_weight_map(CUtensorMap *tm, const void *base, int hidden, int64_t rows,
                       int box_rows = 128) {
    auto fn = get_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)hidden, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)hidden * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult res = fn(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides,
                      box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return res == CUDA_SUCCESS;
}

// 3-D TMA map over the packed producer weights: planes of 128 rows x 64 columns.
bool encode_packed_map(CUtensorMap *tm, const void *base, int64_t planes) {
    auto fn = get_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {64, 128, (cuuint64_t)planes};
    cuuint64_t strides[2] = {128, 128 * 128};
    cuuint32_t box[3] = {64, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult res = fn(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(base), dims, strides,
                      box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return res == CUDA_SUCCESS;
}

int pow2_floor(int x) {
    int p = 1;
    while (p * 2 <= x) p *= 2;
    return p;
}

// Work split of the attention kernel.  A thread-block cluster holds every one of its SM
// slots until its slowest CTA is done, so clusters (merging through distributed shared
// memory, no second kernel) are used only when the whole grid fits in one wave of one
// CTA per SM -- the few-sequence case, where latency rules.  Otherwise each CTA is its
// own group: about four waves of independent CTAs (two per SM) stream the tiles and a
// small combine kernel merges the per-CTA partials.
void choose_split(RingDims &d, int sms, int max_cluster, int tps_req) {
    const int cmax = std::max(1, std::min(kMaxStepCluster, max_cluster));
    const int pairs = d.n_seq * d.n_head_kv;
    if (tps_req > 0) {
        const int tps = std::min(tps_req, d.n_tiles);
        const int ns = (d.n_tiles + tps - 1) / tps;
        d.cluster = std::min(pow2_floor(cmax), pow2_floor(ns));
        while (d.cluster > 1 && attend_cluster_capacity(d.cluster, d.kv_q8 != 0) < 1) d.cluster /= 2;
        d.groups = (ns + d.cluster - 1) / d.cluster;
        d.tiles_per_split = tps;
        d.n_splits = d.cluster * d.groups;
        return;
    }
    // widest cluster (any size up to 16) whose whole grid -- a cluster per pair -- is
    // resident at once and whose CTAs' row shares fit the receive buffers; then the
    // narrowest cluster with as few tiles per CTA, so that no CTA is left without tiles
    auto fits = [&](int c) {
        return c * ((kRows + c - 1) / c) <= kMaxRecvSlots && (int64_t)pairs * c <= std::max(sms, 1) &&
               (int64_t)attend_cluster_capacity(c, d.kv_q8 != 0) >= pairs;
    };
    int c = std::min(cmax, d.n_tiles);
    while (c > 1 && !fits(c)) --c;
    if (c >= 2) c = (d.n_tiles + (d.n_tiles + c - 1) / c - 1) / ((d.n_tiles + c - 1) / c);
    if (c >= 2 && (d.n_tiles + c - 1) / c <= 128) {
        d.cluster = c;
        d.groups = 1;
        d.tiles_per_split = (d.n_tiles + c - 1) / c;
    } else {
        const int slots = 2 * std::max(sms, 1);
        const int64_t work = (int64_t)pairs * d.n_tiles;
        int64_t tps = (work + 4LL * slots - 1) / (4LL * slots);
        tps = std::max<int64_t>(2, std::min<int64_t>(64, tps));
        tps = std::min<int64_t>(tps, d.n_tiles);
        d.cluster = 1;
        d.tiles_per_split = (int)tps;
        d.groups = (d.n_tiles + d.tiles_per_split - 1) / d.tiles_per_split;
    }
    d.n_splits = d.cluster * d.groups;
}

bool check_seq(ring_t *r, int32_t seq) { return r && seq >= 0 && seq < r->d.n_seq; }

}  // namespace

namespace dflash {
bool encode_kv_tensor_map(CUtensorMap *tm, void *base, const RingDims &d) {
    return encode_kv_map(tm, base, d);
}
void set_global_error(const char *msg) { g_init_error = msg; }
}  // namespace dflash

extern "C" {

int ring_init(ring_t **out, int32_t cap, int32_t q_len, int32_t head_dim, int32_t n_head_kv,
              int32_t n_head, int32_t n_layer, float rope_theta) {
    ring_params p{};
    p.cap = cap;
    p.q_len = q_len;
    p.head_dim = head_dim;
    p.n_head_kv = n_head_kv;
    p.n_head = n_head;
    p.n_layer = n_layer;
    p.rope_theta = rope_theta;
    p.n_seq = 1;
    return ring_init_ex(out, &p);
}

int ring_init_ex(ring_t **out, const ring_params *p) {
    if (!out) return fail(nullptr, RING_EINVAL, "ring_init: out is NULL");
    *out = nullptr;
    if (!p) return fail(nullptr, RING_EINVAL, "ring_init: params is NULL");
    const int n_seq = p->n_seq > 0 ? p->n_seq : 1;
    if (p->cap <= 0 || p->q_len <= 0 || p->head_dim <= 0 || p->n_head_kv <= 0 ||
        p->n_head <= 0 || p->n_layer <= 0 || p->swa_window < 0 || p->bulk_chunk < 0 ||
        p->tiles_per_split < 0 || p->max_cluster < 0 || p->step_split < -1 || !(p->rope_theta > 0.f))
        return fail(nullptr, RING_EINVAL, "ring_init: every dimension must be positive");
    if (p->n_head % p->n_head_kv)
        return fail(nullptr, RING_EINVAL, "ring_init: n_head %d not a multiple of n_head_kv %d",
                    p->n_head, p->n_head_kv);
    if (p->head_dim != kHeadDim)
        return fail(nullptr, RING_EINVAL, "ring_init: head_dim %d unsupported (needs %d)",
                    p->head_dim, kHeadDim);
    const int group = p->n_head / p->n_head_kv;
    if ((int64_t)group * p->q_len > kRows || p->q_len > kMaxQWords)
        return fail(nullptr, RING_EINVAL,
                    "ring_init: (n_head/n_head_kv)*q_len = %d exceeds %d query rows per kv head",
                    group * p->q_len, kRows);
    if ((int64_t)p->cap + p->q_len + 32 > (int64_t)INT32_MAX / 2)
        return fail(nullptr, RING_EINVAL, "ring_init: cap too large");
    if (p->kv_format != RING_KV_F16 && p->kv_format != RING_KV_Q8_0)
        return fail(nullptr, RING_EINVAL, "ring_init: unknown kv_format %d", p->kv_format);

    ring_t *r = new dflash_ring();
    RingDims &d = r->d;
    d.cap = p->cap;
    d.q_len = p->q_len;
    d.head_dim = p->head_dim;
    d.n_head_kv = p->n_head_kv;
    d.n_head = p->n_head;
    d.n_layer = p->n_layer;
    d.n_seq = n_seq;
    d.swa_window = p->swa_window;
    d.a_step = 2 * p->q_len + 2;                       // section 1.1
    d.trash_slot = p->cap + p->q_len;
    d.kv_total = (p->cap + p->q_len + 1 + 31) / 32 * 32;
    d.kv_row = p->head_dim * p->n_head_kv;
    d.group = group;
    d.rows = group * p->q_len;
    d.n_tiles = (d.kv_total + kTile - 1) / kTile;
    d.n_kinds = p->swa_window > 0 ? 2 : 1;
    d.bulk_chunk = p->bulk_chunk > 0 ? p->bulk_chunk : 1024;
    d.kv_q8 = p->kv_format == RING_KV_Q8_0 ? 1 : 0;
    r->rope_theta = p->rope_theta;
    r->scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)p->head_dim));

    cudaError_t e = cudaGetDevice(&r->device);
    if (e != cudaSuccess) {
        int rc = cuda_fail(nullptr, e, "ring_init: cudaGetDevice");
        delete r;
        return rc;
    }
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, r->device);
    r->sms = sms;
    e = attend_kernels_init();
    if (e == cudaSuccess) e = produce_kernels_init();
    if (e == cudaSuccess) e = produce_tc_init();
    if (e != cudaSuccess) {
        int rc = cuda_fail(nullptr, e, "ring_init: kernel attributes");
        delete r;
        return rc;
    }
    int max_cluster = p->max_cluster > 0 ? p->max_cluster : 16;
    choose_split(d, sms, max_cluster, p->tiles_per_split);
    {
        // one wave: every CTA (every cluster) of the attention grid resident at once; only
        // then may the kernel release its dependents early (they would otherwise hold SMs
        // that its own later CTAs wait for)
        const int64_t ctas = (int64_t)d.n_splits * d.n_head_kv * d.n_seq;
        if (d.cluster > 1)
            d.single_wave = ctas / d.cluster <= (int64_t)attend_cluster_capacity(d.cluster, d.kv_q8 != 0) &&
                            ctas <= std::max(sms, 1);
        else
            d.single_wave = ctas <= 2LL * std::max(sms, 1) ? 1 : 0;
    }
    // Whole-step attention (ring_step), on request: every layer runs in one persistent
    // kernel, one cluster of c CTAs per (sequence, kv head) (one CTA per SM); c given, or
    // (step_split = -1, with few pairs -- the case the clusters above serve) the widest
    // cluster of which one per pair is resident at once.  F16 slots, up to
    // kMaxStepLayers layers.  By default ring_step launches each layer: measured faster
    // at cap 4096 with one sequence.
    {
        const int pairs = d.n_seq * d.n_head_kv;
        const bool able = p->step_split != 0 && !d.kv_q8 && d.n_layer <= kMaxStepLayers &&
                          d.n_tiles <= kMaxStepTiles && attend_step_init() == cudaSuccess;
        auto fits = [&](int c) {
            return c >= 1 && c <= kMaxStepCluster && c * ((kRows + c - 1) / c) <= kMaxRecvSlots &&
                   attend_step_capacity(c) >= pairs;
        };
        int split = 0;
        if (able && p->step_split > 0) {
            if (fits(p->step_split)) split = p->step_split;
        } else if (able && p->step_split == -1 && d.cluster > 1) {
            for (int c = std::min(kMaxStepCluster, d.n_tiles); c >= 2 && !split; --c)
                if (fits(c)) split = c;
        }
        if (split > 0) {
            r->step_split = split;
            d.step_sync_words = d.n_layer + 1;
        } else if (p->step_split > 0) {
            int rc = fail(nullptr, RING_EINVAL,
                          "ring_init: step_split %d: the whole-step kernel needs F16 slots, at most "
                          "%d layers and %d tiles, clusters of at most %d CTAs with c * ceil(32 / c) "
                          "<= %d, and a cluster for each of the %d pairs resident at once",
                          p->step_split, kMaxStepLayers, kMaxStepTiles, kMaxStepCluster,
                          kMaxRecvSlots, pairs);
            delete r;
            return rc;
        }
    }

    const size_t kv_elems = (size_t)d.n_seq * d.n_layer * d.n_head_kv * d.kv_total * d.head_dim;
    RingDev &m = r->m;
#define ALLOC(ptr, type, count)                                                  \
    do {                                                                         \
        ptr = static_cast<type *>(dalloc(r, sizeof(type) * (size_t)(count), &e)); \
        if (!ptr) {                                                              \
            int rc = cuda_fail(nullptr, e, "ring_init: cudaMalloc " #ptr);       \
            release(r);                                                          \
            return rc;                                                           \
        }                                                                        \
    } while (0)
    if (d.kv_q8) {
        ALLOC(m.kq, int8_t, kv_elems);
        ALLOC(m.vq, int8_t, kv_elems);
        ALLOC(m.ks, uint16_t, kv_elems / 32);
        ALLOC(m.vs, uint16_t, kv_elems / 32);
    } else {
        ALLOC(m.k, uint16_t, kv_elems);
        ALLOC(m.v, uint16_t, kv_elems);
    }
    ALLOC(m.slot_pos, int32_t, (size_t)d.n_seq * d.cap);
    ALLOC(m.mask, float, (size_t)d.n_seq * d.n_kinds * d.q_len * d.kv_total);
    ALLOC(m.flags, uint8_t, (size_t)d.n_seq * d.n_kinds * d.n_tiles);
    ALLOC(m.maskbits, uint64_t, (size_t)d.n_seq * d.n_kinds * d.n_tiles * ((d.q_len + 1) & ~1));
    ALLOC(m.steps, SeqStep, d.n_seq);
    ALLOC(m.rope32, float2, (size_t)d.n_seq * d.q_len * d.head_dim / 2);
    ALLOC(m.part_acc, float, (size_t)d.n_seq * d.n_head_kv * d.groups * kRows * kHeadDim);
    ALLOC(m.part_ml, float2, (size_t)d.n_seq * d.n_head_kv * d.groups * kRows);
    ALLOC(m.err, uint32_t, 1);
    ALLOC(m.inv_freq, double, d.head_dim / 2);
    ALLOC(r->clock_buf, unsigned long long, kClockWords);
    ALLOC(m.probe, uint32_t, 2);
    if (r->step_split > 0) ALLOC(m.step_sync, uint32_t, d.step_sync_words);
#undef ALLOC

    // zeroed once (section 1.1); slot_pos = -1; masks start fully masked
    cudaError_t z = cudaSuccess;
    auto zero = [&](void *ptr, int val, size_t bytes) {
        if (z == cudaSuccess) z = cudaMemset(ptr, val, bytes);
    };
    if (d.kv_q8) {
        zero(m.kq, 0, kv_elems);
        zero(m.vq, 0, kv_elems);
        zero(m.ks, 0, kv_elems / 32 * 2);
        zero(m.vs, 0, kv_elems / 32 * 2);
    } else {
        zero(m.k, 0, kv_elems * 2);
        zero(m.v, 0, kv_elems * 2);
    }
    zero(m.slot_pos, 0xff, (size_t)d.n_seq * d.cap * 4);
    zero(m.mask, 0, (size_t)d.n_seq * d.n_kinds * d.q_len * d.kv_total * 4);
    zero(m.flags, 0, (size_t)d.n_seq * d.n_kinds * d.n_tiles);
    zero(m.maskbits, 0, (size_t)d.n_seq * d.n_kinds * d.n_tiles * ((d.q_len + 1) & ~1) * 8);
    zero(m.steps, 0, sizeof(SeqStep) * d.n_seq);
    zero(m.rope32, 0, (size_t)d.n_seq * d.q_len * d.head_dim / 2 * sizeof(float2));
    zero(m.err, 0, 4);
    zero(m.probe, 0, 8);
    const size_t clock_bank = (size_t)kClockKinds * kClockSlots;
    zero(r->clock_buf, 0xff, clock_bank * 8);                          // earliest start: none yet
    zero(r->clock_buf + clock_bank, 0, (kClockWords - clock_bank) * 8);   // latest end, step counter
    if (m.step_sync) zero(m.step_sync, 0, (size_t)d.step_sync_words * 4);
    std::vector<double> inv(d.head_dim / 2);
    for (int i = 0; i < d.head_dim / 2; ++i)
        inv[i] = std::pow((double)p->rope_theta, -2.0 * i / d.head_dim);
    if (z == cudaSuccess)
        z = cudaMemcpy(m.inv_freq, inv.data(), inv.size() * sizeof(double), cudaMemcpyHostToDevice);
    if (z == cudaSuccess) z = cudaDeviceSynchronize();
    if (z != cudaSuccess) {
        int rc = cuda_fail(nullptr, z, "ring_init: initialising buffers");
        release(r);
        return rc;
    }
    e = cudaMallocHost(reinterpret_cast<void **>(&r->h_steps), sizeof(SeqStep) * kStagingSlots * d.n_seq);
    if (e != cudaSuccess) {
        int rc = cuda_fail(nullptr, e, "ring_init: cudaMallocHost");
        r->h_steps = nullptr;
        release(r);
        return rc;
    }
    for (auto &ev : r->slot_ev) cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    const bool maps_ok = d.kv_q8 ? encode_kv_map(&r->tm_k, m.kq, d) && encode_kv_map(&r->tm_v, m.vq, d)
                                 : encode_kv_map(&r->tm_k, m.k, d) && encode_kv_map(&r->tm_v, m.v, d);
    if (!maps_ok) {
        int rc = fail(nullptr, RING_ECUDA, "ring_init: cuTensorMapEncodeTiled failed");
        release(r);
        return rc;
    }
    r->next_pos.assign(d.n_seq, 0);
    r->committed.assign(d.n_seq, 0);
    *out = r;
    return RING_OK;
}

int ring_destroy(ring_t *r) {
    release(r);
    return RING_OK;
}

int ring_get_geometry(const ring_t *r, ring_geometry *g) {
    if (!r || !g) return RING_EINVAL;
    const RingDims &d = r->d;
    g->cap = d.cap;
    g->q_len = d.q_len;
    g->a_step = d.a_step;
    g->trash_slot = d.trash_slot;
    g->kv_total = d.kv_total;
    g->kv_row = d.kv_row;
    g->head_dim = d.head_dim;
    g->n_head_kv = d.n_head_kv;
    g->n_head = d.n_head;
    g->n_layer = d.n_layer;
    g->n_seq = d.n_seq;
    g->swa_window = d.swa_window;
    g->bulk_chunk = d.bulk_chunk;
    g->tile_slots = kTile;
    g->n_tiles = d.n_tiles;
    g->tiles_per_split = d.tiles_per_split;
    g->n_splits = d.n_splits;
    g->cluster = d.cluster;
    g->groups = d.groups;
    g->cache_bytes = d.kv_q8 ? 2LL * d.n_layer * d.kv_total * (d.kv_row + d.kv_row / 32 * 2)
                             : 2LL * d.n_layer * d.kv_row * d.kv_total * 2;
    g->device_bytes = r->device_bytes;
    g->step_split = r->step_split;
    g->step_ctas = r->step_split * d.n_seq * d.n_head_kv;
    return RING_OK;
}

int ring_rows_needed(const ring_t *r, int32_t seq, int64_t committed, int64_t *start,
                     int32_t *n_new) {
    if (!r || seq < 0 || seq >= r->d.n_seq) return RING_EINVAL;
    const int64_t c = committed, np = r->next_pos[seq];
    if (c < np || c < 0) return RING_ERANGE;
    const int64_t win = std::min<int64_t>(c, r->d.cap);    // section 1.3
    const int64_t lo = c - win;
    const int64_t st = std::max(np, lo);
    if (start) *start = st;
    if (n_new) *n_new = (int32_t)(c - st);
    return RING_OK;
}

}  // extern "C"

namespace {

// Section 1.3 window arithmetic and every argument check of one begin_step; fills the
// per-sequence step records.  Touches no state.
// full_window: every position of [lo, c) is appended again (the page's legacy path that
// recomputes the whole window each step), not only the new ones.
int validate_step(ring_t *r, const char *who, const int64_t *committed, const void *k_rows,
                  const void *v_rows, const int64_t *row_off, const int64_t *first_pos,
                  int64_t n_rows, std::vector<SeqStep> &st, int64_t &max_bulk,
                  bool full_window = false) {
    if (!committed) return fail(r, RING_EINVAL, "%s: committed is NULL", who);
    const RingDims &d = r->d;
    const int64_t pos_limit = (int64_t)INT32_MAX - d.q_len - 1;
    st.assign(d.n_seq, SeqStep{});
    max_bulk = 0;
    bool any_rows = false;
    for (int s = 0; s < d.n_seq; ++s) {
        const int64_t c = committed[s];
        if (c < 0 || c > pos_limit)
            return fail(r, RING_ERANGE, "%s: committed[%d] = %lld out of range", who, s, (long long)c);
        if (c < r->next_pos[s])
            return fail(r, RING_ERANGE, "%s: committed[%d] = %lld went below %lld", who, s,
                        (long long)c, (long long)r->next_pos[s]);
        const int64_t win = std::min<int64_t>(c, d.cap);
        const int64_t lo = c - win;
        const int64_t start = full_window ? lo : std::max(r->next_pos[s], lo);
        const int64_t n_new = c - start;
        SeqStep &x = st[s];
        x.committed = c;
        x.lo = lo;
        x.swa_lo = d.swa_window > 0 ? c - std::min<int64_t>(d.swa_window, win) : lo;
        x.start = start;
        x.n_new = (int32_t)n_new;
        x.fold_rows = n_new <= d.a_step ? (int32_t)n_new : 0;
        x.src_row = 0;
        if (n_new > 0) {
            any_rows = true;
            if (!row_off || !first_pos) return fail(r, RING_EINVAL, "%s: row_off/first_pos are NULL", who);
            if (first_pos[s] > start || first_pos[s] < 0)
                return fail(r, RING_ERANGE, "%s: rows of seq %d start at %lld, after start %lld", who, s,
                            (long long)first_pos[s], (long long)start);
            if (row_off[s] < 0 || row_off[s] + (c - first_pos[s]) > n_rows)
                return fail(r, RING_ERANGE, "%s: rows of seq %d run past n_rows %lld", who, s,
                            (long long)n_rows);
            x.src_row = row_off[s] + (start - first_pos[s]);
            if (n_new > d.a_step) max_bulk = std::max(max_bulk, n_new);
        }
    }
    if (any_rows) {
        if (!k_rows || !v_rows) return fail(r, RING_EINVAL, "%s: rows are NULL", who);
        if ((reinterpret_cast<uintptr_t>(k_rows) | reinterpret_cast<uintptr_t>(v_rows)) & 15)
            return fail(r, RING_EINVAL, "%s: rows must be 16-byte aligned", who);
    }
    return RING_OK;
}

// The step records go to a rotating pinned host slot (*slot), which the begin-step kernel
// reads directly -- no copy ahead of its launch; a device copy is made as well when other
// kernels read the records (bulk chunks, the producer).  Then the bulk chunks (slot_pos of
// those slots is read by the begin kernel, which runs after them).  The caller marks the
// slot busy (mark_slot) after the last launch that reads it.
int stage_and_bulk(ring_t *r, const char *who, const std::vector<SeqStep> &st, const void *k_rows,
                   const void *v_rows, int64_t n_rows, int64_t max_bulk, cudaStream_t cs, int *slot_out,
                   bool device_copy = false) {
    const RingDims &d = r->d;
    const int slot = r->slot_next;
    r->slot_next = (slot + 1) % kStagingSlots;
    if (r->slot_used[slot]) {
        cudaError_t e = cudaEventSynchronize(r->slot_ev[slot]);
        if (e != cudaSuccess) return cuda_fail(r, e, who);
        r->slot_used[slot] = false;
    }
    *slot_out = slot;
    SeqStep *h = r->h_steps + (size_t)slot * d.n_seq;
    std::memcpy(h, st.data(), sizeof(SeqStep) * d.n_seq);
    cudaError_t e = cudaSuccess;
    if (device_copy || max_bulk > 0)
        e = cudaMemcpyAsync(r->m.steps, h, sizeof(SeqStep) * d.n_seq, cudaMemcpyHostToDevice, cs);
    if (e != cudaSuccess) return cuda_fail(r, e, who);
    const auto *kr = static_cast<const uint16_t *>(k_rows);
    const auto *vr = static_cast<const uint16_t *>(v_rows);
    const int n_chunks = (int)((max_bulk + d.bulk_chunk - 1) / d.bulk_chunk);
    for (int c = 0; c < n_chunks && e == cudaSuccess; ++c)
        e = timed(r, 0, cs, [&] { return launch_bulk_append(d, r->m, kr, vr, n_rows, c, cs); });
    return e == cudaSuccess ? RING_OK : cuda_fail(r, e, who);
}

const SeqStep *slot_steps(const ring_t *r, int slot) { return r->h_steps + (size_t)slot * r->d.n_seq; }

// The staging slot may be rewritten once everything enqueued so far on cs has run.
void mark_slot(ring_t *r, int slot, cudaStream_t cs) {
    cudaEventRecord(r->slot_ev[slot], cs);
    r->slot_used[slot] = true;
}

void commit_host(ring_t *r, const int64_t *committed) {
    for (int s = 0; s < r->d.n_seq; ++s) {
        r->next_pos[s] = committed[s];
        r->committed[s] = committed[s];
    }
    r->have_step = true;
}

int validate_attend(ring_t *r, const char *who, int32_t layer, int32_t mask_kind, const void *q,
                    const void *k_noise, const void *v_noise, const void *o) {
    const RingDims &d = r->d;
    if (layer < 0 || layer >= d.n_layer) return fail(r, RING_EINVAL, "%s: layer %d out of range", who, layer);
    if (mask_kind != RING_MASK_FULL && mask_kind != RING_MASK_SWA)
        return fail(r, RING_EINVAL, "%s: unknown mask kind %d", who, mask_kind);
    if (mask_kind == RING_MASK_SWA && d.n_kinds < 2)
        return fail(r, RING_EINVAL, "%s: SWA mask needs swa_window > 0 at init", who);
    if (!q || !k_noise || !v_noise || !o) return fail(r, RING_EINVAL, "%s: NULL input or output", who);
    if ((reinterpret_cast<uintptr_t>(k_noise) | reinterpret_cast<uintptr_t>(v_noise) |
         reinterpret_cast<uintptr_t>(o) | reinterpret_cast<uintptr_t>(q)) & 15)
        return fail(r, RING_EINVAL, "%s: inputs and output must be 16-byte aligned", who);
    return RING_OK;
}

cudaError_t launch_layer(ring_t *r, int32_t layer, int32_t mask_kind, const float *q,
                         const void *k_noise, const void *v_noise, float *o, bool pdl,
                         cudaStream_t cs) {
    const RingDims &d = r->d;
    const auto *kn = static_cast<const uint16_t *>(k_noise);
    const auto *vn = static_cast<const uint16_t *>(v_noise);
    // preloading before the grid dependency is safe unless the ring's previous launch was
    // the begin-step kernel, which writes context rows, flags and bits (and the RoPE table
    // that the query prologue reads)
    const bool preload = !r->last_was_begin;
    const int early = preload ? kAttendPreload : 0;
    r->last_was_begin = false;
    cudaError_t e = timed(r, 2, cs, [&] {
        return launch_attend(d, r->m, &r->tm_k, &r->tm_v, layer, mask_kind, r->scale_log2, q, kn, vn,
                             o, pdl, early, cs);
    });
    if (e == cudaSuccess && d.groups > 1)
        e = timed(r, 3, cs, [&] { return launch_attend_combine(d, r->m, o, cs); });
    return e;
}

}  // namespace

extern "C" {

int ring_begin_step(ring_t *r, const int64_t *committed, const void *k_rows, const void *v_rows,
                    const int64_t *row_off, const int64_t *first_pos, int64_t n_rows,
                    void *stream) {
    if (!r) return RING_EINVAL;
    std::vector<SeqStep> st;
    int64_t max_bulk = 0;
    int rc = validate_step(r, "ring_begin_step", committed, k_rows, v_rows, row_off, first_pos,
                           n_rows, st, max_bulk);
    if (rc != RING_OK) return rc;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    int slot = 0;
    rc = stage_and_bulk(r, "ring_begin_step", st, k_rows, v_rows, n_rows, max_bulk, cs, &slot);
    if (rc != RING_OK) return rc;
    const auto *kr = static_cast<const uint16_t *>(k_rows);
    const auto *vr = static_cast<const uint16_t *>(v_rows);
    cudaError_t e = timed(r, 1, cs, [&] {
        return launch_begin_step(r->d, r->m, kr, vr, n_rows, !r->profiling, slot_steps(r, slot), cs);
    });
    mark_slot(r, slot, cs);
    if (e != cudaSuccess) return cuda_fail(r, e, "ring_begin_step: launch");
    r->last_was_begin = true;
    commit_host(r, committed);
    return RING_OK;
}

int ring_set_producer(ring_t *r, const ring_producer *p) {
    if (!r) return RING_EINVAL;
    auto drop = [&] {
        if (r->w_packed) cudaDeviceSynchronize();   // no step may still read them
        for (void *q : {(void *)r->w_packed, (void *)r->k_norm, (void *)r->q_norm,
                        (void *)r->noise_q, (void *)r->noise_k, (void *)r->noise_v})
            if (q) cudaFree(q);
        r->w_packed = nullptr;
        r->k_norm = r->q_norm = r->noise_q = nullptr;
        r->noise_k = r->noise_v = nullptr;
        r->has_producer = false;
    };
    if (!p) {
        drop();
        return RING_OK;
    }
    const RingDims &d = r->d;
    if (p->hidden <= 0 || p->hidden % 64)
        return fail(r, RING_EINVAL, "ring_set_producer: hidden %d must be a positive multiple of 64",
                    p->hidden);
    if (!p->wk || !p->wv || !p->k_norm)
        return fail(r, RING_EINVAL, "ring_set_producer: weights are NULL");
    if ((reinterpret_cast<uintptr_t>(p->wk) | reinterpret_cast<uintptr_t>(p->wv) |
         reinterpret_cast<uintptr_t>(p->wq)) & 15)
        return fail(r, RING_EINVAL, "ring_set_producer: weights must be 16-byte aligned");
    if (!p->wq != !p->q_norm)
        return fail(r, RING_EINVAL, "ring_set_producer: give both wq and q_norm, or neither");
    if (!(p->eps >= 0.f)) return fail(r, RING_EINVAL, "ring_set_producer: eps must be >= 0");
    drop();
    const int n_q = p->wq ? d.n_head : 0;
    const int out_heads = 2 * d.n_head_kv + n_q;
    const size_t w_elems = (size_t)out_heads * d.n_layer * d.head_dim * p->hidden;
    const size_t kn_bytes = sizeof(float) * (size_t)d.n_layer * d.head_dim;
    const size_t noise_rows = (size_t)d.n_layer * d.n_seq * d.q_len;
    cudaError_t e = cudaMalloc(&r->w_packed, w_elems * 2);
    if (e == cudaSuccess) e = cudaMalloc(&r->k_norm, kn_bytes);
    if (e == cudaSuccess && n_q) e = cudaMalloc(&r->q_norm, kn_bytes);
    if (e == cudaSuccess && n_q) e = cudaMalloc(&r->noise_q, noise_rows * d.n_head * d.head_dim * 4);
    if (e == cudaSuccess && n_q) e = cudaMalloc(&r->noise_k, noise_rows * d.kv_row * 2);
    if (e == cudaSuccess && n_q) e = cudaMalloc(&r->noise_v, noise_rows * d.kv_row * 2);
    if (e == cudaSuccess)
        e = launch_pack_weights(static_cast<const uint16_t *>(p->wk), static_cast<const uint16_t *>(p->wv),
                                static_cast<const uint16_t *>(p->wq), r->w_packed, d.n_layer,
                                d.n_head_kv, n_q, p->hidden, nullptr);
    if (e == cudaSuccess) e = cudaMemcpy(r->k_norm, p->k_norm, kn_bytes, cudaMemcpyDeviceToDevice);
    if (e == cudaSuccess && n_q) e = cudaMemcpy(r->q_norm, p->q_norm, kn_bytes, cudaMemcpyDeviceToDevice);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        int rc = cuda_fail(r, e, "ring_set_producer: packing the weights");
        drop();
        return rc;
    }
    const int64_t planes = (int64_t)d.n_layer * out_heads * (p->hidden / 64);
    if (!encode_packed_map(&r->tm_w, r->w_packed, planes)) {
        drop();
        return fail(r, RING_ECUDA, "ring_set_producer: cuTensorMapEncodeTiled failed");
    }
    r->hidden = p->hidden;
    r->eps = p->eps;
    r->out_heads = out_heads;
    for (int ks = 1; ks <= kProduceMaxSplit; ++ks) r->prod_slots[ks] = produce_capacity(ks, r->sms);
    r->has_producer = true;
    return RING_OK;
}

}  // extern "C"

namespace {
// A draft step's first-layer noise rows, projected in the same launch as its context rows.
struct NoiseJob {
    const void *h;            // every layer's hidden states [n_layer][n_seq][q_len][hidden]
    const CUtensorMap *tm;    // 2-D TMA map over them
};

int begin_step_features(ring_t *r, const char *who, const int64_t *committed, const void *feat,
                        const int64_t *row_off, const int64_t *first_pos, int64_t n_rows,
                        void *stream, bool full_window, const NoiseJob *noise = nullptr) {
    if (!r) return RING_EINVAL;
    if (!r->has_producer)
        return fail(r, RING_ESTATE, "%s: no producer set (ring_set_producer)", who);
    const RingDims &d = r->d;
    std::vector<SeqStep> st;
    int64_t max_bulk = 0;
    int rc = validate_step(r, who, committed, feat, feat, row_off, first_pos, n_rows, st, max_bulk,
                           full_window);
    if (rc != RING_OK) return rc;
    int64_t m_total = 0;
    for (auto &x : st) {
        x.prod_base = m_total;
        m_total += x.n_new;
    }
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    // Few sequences: the row ranges travel as kernel parameters; otherwise the projection
    // reads the staged step records from the device.
    ProduceSeqs ps{};
    if (d.n_seq <= kProduceParamSeqs) {
        ps.n = d.n_seq;
        for (int s = 0; s < d.n_seq; ++s) {
            ps.base[s] = st[s].prod_base;
            ps.n_new[s] = st[s].n_new;
            ps.start[s] = st[s].start;
            ps.src_row[s] = st[s].src_row;
        }
    }
    CUtensorMap tm_feat{};
    if (m_total > 0 && !encode_weight_map(&tm_feat, feat, r->hidden, n_rows, 32))
        return fail(r, RING_ECUDA, "%s: cuTensorMapEncodeTiled failed", who);
    // Order: the step records, the projection, then the begin-step kernel.  The projection
    // streams its first weight tiles while the previous kernel (the last reader of the ring)
    // finishes and waits for it before it reads rows or writes slots; the begin-step kernel
    // computes the slot_pos of the new rows itself, so it runs alongside the projection once
    // that has passed its wait, and waits for it only before exiting.
    int slot = 0;
    rc = stage_and_bulk(r, who, st, nullptr, nullptr, n_rows, 0, cs, &slot, ps.n == 0 && m_total > 0);
    if (rc != RING_OK) return rc;
    cudaError_t e = cudaSuccess;
    const bool produce = m_total > 0 || noise;
    // Many rows in one contiguous run of features: the context rows go to the tensor-core
    // kernel (a dense contraction), the noise rows (if any) to the streaming kernel after it.
    int64_t frow_base = -1;
    bool tc = m_total >= kProduceTcMinRows;
    for (int s = 0; s < d.n_seq && tc; ++s) {
        if (st[s].n_new == 0) continue;
        const int64_t b = st[s].src_row - st[s].prod_base;
        if (frow_base < 0) frow_base = b;
        tc = b == frow_base;
    }
    if (tc) {
        CUtensorMap tm_feat128{};
        if (!encode_weight_map(&tm_feat128, feat, r->hidden, n_rows, 128))
            return fail(r, RING_ECUDA, "%s: cuTensorMapEncodeTiled failed", who);
        e = timed(r, 5, cs, [&] {
            return launch_produce_tc(d, r->m, &r->tm_w, &tm_feat128, r->hidden, m_total, frow_base,
                                     r->out_heads, r->k_norm, r->eps, ps, r->sms, !r->profiling, cs);
        });
    }
    if (e == cudaSuccess && ((m_total > 0 && !tc) || noise)) {
        ProduceLaunch L{};
        const uint16_t *in[2] = {nullptr, nullptr};
        const CUtensorMap *tm[2] = {nullptr, nullptr};
        int64_t units = 0;
        if (m_total > 0 && !tc) {
            L.job[L.n_jobs] = ProduceJob{0, 0, m_total, produce_units(d, 0, m_total, r->out_heads)};
            in[L.n_jobs] = static_cast<const uint16_t *>(feat);
            tm[L.n_jobs] = &tm_feat;
            units += L.job[L.n_jobs++].units;
        }
        if (noise) {
            const int64_t nrow = (int64_t)d.n_seq * d.q_len;
            L.job[L.n_jobs] = ProduceJob{1, 0, nrow, produce_units(d, 1, nrow, r->out_heads)};
            in[L.n_jobs] = static_cast<const uint16_t *>(noise->h);
            tm[L.n_jobs] = noise->tm;
            units += L.job[L.n_jobs++].units;
        }
        L.ks = produce_split(units, r->hidden, r->prod_slots);
        L.out_heads = r->out_heads;
        const NoiseOut nout{r->noise_q, r->noise_k, r->noise_v, r->q_norm};
        e = timed(r, 5, cs, [&] {
            return launch_produce(d, r->m, &r->tm_w, tm[0], tm[1], in[0], in[1], r->hidden, L,
                                  r->k_norm, r->eps, ps, nout, !r->profiling, r->prod_slots[L.ks],
                                  cs);
        });
    }
    if (e == cudaSuccess)
        e = timed(r, 1, cs, [&] {
            return launch_begin_step(d, r->m, nullptr, nullptr, n_rows, !r->profiling,
                                     slot_steps(r, slot), cs, produce);
        });
    mark_slot(r, slot, cs);
    if (e != cudaSuccess) return cuda_fail(r, e, who);
    r->last_was_begin = true;
    commit_host(r, committed);
    return RING_OK;
}
}  // namespace

extern "C" {

int ring_begin_step_features(ring_t *r, const int64_t *committed, const void *feat,
                             const int64_t *row_off, const int64_t *first_pos, int64_t n_rows,
                             void *stream) {
    return begin_step_features(r, "ring_begin_step_features", committed, feat, row_off, first_pos,
                               n_rows, stream, false);
}

int ring_recompute_window(ring_t *r, const int64_t *committed, const void *feat,
                          const int64_t *row_off, const int64_t *first_pos, int64_t n_rows,
                          void *stream) {
    return begin_step_features(r, "ring_recompute_window", committed, feat, row_off, first_pos,
                               n_rows, stream, true);
}

int ring_draft_step(ring_t *r, const int64_t *committed, const void *feat,
                    const int64_t *row_off, const int64_t *first_pos, int64_t n_rows,
                    const void *noise_h, const int32_t *mask_kinds, float *const *o, void *stream) {
    if (!r) return RING_EINVAL;
    const RingDims &d = r->d;
    const char *who = "ring_draft_step";
    if (!r->has_producer || !r->noise_q)
        return fail(r, RING_ESTATE, "%s: no producer with W_q set (ring_set_producer)", who);
    if (!noise_h || !mask_kinds || !o) return fail(r, RING_EINVAL, "%s: NULL argument", who);
    if (reinterpret_cast<uintptr_t>(noise_h) & 15)
        return fail(r, RING_EINVAL, "%s: noise_h must be 16-byte aligned", who);
    const int64_t nrow = (int64_t)d.n_seq * d.q_len;
    for (int l = 0; l < d.n_layer; ++l) {
        int rc = validate_attend(r, who, l, mask_kinds[l], r->noise_q, r->noise_k, r->noise_v, o[l]);
        if (rc != RING_OK) return rc;
    }
    CUtensorMap tm_h{};
    if (!encode_weight_map(&tm_h, noise_h, r->hidden, nrow * d.n_layer, 32))
        return fail(r, RING_ECUDA, "%s: cuTensorMapEncodeTiled failed", who);
    // layer 0's hidden states are there from the start (the noise block's embeddings): its
    // projection shares the context rows' launch
    const NoiseJob first{noise_h, &tm_h};
    int rc = begin_step_features(r, who, committed, feat, row_off, first_pos, n_rows, stream, false,
                                 &first);
    if (rc != RING_OK) return rc;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const int64_t units = produce_units(d, 1, nrow, r->out_heads);
    const int ks = produce_split(units, r->hidden, r->prod_slots);
    const NoiseOut nout{r->noise_q, r->noise_k, r->noise_v, r->q_norm};
    ProduceSeqs ps{};
    const bool pdl = !r->profiling;
    for (int l = 0; l < d.n_layer; ++l) {
        cudaError_t e = cudaSuccess;
        if (l > 0) {
            // this layer's noise rows (Q, K, V from its hidden states, which in a draft
            // model come from the layer before: read after that kernel is done)
            ProduceLaunch L{};
            L.job[0] = ProduceJob{1, l, nrow, units};
            L.n_jobs = 1;
            L.ks = ks;
            L.out_heads = r->out_heads;
            e = timed(r, 5, cs, [&] {
                return launch_produce(d, r->m, &r->tm_w, &tm_h, nullptr,
                                      static_cast<const uint16_t *>(noise_h), nullptr, r->hidden, L,
                                      r->k_norm, r->eps, ps, nout, pdl, r->prod_slots[ks], cs);
            });
            if (e != cudaSuccess) return cuda_fail(r, e, who);
        }
        const int64_t qoff = (int64_t)l * nrow * d.n_head * d.head_dim;
        const int64_t koff = (int64_t)l * nrow * d.kv_row;
        // the projection writes no ring state, so the attention may fill its first stages
        // early -- except right after the begin-step kernel (layer 0), whose completion
        // stands for this step's context rows
        r->last_was_begin = l == 0;
        e = launch_layer(r, l, mask_kinds[l], r->noise_q + qoff, r->noise_k + koff,
                         r->noise_v + koff, o[l], pdl, cs);
        if (e != cudaSuccess) return cuda_fail(r, e, who);
    }
    return RING_OK;
}

int ring_attend(ring_t *r, int32_t layer, int32_t mask_kind, const float *q, const void *k_noise,
                const void *v_noise, float *o, void *stream) {
    if (!r) return RING_EINVAL;
    int rc = validate_attend(r, "ring_attend", layer, mask_kind, q, k_noise, v_noise, o);
    if (rc != RING_OK) return rc;
    if (!r->have_step) return fail(r, RING_ESTATE, "ring_attend: no ring_begin_step yet");
    cudaError_t e = launch_layer(r, layer, mask_kind, q, k_noise, v_noise, o, !r->profiling,
                                 static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(r, e, "ring_attend: launch");
    return RING_OK;
}

int ring_step(ring_t *r, const int64_t *committed, const void *k_rows, const void *v_rows,
              const int64_t *row_off, const int64_t *first_pos, int64_t n_rows, int32_t mask_kind,
              const float *const *q, const void *const *k_noise, const void *const *v_noise,
              float *const *o, void *stream) {
    if (!r) return RING_EINVAL;
    const RingDims &d = r->d;
    if (!q || !k_noise || !v_noise || !o)
        return fail(r, RING_EINVAL, "ring_step: per-layer pointer arrays are NULL");
    for (int l = 0; l < d.n_layer; ++l) {
        int rc = validate_attend(r, "ring_step", l, mask_kind, q[l], k_noise[l], v_noise[l], o[l]);
        if (rc != RING_OK) return rc;
    }
    std::vector<SeqStep> st;
    int64_t max_bulk = 0;
    int rc = validate_step(r, "ring_step", committed, k_rows, v_rows, row_off, first_pos, n_rows,
                           st, max_bulk);
    if (rc != RING_OK) return rc;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    int slot = 0;
    rc = stage_and_bulk(r, "ring_step", st, k_rows, v_rows, n_rows, max_bulk, cs, &slot);
    if (rc != RING_OK) return rc;

    // the fixed-topology step graph: captured once per staging slot, re-captured only when
    // a pointer the kernels take as a parameter changes
    GraphKey key;
    key.k_rows = k_rows;
    key.v_rows = v_rows;
    key.n_rows = n_rows;
    key.kind = mask_kind;
    for (int l = 0; l < d.n_layer; ++l) {
        key.ptrs.push_back(q[l]);
        key.ptrs.push_back(k_noise[l]);
        key.ptrs.push_back(v_noise[l]);
        key.ptrs.push_back(o[l]);
    }
    key.clock = r->clock_on;
    cudaError_t e = cudaSuccess;
    if (!(key == r->graph_key)) {
        for (auto &ge : r->graph_exec)
            if (ge) cudaGraphExecDestroy(ge);
        for (auto &ge : r->graph_exec) ge = nullptr;
        r->graph_key = key;
    }
    cudaGraphExec_t &gexec = r->graph_exec[slot];
    if (!gexec) {
        if (!r->cap_stream) {
            e = cudaStreamCreateWithFlags(&r->cap_stream, cudaStreamNonBlocking);
            if (e != cudaSuccess) return cuda_fail(r, e, "ring_step: capture stream");
        }
        const bool prof = r->profiling;
        r->profiling = false;              // no events inside the graph
        // capture: the begin-step kernel, then either the whole-step attention kernel or one
        // attention launch (+ combine) per layer
        auto capture = [&]() -> cudaError_t {
            cudaError_t ce = cudaStreamBeginCapture(r->cap_stream, cudaStreamCaptureModeThreadLocal);
            if (ce != cudaSuccess) return ce;
            const auto *kr = static_cast<const uint16_t *>(k_rows);
            const auto *vr = static_cast<const uint16_t *>(v_rows);
            cudaError_t le = launch_begin_step(d, r->m, kr, vr, n_rows, true, slot_steps(r, slot),
                                               r->cap_stream);
            r->last_was_begin = true;
            if (r->step_split > 0) {
                StepIO io{};
                for (int l = 0; l < d.n_layer; ++l) {
                    io.q[l] = q[l];
                    io.k_noise[l] = static_cast<const uint16_t *>(k_noise[l]);
                    io.v_noise[l] = static_cast<const uint16_t *>(v_noise[l]);
                    io.o[l] = o[l];
                }
                if (le == cudaSuccess)
                    le = timed(r, 2, r->cap_stream, [&] {
                        return launch_attend_step(d, r->m, &r->tm_k, &r->tm_v, mask_kind, r->scale_log2,
                                                  io, r->step_split, r->step_pdl, r->cap_stream);
                    });
                r->last_was_begin = false;
            } else {
                for (int l = 0; l < d.n_layer && le == cudaSuccess; ++l)
                    le = launch_layer(r, l, mask_kind, q[l], k_noise[l], v_noise[l], o[l], true,
                                      r->cap_stream);
            }
            cudaGraph_t graph = nullptr;
            ce = cudaStreamEndCapture(r->cap_stream, &graph);
            if (le != cudaSuccess) ce = le;
            if (ce == cudaSuccess) ce = cudaGraphInstantiate(&gexec, graph, 0);
            if (graph) cudaGraphDestroy(graph);
            return ce;
        };
        e = capture();
        if (e != cudaSuccess && r->step_split > 0 && r->step_pdl) {
            // a cooperative launch that may not overlap its predecessor: capture it plainly
            cudaGetLastError();
            if (gexec) cudaGraphExecDestroy(gexec);
            gexec = nullptr;
            r->step_pdl = false;
            e = capture();
        }
        r->profiling = prof;
        if (e != cudaSuccess) {
            if (gexec) cudaGraphExecDestroy(gexec);
            gexec = nullptr;
            return cuda_fail(r, e, "ring_step: graph capture");
        }
        r->graph_kernels = r->step_split > 0 ? 2 : 1 + d.n_layer * (d.groups > 1 ? 2 : 1);
    }
    e = timed(r, 4, cs, [&] { return cudaGraphLaunch(gexec, cs); });
    mark_slot(r, slot, cs);
    if (e != cudaSuccess) return cuda_fail(r, e, "ring_step: graph launch");
    r->launches += r->graph_kernels - 1;   // timed() counted the launch itself once
    commit_host(r, committed);
    return RING_OK;
}

int ring_get_slot_pos(ring_t *r, int32_t seq, int32_t *out) {
    if (!check_seq(r, seq) || !out) return RING_EINVAL;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess)
        e = cudaMemcpy(out, r->m.slot_pos + (size_t)seq * r->d.cap, sizeof(int32_t) * r->d.cap,
                       cudaMemcpyDeviceToHost);
    return e == cudaSuccess ? RING_OK : cuda_fail(r, e, "ring_get_slot_pos");
}

int ring_get_mask(ring_t *r, int32_t seq, int32_t mask_kind, float *out) {
    if (!check_seq(r, seq) || !out || mask_kind < 0 || mask_kind >= r->d.n_kinds)
        return RING_EINVAL;
    const RingDims &d = r->d;
    const size_t n = (size_t)d.q_len * d.kv_total;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess)
        e = cudaMemcpy(out, r->m.mask + ((size_t)seq * d.n_kinds + mask_kind) * n, n * sizeof(float),
                       cudaMemcpyDeviceToHost);
    return e == cudaSuccess ? RING_OK : cuda_fail(r, e, "ring_get_mask");
}

int ring_get_tile_flags(ring_t *r, int32_t seq, int32_t mask_kind, uint8_t *out) {
    if (!check_seq(r, seq) || !out || mask_kind < 0 || mask_kind >= r->d.n_kinds)
        return RING_EINVAL;
    const RingDims &d = r->d;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess)
        e = cudaMemcpy(out, r->m.flags + ((size_t)seq * d.n_kinds + mask_kind) * d.n_tiles,
                       d.n_tiles, cudaMemcpyDeviceToHost);
    return e == cudaSuccess ? RING_OK : cuda_fail(r, e, "ring_get_tile_flags");
}

int ring_get_kv(ring_t *r, int32_t seq, int32_t layer, uint16_t *k, uint16_t *v) {
    if (!check_seq(r, seq) || layer < 0 || layer >= r->d.n_layer) return RING_EINVAL;
    const RingDims &d = r->d;
    if (d.kv_q8) return fail(r, RING_ESTATE, "ring_get_kv: the ring holds q8_0 slots (ring_get_kv_q8)");
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(r, e, "ring_get_kv");
    // device [kv head][slot][head_dim] -> host [slot][kv head * head_dim]
    const size_t head_elems = (size_t)d.kv_total * d.head_dim;
    for (int t = 0; t < 2; ++t) {
        uint16_t *dst = t == 0 ? k : v;
        if (!dst) continue;
        const uint16_t *src = (t == 0 ? r->m.k : r->m.v) +
                              ((size_t)seq * d.n_layer + layer) * d.n_head_kv * head_elems;
        e = cudaMemcpy2D(dst, (size_t)d.kv_row * 2, src, (size_t)d.head_dim * 2,
                         (size_t)d.head_dim * 2, d.kv_total, cudaMemcpyDeviceToHost);
        for (int g = 1; g < d.n_head_kv && e == cudaSuccess; ++g)
            e = cudaMemcpy2D(dst + (size_t)g * d.head_dim, (size_t)d.kv_row * 2,
                             src + g * head_elems, (size_t)d.head_dim * 2, (size_t)d.head_dim * 2,
                             d.kv_total, cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) return cuda_fail(r, e, "ring_get_kv");
    }
    return RING_OK;
}

int ring_get_kv_q8(ring_t *r, int32_t seq, int32_t layer, int8_t *k_codes, uint16_t *k_scales,
                   int8_t *v_codes, uint16_t *v_scales) {
    if (!check_seq(r, seq) || layer < 0 || layer >= r->d.n_layer) return RING_EINVAL;
    const RingDims &d = r->d;
    if (!d.kv_q8) return fail(r, RING_ESTATE, "ring_get_kv_q8: the ring holds F16 slots");
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(r, e, "ring_get_kv_q8");
    // device [kv head][slot][x] -> host [slot][kv head * x], x = 128 codes or 4 scales
    const size_t plane = (size_t)(seq * d.n_layer + layer) * d.n_head_kv;
    for (int t = 0; t < 4 && e == cudaSuccess; ++t) {
        void *dst = t == 0 ? (void *)k_codes : t == 1 ? (void *)k_scales : t == 2 ? (void *)v_codes
                                                                                  : (void *)v_scales;
        if (!dst) continue;
        const bool codes = t % 2 == 0;
        const size_t width = codes ? (size_t)d.head_dim : (size_t)d.head_dim / 32;   // per head
        const size_t esz = codes ? 1 : 2;
        const uint8_t *base = codes ? reinterpret_cast<const uint8_t *>(t == 0 ? r->m.kq : r->m.vq)
                                    : reinterpret_cast<const uint8_t *>(t == 1 ? r->m.ks : r->m.vs);
        for (int g = 0; g < d.n_head_kv && e == cudaSuccess; ++g)
            e = cudaMemcpy2D(static_cast<uint8_t *>(dst) + g * width * esz, width * d.n_head_kv * esz,
                             base + ((plane + g) * d.kv_total) * width * esz, width * esz,
                             width * esz, d.kv_total, cudaMemcpyDeviceToHost);
    }
    if (e != cudaSuccess) return cuda_fail(r, e, "ring_get_kv_q8");
    return RING_OK;
}

int ring_device_error(ring_t *r, uint32_t *bits) {
    if (!r) return RING_EINVAL;
    uint32_t w = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(&w, r->m.err, 4, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && w) e = cudaMemset(r->m.err, 0, 4);
    if (e != cudaSuccess) return cuda_fail(r, e, "ring_device_error");
    if (bits) *bits = w;
    if (w) return fail(r, RING_EDEVICE, "device error word 0x%x", w);
    return RING_OK;
}

int ring_describe(const ring_t *r, char *buf, size_t len) {
    if (!r || !buf || !len) return RING_EINVAL;
    const RingDims &d = r->d;
    // F16: 2 bytes a value; q8_0: 34 bytes per 32 values (codes + one F16 scale)
    const double row_bytes = d.kv_q8 ? d.kv_row + d.kv_row / 32 * 2.0 : d.kv_row * 2.0;
    const double mib = 2.0 * d.n_layer * row_bytes * d.kv_total / 1048576.0;
    snprintf(buf, len,
             "[draft-kv] ctx-KV ring active: cap=%d kv_total=%d a_step=%d layers=%d %s cache %.1f MiB",
             d.cap, d.kv_total, d.a_step, d.n_layer, d.kv_q8 ? "q8_0" : "f16", mib);
    return RING_OK;
}

int ring_profile_enable(ring_t *r, int32_t on) {
    if (!r) return RING_EINVAL;
    r->profiling = on != 0;
    return RING_OK;
}

int ring_profile_read(ring_t *r, ring_profile *out) {
    if (!r || !out) return RING_EINVAL;
    for (auto &rec : r->recs) {
        cudaError_t e = cudaEventSynchronize(rec.b);
        if (e != cudaSuccess) return cuda_fail(r, e, "ring_profile_read");
        float ms = 0.f;
        cudaEventElapsedTime(&ms, rec.a, rec.b);
        if (rec.cls >= 0 && rec.cls < kKinds) {
            out->launches[rec.cls] += 1;
            out->total_ms[rec.cls] += ms;
        }
        r->ev_pool.push_back(rec.a);
        r->ev_pool.push_back(rec.b);
    }
    r->recs.clear();
    return RING_OK;
}

int64_t ring_launch_count(const ring_t *r) { return r ? r->launches : 0; }

int ring_clock_enable(ring_t *r, int32_t on) {
    if (!r) return RING_EINVAL;
    r->clock_on = on != 0;
    r->m.clock = r->clock_on ? r->clock_buf : nullptr;
    return RING_OK;
}

int ring_clock_read(ring_t *r, int32_t kind, double *total_ms, int64_t *launches) {
    if (!r) return RING_EINVAL;
    if (kind < 0 || kind >= kClockKinds)
        return fail(r, RING_EINVAL, "ring_clock_read: kind %d outside [0, %d)", kind, kClockKinds);
    const size_t bank = (size_t)kClockKinds * kClockSlots;
    unsigned long long *t0w = r->clock_buf + (size_t)kind * kClockSlots;
    unsigned long long *t1w = r->clock_buf + bank + (size_t)kind * kClockSlots;
    std::vector<unsigned long long> w(2 * (size_t)kClockSlots);
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess)
        e = cudaMemcpy(w.data(), t0w, (size_t)kClockSlots * 8, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess)
        e = cudaMemcpy(w.data() + kClockSlots, t1w, (size_t)kClockSlots * 8, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(t0w, 0xff, (size_t)kClockSlots * 8);
    if (e == cudaSuccess) e = cudaMemset(t1w, 0, (size_t)kClockSlots * 8);
    if (e != cudaSuccess) return cuda_fail(r, e, "ring_clock_read");
    double ns = 0.0;
    int64_t n = 0;
    for (int s = 0; s < kClockSlots; ++s) {
        const unsigned long long t0 = w[s], t1 = w[kClockSlots + s];
        if (t0 != ~0ull && t1 >= t0) {
            ns += (double)(t1 - t0);
            ++n;
        }
    }
    if (total_ms) *total_ms = ns * 1e-6;
    if (launches) *launches = n;
    return RING_OK;
}

int ring_check_bounded_wait(ring_t *r, int32_t which, int32_t limit_us, void *stream) {
    if (!r) return RING_EINVAL;
    if (which != 0 && which != 1)
        return fail(r, RING_EINVAL, "ring_check_bounded_wait: which must be 0 or 1, got %d", which);
    if (limit_us < 1 || limit_us > 2000000)
        return fail(r, RING_EINVAL, "ring_check_bounded_wait: limit %d us outside [1, 2e6]", limit_us);
    cudaError_t e = launch_wait_probe(r->m, which, (unsigned long long)limit_us * 1000ull,
                                      static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(r, e, "ring_check_bounded_wait: launch");
    ++r->launches;
    return RING_OK;
}

const char *ring_last_error(const ring_t *r) {
    return r ? r->err.c_str() : g_init_error.c_str();
}

}  // extern "C"
