// Every layer's attention of one step in one persistent kernel (few sequences).
//
// Page "DFLASH2_RING_PORT.md", sections 1.4-1.6: after begin_step every layer attends its
// q_len noise queries over the same slot map; the step is one fixed graph replayed every
// step, and the layers run in order.  With few (sequence, kv head) pairs one layer moves
// ~17 MB at cap 4096 -- a few microseconds of HBM time -- so launching the layers one by
// one leaves the GPU waiting on per-layer chains of dependent work.  This kernel keeps
// one CTA per SM for the whole step instead:
//
//   * Each pair is one thread-block cluster of `c` CTAs; cluster rank j serves the j-th of
//     c equal chunks of the pair's visible 64-slot tiles (the same chunk in every layer:
//     tile flags do not depend on the layer).
//   * Its producer warp streams the chunk's tiles of layer 0, 1, 2, ... through a ring of
//     shared-memory stages by TMA without waiting for the layers: every layer's context
//     K/V is final once begin_step has run.  Only a tile holding the layer's noise slots
//     waits for the consumers to have written that layer's noise rows.
//   * Its consumer warps run the layers strictly in order.  Layer l starts (reads its
//     queries and noise rows) only once every CTA has finished layer l-1's output, as a
//     drafter's layer l needs layer l-1's result: a grid-wide counter, polled with a
//     bounded wait.  Within a layer, warp pair k takes every fourth tile of the chunk
//     (16 query rows per warp, all 64 keys of the tile), so the chunk's tiles are worked
//     on side by side.  The four pairs' softmax states merge in shared memory; the CTA's
//     state of each query row is then pushed into the shared memory of the cluster CTA
//     that owns the row (distributed shared memory, announced by a remote mbarrier
//     arrival), and each CTA merges the c states of its rows and writes their outputs.
//
// The launch is cooperative (every CTA resident at once), so CTAs may wait on each
// other; every wait is bounded (2 s) and a CTA that gives up raises a grid-wide abort
// flag and the device error word, so the others stop too.
#include "ring_internal.h"
#include "ptx.h"

#include <cuda_fp16.h>

namespace dflash {
namespace {

constexpr int kCW = 8;                           // consumer warps: 4 pairs x 2 row blocks
constexpr int kConsumers = kCW * 32;
constexpr int kThreads = kConsumers + 32;        // + one producer warp
constexpr int kStages = 5;
constexpr int kTileBytes = kTile * kHeadDim * 2;  // K or V of one 64-slot tile (16 KiB)
constexpr int kHalfBox = kTileBytes / 2;          // TMA box: 64 slots x 64 columns
constexpr int kStageBytes = 2 * kTileBytes;
constexpr int kQBytes = kRows * kHeadDim * 2;
constexpr int kBitsPerStage = kMaxQWords * 8;
constexpr int kXPer = 68 * 32;                   // one warp's state: 64 numerators + 2 max + 2 sum per lane
constexpr int kOffQ = kStages * kStageBytes;
constexpr int kOffX = kOffQ + kQBytes;           // merge scratch [2 slots][2 row blocks][kXPer]
constexpr int kXBytes = 2 * 2 * kXPer * 4;
constexpr int kOffBits = kOffX + kXBytes;
constexpr int kOffFlags = kOffBits + kStages * kBitsPerStage;
// receive buffer: for each source CTA of the cluster, the state of each row this CTA owns
// -- 128 numerators, max, sum (rows padded to 132 floats, 16-byte aligned)
constexpr int kRecvStride = 132;
constexpr int kOffRecv = kOffFlags + kMaxStepTiles;
constexpr int kOffBars = kOffRecv + kMaxRecvSlots * kRecvStride * 4;
constexpr int kSmem = 1024 + kOffBars + (2 * kStages + 2) * 8;
static_assert(kOffQ % 1024 == 0, "query tile keeps the 128-byte swizzle's 1024-byte alignment");
static_assert(kOffRecv % 16 == 0, "receive rows are read as float4");
static_assert(kSmem <= 227 * 1024, "dynamic shared memory of one CTA");

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_add(uint32_t *p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Spin until *ctr >= target: false once limit_ns have passed or another CTA raised the
// abort flag.  Called by one thread.
__device__ bool wait_count(const uint32_t *ctr, uint32_t target, const uint32_t *abort,
                           uint64_t limit_ns) {
    if (ld_acquire(ctr) >= target) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t it = 1; it < (1u << 30); ++it) {
        if (ld_acquire(ctr) >= target) return true;
        if ((it & 63u) == 0) {
            if (ld_acquire(abort) != 0u) return false;
            if (global_ns() - t0 > limit_ns) return false;
        }
    }
    return false;
}

struct StepSync {
    uint32_t *layer_ctr;   // [n_layer]  CTAs done with that layer's outputs
    uint32_t *abort;       // [1]        a CTA gave up on a bounded wait
};

__device__ __forceinline__ StepSync step_sync(const RingDev &m, int n_layer) {
    StepSync y;
    y.layer_ctr = m.step_sync;
    y.abort = m.step_sync + n_layer;
    return y;
}


// ---------------------------------------------------------------------------------
// Grid: pairs * c CTAs in clusters of c (cooperative, one CTA per SM), kThreads threads.
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1)
k_attend_step(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
              RingDims d, RingDev m, int kind, float scale_log2, StepIO io) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sq = smem + kOffQ;
    float *xs = reinterpret_cast<float *>(smem + kOffX);
    const uint64_t *sbits = reinterpret_cast<const uint64_t *>(smem + kOffBits);
    uint8_t *sflags = smem + kOffFlags;
    float *recv = reinterpret_cast<float *>(smem + kOffRecv);
    // full[0..S-1], empty[0..S-1], noise rows written, cluster states received
    const uint32_t bar0 = smem_u32(smem + kOffBars);
    const uint32_t noise_bar = bar0 + 16 * kStages, recv_bar = noise_bar + 8;
    __shared__ int s_tb, s_te, s_nmine, s_ok;
    // set only by consumer warps (a stage load they waited for never came), read by the
    // consumers after a consumer barrier -- so they all take the same branch -- and by
    // the producer, which then stops issuing
    __shared__ volatile int s_cfail;

    const int n_split = (int)cluster_size(), j = (int)cluster_rank();
    const int pr = blockIdx.x / n_split;
    const int rmax = (kRows + n_split - 1) / n_split;   // rows a cluster rank owns, at most
    const int s = pr / d.n_head_kv, gk = pr % d.n_head_kv;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tn0 = d.cap / kTile, tn1 = (d.cap + d.q_len - 1) / kTile;
    const int64_t fbase = ((int64_t)s * d.n_kinds + kind) * d.n_tiles;
    const int qw = (d.q_len + 1) & ~1;
    const StepSync ys = step_sync(m, d.n_layer);

    if (threadIdx.x == 0) {
        for (int k = 0; k < kStages; ++k) {
            mbar_init(bar0 + 8 * k, 1);
            mbar_init(bar0 + 8 * (kStages + k), 2);     // the two warps of the pair that used it
        }
        mbar_init(noise_bar, kCW);
        mbar_init(recv_bar, 4 * n_split);            // four pushing warps of every cluster CTA
        s_cfail = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    // every CTA of the cluster has initialised its barriers before any remote access
    cluster_arrive_relaxed();
    cluster_wait();
    // Everything below reads ring state written by begin_step.
    pdl_wait();
    int clk_slot = 0;     // kernel clock slot of this launch (thread 0)
    if (threadIdx.x == 0 && m.clock) clk_slot = clock_start(m.clock, kClockAttend, 0);

    // This CTA's chunk of the visible tiles: [vb, ve) in visible order, raw range [tb, te).
    for (int t = threadIdx.x; t < d.n_tiles; t += kThreads) sflags[t] = m.flags[fbase + t];
    __syncthreads();
    if (warp == 0) {
        int n_vis = 0;
        for (int c0 = 0; c0 < d.n_tiles; c0 += 32)
            n_vis += __popc(__ballot_sync(0xffffffffu, c0 + lane < d.n_tiles && sflags[c0 + lane] != 0));
        const int vb = (int)((int64_t)j * n_vis / n_split), ve = (int)((int64_t)(j + 1) * n_vis / n_split);
        // raw index of the k-th visible tile (k counted from 0) within a chunk of 32 flags
        // whose visible-tile bits are v: the lane holding a visible tile with k visible
        // tiles below it
        auto kth = [&](uint32_t v, int k) {
            const bool hit = ((v >> lane) & 1u) && __popc(v & ((1u << lane) - 1u)) == k;
            return __ffs(__ballot_sync(0xffffffffu, hit)) - 1;
        };
        int seen = 0, tb = d.n_tiles, te = d.n_tiles;
        for (int c0 = 0; c0 < d.n_tiles; c0 += 32) {
            const uint32_t v = __ballot_sync(0xffffffffu, c0 + lane < d.n_tiles && sflags[c0 + lane] != 0);
            const int n = __popc(v);
            if (tb == d.n_tiles && vb < seen + n) tb = c0 + kth(v, vb - seen);
            if (te == d.n_tiles && ve < seen + n) te = c0 + kth(v, ve - seen);
            seen += n;
        }
        if (vb >= n_vis) tb = te = d.n_tiles;
        if (lane == 0) {
            s_tb = tb;
            s_te = te;
            s_nmine = ve - vb;
        }
    }
    __syncthreads();
    const int tb = s_tb, te = s_te, n_mine = s_nmine;
    const bool owns_noise = tb < te && tb <= tn1 && te > tn0;

    if (warp == kCW) {
        // ---------------- producer: every layer's tiles of this chunk, in order ----------------
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (int l = 0; l < d.n_layer && ok; ++l) {
                const int zrow = (s * d.n_layer + l) * d.n_head_kv + gk;
                bool noise_ready = false;
                for (int t = tb; t < te && ok; ++t) {
                    const int flag = sflags[t];
                    if (flag == 0) continue;
                    if (!noise_ready && t >= tn0 && t <= tn1) {
                        // this layer's noise rows are in its slots (written by the consumers)
                        if (!mbar_wait(noise_bar, (uint32_t)l & 1u)) {
                            atomicOr(m.err, kErrWaitNoise);
                            ok = false;
                            break;
                        }
                        noise_ready = true;
                    }
                    const int stg = it % kStages;
                    if (!mbar_wait(bar0 + 8 * (kStages + stg), ((uint32_t)(it / kStages) & 1u) ^ 1u)) {
                        atomicOr(m.err, kErrWaitEmpty);
                        ok = false;
                        break;
                    }
                    if (s_cfail) {
                        ok = false;
                        break;
                    }
                    const uint32_t full = bar0 + 8 * stg;
                    const uint32_t dk = smem_u32(smem + stg * kStageBytes), dv = dk + kTileBytes;
                    const uint32_t nbits = flag == 2 ? (uint32_t)qw * 8u : 0u;
                    mbar_expect_tx(full, kStageBytes + nbits);
                    tma_load_3d(dk, &tm_k, 0, t * kTile, zrow, full);
                    tma_load_3d(dk + kHalfBox, &tm_k, 64, t * kTile, zrow, full);
                    tma_load_3d(dv, &tm_v, 0, t * kTile, zrow, full);
                    tma_load_3d(dv + kHalfBox, &tm_v, 64, t * kTile, zrow, full);
                    if (nbits)
                        bulk_g2s(smem_u32(smem + kOffBits + stg * kBitsPerStage),
                                 m.maskbits + (fbase + t) * qw, nbits, full);
                    ++it;
                }
            }
            if (!ok) atomicExch(ys.abort, 1u);
            // no copy may land after the CTA exits: wait for the last load of every stage
            for (int k = max(0, it - kStages); k < it; ++k) {
                if (!mbar_wait(bar0 + 8 * (k % kStages), (uint32_t)(k / kStages) & 1u)) {
                    atomicOr(m.err, kErrDrain);
                    break;
                }
            }
        }
        __syncwarp();
        cluster_sync();      // peers may still push into this CTA's shared memory
        return;
    }

    // ---------------- consumers ----------------
    const int tid = threadIdx.x;
    const int half = kHeadDim / 2;
    const float2 *csq = m.rope32 + (int64_t)s * d.q_len * half;
    const int kp = warp >> 1, mb = warp & 1;
    const int g = lane >> 2, c = lane & 3;
    const int r0 = mb * 16 + g, r1 = r0 + 8;
    const int i0 = r0 < d.rows ? r0 % d.q_len : 0;
    const int i1 = r1 < d.rows ? r1 % d.q_len : 0;
    int it_base = 0;     // stage index of this layer's first tile
    bool alive = true;

    // one thread waits, the rest meet it at the consumer barrier; false: give up
    auto sync_wait = [&](const uint32_t *ctr, uint32_t target) -> bool {
        if (tid == 0) {
            const bool ok = wait_count(ctr, target, ys.abort, kWaitNs);
            if (!ok) {
                atomicOr(m.err, kErrWaitPeer);
                atomicExch(ys.abort, 1u);
            }
            __threadfence();
            s_ok = ok ? 1 : 0;
        }
        bar_sync(1, kConsumers);
        return s_ok != 0;
    };

    for (int l = 0; l < d.n_layer && alive; ++l) {
        if (l > 0 && !sync_wait(ys.layer_ctr + (l - 1), gridDim.x)) {
            alive = false;
            break;
        }
        const float *q = io.q[l];
        {   // queries of this kv head, RoPE at committed + i, F16, swizzled like the K tiles
            constexpr int kPer = kRows * (kHeadDim / 2) / 4 / kConsumers;
            float4 xa[kPer], xb[kPer], ca[kPer], cb[kPer];
#pragma unroll
            for (int b = 0; b < kPer; ++b) {
                const int u = b * kConsumers + tid;
                const int r = u >> 4, j0 = (u & 15) * 4;
                if (r < d.rows) {
                    const int hh = r / d.q_len, i = r - hh * d.q_len;
                    const float *qs = q + (((int64_t)s * d.q_len + i) * d.n_head + gk * d.group + hh) * kHeadDim;
                    // at L2: a layer's queries may be the previous layer's output, written by
                    // other CTAs of this kernel
                    xa[b] = __ldcg(reinterpret_cast<const float4 *>(qs + j0));
                    xb[b] = __ldcg(reinterpret_cast<const float4 *>(qs + j0 + half));
                    ca[b] = *reinterpret_cast<const float4 *>(csq + i * half + j0);
                    cb[b] = *reinterpret_cast<const float4 *>(csq + i * half + j0 + 2);
                } else {
                    xa[b] = xb[b] = ca[b] = cb[b] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
#pragma unroll
            for (int b = 0; b < kPer; ++b) {
                const int u = b * kConsumers + tid;
                const int r = u >> 4, j0 = (u & 15) * 4;
                const float x1[4] = {xa[b].x, xa[b].y, xa[b].z, xa[b].w};
                const float x2[4] = {xb[b].x, xb[b].y, xb[b].z, xb[b].w};
                const float cc[4] = {ca[b].x, ca[b].z, cb[b].x, cb[b].z};
                const float sn[4] = {ca[b].y, ca[b].w, cb[b].y, cb[b].w};
                __half2 lo[2], hi[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    lo[e] = __floats2half2_rn(fmaf(x1[2 * e], cc[2 * e], -x2[2 * e] * sn[2 * e]),
                                              fmaf(x1[2 * e + 1], cc[2 * e + 1], -x2[2 * e + 1] * sn[2 * e + 1]));
                    hi[e] = __floats2half2_rn(fmaf(x1[2 * e], sn[2 * e], x2[2 * e] * cc[2 * e]),
                                              fmaf(x1[2 * e + 1], sn[2 * e + 1], x2[2 * e + 1] * cc[2 * e + 1]));
                }
                *reinterpret_cast<uint2 *>(sq + swz(r, j0 & ~7, kRows) + (j0 & 7) * 2) =
                    *reinterpret_cast<const uint2 *>(lo);
                *reinterpret_cast<uint2 *>(sq + swz(r, (j0 + half) & ~7, kRows) + (j0 & 7) * 2) =
                    *reinterpret_cast<const uint2 *>(hi);
            }
        }
        if (owns_noise) {
            // noise block of this head and layer: K turned at committed + i, V copied, into
            // slots cap + i; then the producer may fetch the tile that holds them
            const uint16_t *k_noise = io.k_noise[l], *v_noise = io.v_noise[l];
            const int64_t head = ((int64_t)s * d.n_layer + l) * d.n_head_kv + gk;
            const int n_items = d.q_len * (half / 8);
            for (int u = tid; u < n_items; u += kConsumers) {
                const int i = u / (half / 8), jc = u - i * (half / 8);
                const uint16_t *ks = k_noise + ((int64_t)s * d.q_len + i) * d.kv_row + gk * kHeadDim + jc * 8;
                const uint16_t *vs = v_noise + ((int64_t)s * d.q_len + i) * d.kv_row + gk * kHeadDim + jc * 8;
                const uint4 a = __ldcg(reinterpret_cast<const uint4 *>(ks));
                const uint4 bq = __ldcg(reinterpret_cast<const uint4 *>(ks + half));
                const uint4 va = __ldcg(reinterpret_cast<const uint4 *>(vs));
                const uint4 vb = __ldcg(reinterpret_cast<const uint4 *>(vs + half));
                float2 cs8[8];
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    const float4 t4 = *reinterpret_cast<const float4 *>(csq + i * half + jc * 8 + e);
                    cs8[e] = make_float2(t4.x, t4.y);
                    cs8[e + 1] = make_float2(t4.z, t4.w);
                }
                const uint16_t *a16 = reinterpret_cast<const uint16_t *>(&a);
                const uint16_t *b16 = reinterpret_cast<const uint16_t *>(&bq);
                uint4 ya, yb;
                uint16_t *ya16 = reinterpret_cast<uint16_t *>(&ya);
                uint16_t *yb16 = reinterpret_cast<uint16_t *>(&yb);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float2 rr = rope_rotate(a16[e], b16[e], cs8[e]);
                    ya16[e] = __half_as_ushort(__float2half_rn(rr.x));
                    yb16[e] = __half_as_ushort(__float2half_rn(rr.y));
                }
                const int64_t dst = (head * d.kv_total + d.cap + i) * kHeadDim + jc * 8;
                *reinterpret_cast<uint4 *>(m.k + dst) = ya;
                *reinterpret_cast<uint4 *>(m.k + dst + half) = yb;
                *reinterpret_cast<uint4 *>(m.v + dst) = va;
                *reinterpret_cast<uint4 *>(m.v + dst + half) = vb;
            }
            // generic-proxy stores, then the TMA (async proxy) reads them
            asm volatile("fence.proxy.async.global;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(noise_bar);
        }
        bar_sync(1, kConsumers);      // the query tile is complete

        uint32_t qf[8][4];
        {
            const uint32_t sqa = smem_u32(sq);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                ldsm_x4(sqa + swz(mb * 16 + (lane & 15), ks * 16 + ((lane >> 4) << 3), kRows),
                        qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
        }
        float oacc[16][4];
#pragma unroll
        for (int n = 0; n < 16; ++n) oacc[n][0] = oacc[n][1] = oacc[n][2] = oacc[n][3] = 0.f;
        float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};

        // this pair's tiles: the v-th visible tile of the chunk with v % 4 == kp
        int v = 0;
        for (int t = tb; t < te; ++t) {
            const int flag = sflags[t];
            if (flag == 0) continue;
            const int vi = v++;
            if ((vi & 3) != kp) continue;
            const int itg = it_base + vi;
            const int stg = itg % kStages;
            if (!__all_sync(0xffffffffu, mbar_wait(bar0 + 8 * stg, (uint32_t)(itg / kStages) & 1u))) {
                if (lane == 0) atomicOr(m.err, kErrWaitFull);
                s_cfail = 1;
                break;
            }
            const uint32_t sk = smem_u32(smem + stg * kStageBytes), sv = sk + kTileBytes;
            float sc[8][4];
#pragma unroll
            for (int n = 0; n < 8; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
            // S = Q K^T over the tile's 64 keys (two n-tiles of 8 keys per ldmatrix)
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    const int key = np * 16 + (lane & 7) + ((lane >> 4) << 3);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(sk + swz(key, ks * 16 + (((lane >> 3) & 1) << 3), kTile), b0, b1, b2, b3);
                    mma16816(sc[np * 2], qf[ks], b0, b1);
                    mma16816(sc[np * 2 + 1], qf[ks], b2, b3);
                }
            }
#pragma unroll
            for (int n = 0; n < 8; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) sc[n][e] *= scale_log2;
            if (flag == 2) {
                const uint64_t w0 = sbits[stg * kMaxQWords + i0];
                const uint64_t w1 = sbits[stg * kMaxQWords + i1];
#pragma unroll
                for (int n = 0; n < 8; ++n)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int bit = n * 8 + 2 * c + e;
                        if (!((w0 >> bit) & 1ull)) sc[n][e] = -INFINITY;
                        if (!((w1 >> bit) & 1ull)) sc[n][2 + e] = -INFINITY;
                    }
            }
            // online softmax in the log2 domain, rows r0 (jj = 0) and r1 (jj = 1)
            float alpha[2];
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                float mx = -INFINITY;
#pragma unroll
                for (int n = 0; n < 8; ++n) mx = fmaxf(mx, fmaxf(sc[n][2 * jj], sc[n][2 * jj + 1]));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const float mnew = fmaxf(mrow[jj], mx);
                const float muse = mnew == -INFINITY ? 0.f : mnew;
                alpha[jj] = exp2f(mrow[jj] - muse);
                mrow[jj] = mnew;
                float rs = 0.f;
#pragma unroll
                for (int n = 0; n < 8; ++n) {
                    const float p0 = exp2f(sc[n][2 * jj] - muse);
                    const float p1 = exp2f(sc[n][2 * jj + 1] - muse);
                    sc[n][2 * jj] = p0;
                    sc[n][2 * jj + 1] = p1;
                    rs += p0 + p1;
                }
                lrow[jj] = lrow[jj] * alpha[jj] + rs;
            }
            if (!__all_sync(0xffffffffu, alpha[0] == 1.f && alpha[1] == 1.f)) {
#pragma unroll
                for (int n = 0; n < 16; ++n) {
                    oacc[n][0] *= alpha[0];
                    oacc[n][1] *= alpha[0];
                    oacc[n][2] *= alpha[1];
                    oacc[n][3] *= alpha[1];
                }
            }
            // O += P V, 16 keys per k step
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                uint32_t pa[4];
                pa[0] = pack_half2(sc[2 * kk][0], sc[2 * kk][1]);
                pa[1] = pack_half2(sc[2 * kk][2], sc[2 * kk][3]);
                pa[2] = pack_half2(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
                pa[3] = pack_half2(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
                const int key = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
                for (int dp = 0; dp < 8; ++dp) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(sv + swz(key, dp * 16 + ((lane >> 4) << 3), kTile), b0, b1, b2, b3);
                    mma16816(oacc[dp * 2], pa, b0, b1);
                    mma16816(oacc[dp * 2 + 1], pa, b2, b3);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar0 + 8 * (kStages + stg));
        }
        it_base += n_mine;
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
            lrow[jj] += __shfl_xor_sync(0xffffffffu, lrow[jj], 1);
            lrow[jj] += __shfl_xor_sync(0xffffffffu, lrow[jj], 2);
        }

        // ---- merge the four pairs' states of each row block: pairs 2, 3 into 0, 1; then
        // pairs 0 and 1 each finish half of the 128 columns from the other's half ----
        // numerator groups n0 .. n0 + nn - 1 (8 columns each) and the row's (max, sum)
        auto put = [&](int slot, int n0, int nn) {
            float *x = xs + (slot * 2 + mb) * kXPer;
#pragma unroll
            for (int n = 0; n < 16; ++n)
                if (n >= n0 && n < n0 + nn)
#pragma unroll
                    for (int e = 0; e < 4; ++e) x[((n - n0) * 4 + e) * 32 + lane] = oacc[n][e];
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                x[(64 + jj) * 32 + lane] = mrow[jj];
                x[(66 + jj) * 32 + lane] = lrow[jj];
            }
        };
        auto take = [&](int slot, int n0, int nn) {
            const float *x = xs + (slot * 2 + mb) * kXPer;
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const float m1 = x[(64 + jj) * 32 + lane], l1 = x[(66 + jj) * 32 + lane];
                const float mm = fmaxf(mrow[jj], m1);
                const float muse = mm == -INFINITY ? 0.f : mm;
                const float a0 = exp2f(mrow[jj] - muse), a1 = exp2f(m1 - muse);
                lrow[jj] = lrow[jj] * a0 + l1 * a1;
                mrow[jj] = mm;
#pragma unroll
                for (int n = 0; n < 16; ++n)
                    if (n >= n0 && n < n0 + nn) {
                        oacc[n][2 * jj] = oacc[n][2 * jj] * a0 + x[((n - n0) * 4 + 2 * jj) * 32 + lane] * a1;
                        oacc[n][2 * jj + 1] = oacc[n][2 * jj + 1] * a0 + x[((n - n0) * 4 + 2 * jj + 1) * 32 + lane] * a1;
                    }
            }
        };
        bar_sync(1, kConsumers);          // every warp is past its tiles (and past reading xs)
        if (s_cfail) {
            alive = false;
            break;
        }
        if (kp >= 2) put(kp - 2, 0, 16);
        bar_sync(1, kConsumers);
        const int h0 = kp == 0 ? 0 : 8;   // pair 0 finishes columns 0-63, pair 1 columns 64-127
        if (kp < 2) {
            take(kp, 0, 16);
            put(kp, 8 - h0, 8);           // the half the other pair finishes (own slot: read above)
        }
        bar_sync(1, kConsumers);
        if (kp < 2) {
            take(1 - kp, h0, 8);
            // push this CTA's state of rows r0, r1 -- this pair's half of the columns, and
            // (pair 0) the row's max and sum -- into the CTA of the cluster that owns each
            // row: slot (this rank, row within the owner's rows) of its receive buffer
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const int r = jj ? r1 : r0;
                const int owner = r * n_split / kRows, lr = r - cluster_first_row(owner, n_split);
                const uint32_t dst = map_rank(smem_u32(recv + (j * rmax + lr) * kRecvStride), (uint32_t)owner);
#pragma unroll
                for (int n = 0; n < 16; ++n)
                    if (n >= h0 && n < h0 + 8)
                        st_cluster_v2(dst + 4u * (n * 8 + 2 * c), oacc[n][2 * jj], oacc[n][2 * jj + 1]);
                if (kp == 0 && c == 0) st_cluster_v2(dst + 4u * kHeadDim, mrow[jj], lrow[jj]);
            }
            // the warp's stores are ordered before the arrivals, whose release makes them
            // visible to the owner's acquiring wait; every pushing warp announces itself
            // to every CTA of the cluster (4 per CTA)
            __syncwarp();
            if (lane < n_split) mbar_arrive_remote(map_rank(recv_bar, (uint32_t)lane));
        }
        // ---- the states of this CTA's rows from every CTA of the cluster ----
        if (!mbar_wait_cluster(recv_bar, (uint32_t)l & 1u)) {
            if (lane == 0) atomicOr(m.err, kErrWaitPeer);
            s_cfail = 1;
        }
        bar_sync(1, kConsumers);
        if (s_cfail) {
            alive = false;
            break;
        }
        {
            const int row0 = cluster_first_row(j, n_split);
            const int nrows = min(kRows, cluster_first_row(j + 1, n_split)) - row0;
            float *o = io.o[l];
            for (int u = tid; u < nrows * (kHeadDim / 4); u += kConsumers) {
                const int lr = u / (kHeadDim / 4), c4 = (u % (kHeadDim / 4)) * 4;
                float mm = -INFINITY;
#pragma unroll 4
                for (int p = 0; p < n_split; ++p) mm = fmaxf(mm, recv[(p * rmax + lr) * kRecvStride + kHeadDim]);
                const float muse = mm == -INFINITY ? 0.f : mm;
                float lsum = 0.f;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
                for (int p = 0; p < n_split; ++p) {
                    const float *x = recv + (p * rmax + lr) * kRecvStride;
                    const float w = exp2f(x[kHeadDim] - muse);
                    const float4 v = *reinterpret_cast<const float4 *>(x + c4);
                    lsum += w * x[kHeadDim + 1];
                    acc.x += w * v.x;
                    acc.y += w * v.y;
                    acc.z += w * v.z;
                    acc.w += w * v.w;
                }
                const int r = row0 + lr;
                if (r < d.rows) {
                    const int hh = r / d.q_len, i = r - hh * d.q_len;
                    const int h = gk * d.group + hh;
                    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
                    *reinterpret_cast<float4 *>(o + (((int64_t)s * d.q_len + i) * d.n_head + h) * kHeadDim + c4) =
                        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
                }
            }
        }
        bar_sync(1, kConsumers);
        // release: every consumer's output stores (ordered before it by the barrier) are
        // visible before the count that lets the next layer start
        if (tid == 0) red_release_add(ys.layer_ctr + l, 1u);
    }
    if (!alive && tid == 0) atomicExch(ys.abort, 1u);
    if (tid == 0 && m.clock) clock_stop(m.clock, clk_slot);
    cluster_sync();          // no CTA leaves while a peer may still push into its shared memory
}

// Bounded waits that run out: an mbarrier nobody arrives at, and a counter nobody raises.
// Test-only: each must give up after limit_ns, set its bit in the device error word and
// let the kernel return.
__global__ void k_wait_probe(RingDev m, int which, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (which == 0) {
        if (!__all_sync(0xffffffffu, mbar_wait(b, 0u, limit_ns)) && threadIdx.x == 0)
            atomicOr(m.err, kErrWaitFull);
    } else if (threadIdx.x == 0) {
        // m.probe[0] (the counter) and m.probe[1] (the abort word) stay 0
        if (!wait_count(m.probe, 0xffffffffu, m.probe + 1, limit_ns)) atomicOr(m.err, kErrWaitPeer);
    }
}

}  // namespace

size_t attend_step_smem_bytes() { return (size_t)kSmem; }

cudaError_t attend_step_init() {
    cudaError_t e = cudaFuncSetAttribute(k_attend_step, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_attend_step, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
}

int attend_step_capacity(int cluster) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cluster);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, k_attend_step, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

cudaError_t launch_attend_step(const RingDims &d, const RingDev &m, const CUtensorMap *tm_k,
                               const CUtensorMap *tm_v, int kind, float scale_log2,
                               const StepIO &io, int cluster, bool pdl, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(d.n_seq * d.n_head_kv * cluster);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[3];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    attr[2].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[2].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 3 : 2;
    return cudaLaunchKernelEx(&cfg, k_attend_step, *tm_k, *tm_v, d, m, kind, scale_log2, io);
}

cudaError_t launch_wait_probe(const RingDev &m, int which, unsigned long long limit_ns,
                              cudaStream_t st) {
    k_wait_probe<<<1, 32, 0, st>>>(m, which, limit_ns);
    return cudaGetLastError();
}

}  // namespace dflash
