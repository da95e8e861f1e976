// Masked GQA attention of the noise block over the ring (split-KV flash-decode).
//
// Page "DFLASH2_RING_PORT.md", sections 1.1 and 1.4: the q_len noise queries attend to
// all kv_total slots of the layer's F16 K/V tensors under mask_full or mask_swa.  The
// kernel streams each kv head's visible 64-slot tiles with 3-D TMA boxes into a
// shared-memory ring of stages (128-byte swizzle), guarded by mbarriers.  One producer
// warp issues the copies (plus a 16-byte-aligned bulk copy of the tile's per-row
// visibility bits when the tile is only partly visible); the consumer warps compute
// S = Q K^T and O += P V on the F16 tensor cores (m16n8k16, F32 accumulation) with an
// online softmax in F32 registers (its reference maximum moved lazily where the kernel is
// bound by instruction issue).  All 32 query rows that share a kv head (4 heads x 8
// queries) ride in one CTA, so each K/V byte is read from HBM once per step and layer.
// Tiles whose flag says "no visible slot" are never fetched.
//
// Two shapes of the same kernel:
//   * many (sequence, kv head) pairs -- a multi-wave grid of independent CTAs, 4 consumer
//     warps, two CTAs per SM; each CTA writes a partial softmax state and a combine
//     kernel merges them (unless a pair has a single CTA);
//   * few pairs -- one wave of thread-block clusters, 8 consumer warps per CTA (one CTA
//     per SM, so per-tile latency halves); the warps' key slices are merged in shared
//     memory, each row's CTA state is pushed into the shared memory of the CTA that owns
//     the row (distributed shared memory stores), and after one cluster barrier each CTA
//     finishes 32 / cluster rows locally.
// q8_0 slots (int8 codes + one F16 scale per 32 values) take either shape with 17 KiB
// stages of codes and scales; the consumers turn the codes straight into F16 MMA operands
// in registers (no second pass through shared memory).
#include "ring_internal.h"
#include "ptx.h"

#include <cuda_fp16.h>

namespace dflash {
namespace {

// 2^x on the special-function unit (ex2.approx.ftz: relative error below 2^-22, results
// under 2^-126 flushed to zero), for the probabilities, which are rounded to F16 next
__device__ __forceinline__ float ex2_fast(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

constexpr int kTileBytes = kTile * kHeadDim * 2;   // one 64-slot tile of one head, K or V
constexpr int kHalfBox = kTileBytes / 2;           // TMA box: 64 slots x 64 columns
constexpr int kStageBytes = 2 * kTileBytes;        // K + V
constexpr int kQBytes = kRows * kHeadDim * 2;
constexpr int kBitsPerStage = kMaxQWords * 8;      // visibility words of one tile

// Two shapes of one kernel.  CLUSTER: 8 consumer warps (4 key slices), 6 stages, one CTA
// per SM, partial states pushed to the owning CTA of the cluster.  Plain: 4 consumer warps
// (2 key halves), 3 stages, two CTAs per SM, key halves merged in shared memory and the
// CTA's partial written straight from registers.
template <bool CLUSTER, bool Q8 = false>
struct Shape {
    static constexpr int CW = CLUSTER ? 8 : 4;      // consumer warps
    static constexpr int kConsumers = CW * 32;
    static constexpr int kThreads = kConsumers + 32;
    static constexpr int kStages = CLUSTER ? (Q8 ? 10 : 6) : (Q8 ? 5 : 3);
    static constexpr int kSlices = CW / 2;          // key slices per tile
    static constexpr int kKeys = kTile / kSlices;   // keys per warp per tile (32 or 16)
    static constexpr int kNT = kKeys / 8;           // n-tiles of S per warp
    static constexpr int kKK = kKeys / 16;          // k-steps of P V per warp
    static constexpr int kMinBlocks = CLUSTER ? 1 : 2;
    // how far (log2) a row maximum may outgrow the softmax reference before O and l are
    // rescaled (P stays within [0, 2^kLazyLog2]): the latency- and issue-bound instances
    // skip most rescales; the HBM-bound plain F16 instance keeps the plain online softmax
    // (exact running maximum), which it runs with fewer registers
    static constexpr bool kLazy = CLUSTER || Q8;
    static constexpr float kLazyLog2 = 8.f;
    // q8_0 slots: a stage holds a tile's K and V codes (two 128 x 64-byte TMA boxes) and
    // their scales (2 x 512 bytes); the consumers turn codes into F16 MMA operands in
    // registers, so a stage costs 17 KiB instead of 32 and five (plain) or ten (cluster)
    // of them fit
    static constexpr int kStageBytesT = Q8 ? 2 * kTile * 128 + 2 * kTile * 8 : kStageBytes;
    static constexpr int kOffQ = kStages * kStageBytesT;  // 1024-aligned (swizzled like K)
    static constexpr int kOffBits = kOffQ + kQBytes;
    static constexpr int kOffBars = kOffBits + kStages * kBitsPerStage;
    static constexpr int kOffRecv = kOffBars + 2 * kStages * 8 + 16;
    // cluster receive buffer: one partial per CTA of the cluster for each of the at most
    // ceil(32 / cluster) rows this CTA finishes -- numerators, then (max, sum) per slot
    static constexpr int kRecvAcc = kMaxRecvSlots * kHeadDim * 4;
    static constexpr int kRecvBytes = kRecvAcc + kMaxRecvSlots * 8;
    // key-slice pre-merge scratch (in the idle stage buffers): every warp's partial,
    // 64 numerators + 2 maxima + 2 sums per lane
    static constexpr int kXPer = 68 * 32;
    static_assert(kSlices * 2 * kXPer * 4 <= kStages * kStageBytesT, "pre-merge scratch");
    static_assert(2 * 64 * 32 * 4 + 2 * 2 * 2 * 32 * 4 <= kStages * kStageBytesT,
                  "key-half merge scratch must fit in the idle stage buffers");
    static_assert(kStageBytesT % 1024 == 0, "stages keep TMA boxes 1024-aligned");
    static constexpr int kSmem = 1024 + kOffRecv + (CLUSTER ? kRecvBytes : 0);
    static_assert(kSmem <= 227 * 1024, "dynamic shared memory of one CTA");
};


// ---------------------------------------------------------------------------------
// Split-KV attention of one layer.  Grid (n_splits, n_head_kv, n_seq) in clusters of
// `cluster` CTAs along x; CW consumer warps + one producer warp.
//
//   prologue   consumers turn this kv head's 32 query rows by RoPE at committed + i
//              (float32, the step's cos/sin table) into F16 shared memory; the CTA whose
//              tiles hold the noise slots writes the noise block's K (RoPE at
//              committed + j) and V rows of this head to slots cap + j.  Meanwhile the
//              producer already streams the context tiles.
//   main loop  consumer warp w owns query rows 16*(w & 1) .. +16 and key slice (w >> 1)
//              of every 64-slot tile: S = Q K^T, online softmax, O += P V.
//   merge      without a cluster the two key halves merge in shared memory and the CTA
//              writes O (or its partial for the combine kernel); in a cluster the key
//              slices merge in shared memory, each row's CTA state goes to the receive
//              buffer of the CTA that finishes the row, and after one cluster barrier that
//              CTA merges the cluster's states of its rows and writes O (or a group
//              partial for the combine kernel).
// ---------------------------------------------------------------------------------
template <bool CLUSTER, bool Q8>
__global__ void __launch_bounds__(Shape<CLUSTER, Q8>::kThreads, Shape<CLUSTER, Q8>::kMinBlocks)
k_attend(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
         RingDims d, RingDev m, int layer, int kind, float scale_log2,
         const float *__restrict__ q, const uint16_t *__restrict__ k_noise,
         const uint16_t *__restrict__ v_noise, float *__restrict__ o, int early) {
    using SH = Shape<CLUSTER, Q8>;
    constexpr int CW = SH::CW;
    constexpr int kStageB = SH::kStageBytesT;
    constexpr int kStages = SH::kStages;
    constexpr int kOffQ = SH::kOffQ, kOffBits = SH::kOffBits, kOffBars = SH::kOffBars,
                  kOffRecv = SH::kOffRecv;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sq = smem + kOffQ;
    const uint64_t *sbits = reinterpret_cast<const uint64_t *>(smem + kOffBits);
    const uint32_t bar0 = smem_u32(smem + kOffBars);   // full[0..S-1], then empty[0..S-1]
    __shared__ volatile int s_abort;
    int clk_slot = 0;     // kernel clock slot of this launch (thread 0)

    const uint32_t nct = CLUSTER ? cluster_size() : 1u, rank = CLUSTER ? cluster_rank() : 0u;
    // receive buffer (clusters only): dedicated, since other CTAs of the cluster push into
    // it while this CTA may still be streaming
    float *recv_acc = reinterpret_cast<float *>(smem + kOffRecv);
    float2 *recv_ml = reinterpret_cast<float2 *>(reinterpret_cast<uint8_t *>(recv_acc) + SH::kRecvAcc);
    const int rmax = (kRows + (int)nct - 1) / (int)nct;   // rows a cluster rank finishes, at most

    const int sp = blockIdx.x, gk = blockIdx.y, s = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = sp * d.tiles_per_split;
    const int t1 = min(d.n_tiles, t0 + d.tiles_per_split);
    const int tn0 = d.cap / kTile, tn1 = (d.cap + d.q_len - 1) / kTile;
    const bool owns_noise = t0 < t1 && t0 <= tn1 && t1 > tn0;
    const int64_t fbase = ((int64_t)s * d.n_kinds + kind) * d.n_tiles;
    const uint8_t *flags = m.flags + fbase;
    const int qw = (d.q_len + 1) & ~1;

    if (threadIdx.x == 0) {
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        for (int k = 0; k < kStages; ++k) {
            mbar_init(bar0 + 8 * k, 1);
            mbar_init(bar0 + 8 * (kStages + k), CW);
        }
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    if constexpr (CLUSTER) cluster_arrive_relaxed();

    if (warp == CW) {
        // ---------------- producer ----------------
        // The whole warp walks the tile list (so every barrier it meets is met by all 32
        // lanes together); lane 0 alone waits on the stage barriers and issues the copies.
        const int zrow = (s * d.n_layer + layer) * d.n_head_kv + gk;
        // lane 0: one stage's copies of tile t (F16: four 64 x 64 boxes; q8_0: two 128 x 64
        // code boxes and the scales of the tile's rows), plus its visibility bits
        auto issue = [&](int stg, int t, int flag) {
            const uint32_t full = bar0 + 8 * stg;
            const uint32_t dk = smem_u32(smem + stg * kStageB);
            const uint32_t nbits = flag == 2 ? (uint32_t)qw * 8u : 0u;
            if constexpr (Q8) {
                const int rows = min(kTile, d.kv_total - t * kTile);     // 64 or 32
                mbar_expect_tx(full, 2 * kTile * 128 + 2 * rows * 8 + nbits);
                tma_load_3d(dk, &tm_k, 0, t * kTile, zrow, full);
                tma_load_3d(dk + kTile * 128, &tm_v, 0, t * kTile, zrow, full);
                const int64_t so = ((int64_t)zrow * d.kv_total + (int64_t)t * kTile) * (kHeadDim / 32);
                bulk_g2s(dk + 2 * kTile * 128, m.ks + so, rows * 8, full);
                bulk_g2s(dk + 2 * kTile * 128 + kTile * 8, m.vs + so, rows * 8, full);
            } else {
                const uint32_t dv = dk + kTileBytes;
                mbar_expect_tx(full, kStageBytes + nbits);
                tma_load_3d(dk, &tm_k, 0, t * kTile, zrow, full);
                tma_load_3d(dk + kHalfBox, &tm_k, 64, t * kTile, zrow, full);
                tma_load_3d(dv, &tm_v, 0, t * kTile, zrow, full);
                tma_load_3d(dv + kHalfBox, &tm_v, 64, t * kTile, zrow, full);
            }
            if (nbits)
                bulk_g2s(smem_u32(smem + kOffBits + stg * kBitsPerStage),
                         m.maskbits + (fbase + t) * qw, nbits, full);
        };
        bool noise_ready = false;
        int it = 0;
        // visible tiles of this split in order, 32 flags per load: `pt` is the next tile
        // not yet issued (-1 past the end), `pflag` its flag
        int cbase = t0, pt = -1, pflag = 0;
        uint32_t vis = 0u, part = 0u;
        auto advance = [&]() {
            pt = -1;
            while (vis == 0u) {
                if (cbase >= t1) return;
                const int u = cbase + lane;
                const int f = u < t1 ? (int)flags[u] : 0;
                vis = __ballot_sync(0xffffffffu, f != 0);
                part = __ballot_sync(0xffffffffu, f == 2);
                cbase += 32;
            }
            const int bit = __ffs(vis) - 1;
            vis &= vis - 1u;
            pt = cbase - 32 + bit;
            pflag = ((part >> bit) & 1u) ? 2 : 1;
        };
        {
            // L2 prefetch of this CTA's query rows, the step's RoPE table and the noise
            // rows: a hint only (L2 is coherent), so it is safe whatever runs before
            const int half = kHeadDim / 2;
            for (int u = lane; u < d.rows * 4; u += 32) {
                const int r = u >> 2, hh = r / d.q_len, i = r - hh * d.q_len;
                prefetch_l2(q + (((int64_t)s * d.q_len + i) * d.n_head + gk * d.group + hh) * kHeadDim + (u & 3) * 32);
            }
            for (int u = lane; u < d.q_len * half * 8 / 128; u += 32)
                prefetch_l2(reinterpret_cast<const uint8_t *>(m.rope32 + (int64_t)s * d.q_len * half) + u * 128);
            if (owns_noise)
                for (int u = lane; u < d.q_len * 2; u += 32) {
                    const int i = u >> 1;
                    const uint16_t *base = (u & 1) ? v_noise : k_noise;
                    prefetch_l2(base + ((int64_t)s * d.q_len + i) * d.kv_row + gk * kHeadDim);
                    prefetch_l2(base + ((int64_t)s * d.q_len + i) * d.kv_row + gk * kHeadDim + 64);
                }
        }
        if (early & kAttendPreload) {
            // The kernel before this one (an attention kernel of another layer, or one
            // that does not overlap this grid at all) writes none of this layer's context
            // tiles, flags or bits, so the first stages can be filled before the grid
            // dependency resolves.  The host never asks for this right after begin_step.
            // A tile holding noise slots is not touched before the noise rows are written.
            advance();
            while (pt >= 0 && it < kStages && !(pt >= tn0 && pt <= tn1)) {
                if (lane == 0) issue(it, pt, pflag);
                __syncwarp();
                ++it;
                advance();
            }
        }
        pdl_wait();
        // A grid that fits in one wave lets the next kernel's CTAs settle onto idle SMs
        // now; a multi-wave grid must not, or they would take slots its own later CTAs need.
        if (d.single_wave) pdl_trigger();
        if (!(early & kAttendPreload)) advance();
        for (; pt >= 0; advance()) {
            const int t = pt, flag = pflag;
            if (!noise_ready && t >= tn0 && t <= tn1) {
                __syncwarp();
                bar_sync(2, SH::kThreads);
                noise_ready = true;
            }
            int ok = 1;
            if (lane == 0) {
                const int stg = it % kStages;
                const uint32_t ph = (uint32_t)(it / kStages) & 1u;
                if (!mbar_wait(bar0 + 8 * (kStages + stg), ph ^ 1u)) {
                    atomicOr(m.err, kErrWaitEmpty);
                    s_abort = 1;
                    ok = 0;
                } else if (s_abort) {
                    ok = 0;
                } else {
                    issue(stg, t, flag);
                }
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            ++it;
        }
        if constexpr (CLUSTER) {
            // Every layer's context K/V is final once begin_step has run: with this layer's
            // copies all issued, pull this CTA's tiles of the next layer into L2, so that the
            // next layer's CTAs -- some launch only when this grid's CTAs leave -- find them
            // there.  A hint: the next layer's noise rows, written later, update L2 as usual.
            if (lane == 0 && layer + 1 < d.n_layer && !s_abort) {
                const int zn = zrow + d.n_head_kv;
                for (int u = t0; u < t1; ++u) {
                    if (flags[u] == 0) continue;
                    if constexpr (Q8) {
                        const int rows = min(kTile, d.kv_total - u * kTile);
                        const int64_t so = ((int64_t)zn * d.kv_total + (int64_t)u * kTile) * (kHeadDim / 32);
                        tma_prefetch_3d(&tm_k, 0, u * kTile, zn);
                        tma_prefetch_3d(&tm_v, 0, u * kTile, zn);
                        bulk_prefetch_l2(m.ks + so, rows * 8);
                        bulk_prefetch_l2(m.vs + so, rows * 8);
                    } else {
                        tma_prefetch_3d(&tm_k, 0, u * kTile, zn);
                        tma_prefetch_3d(&tm_k, 64, u * kTile, zn);
                        tma_prefetch_3d(&tm_v, 0, u * kTile, zn);
                        tma_prefetch_3d(&tm_v, 64, u * kTile, zn);
                    }
                }
            }
        }
        __syncwarp();
        if (!noise_ready) bar_sync(2, SH::kThreads);
        if (lane == 0) {
            // No copy may land after the CTA exits: wait for the last load of every stage.
            for (int k = max(0, it - kStages); k < it; ++k) {
                if (!mbar_wait(bar0 + 8 * (k % kStages), (uint32_t)(k / kStages) & 1u)) {
                    atomicOr(m.err, kErrDrain);
                    break;
                }
            }
        }
        __syncwarp();
        if constexpr (CLUSTER) cluster_wait();
    } else {
        // ---------------- consumers ----------------
        // ring state written by begin_step (and earlier kernels) is visible after the grid
        // dependency
        pdl_wait();
        if (d.single_wave) pdl_trigger();
        if (threadIdx.x == 0 && m.clock) clk_slot = clock_start(m.clock, kClockAttend, layer);
        // clusters: the split's first 32 tile flags, loaded now so that the load overlaps
        // the query prologue's
        const int f_first = CLUSTER && t0 + lane < t1 ? (int)flags[t0 + lane] : 0;
        const int tid = threadIdx.x;
        const int half = kHeadDim / 2;
        const float2 *csq = m.rope32 + (int64_t)s * d.q_len * half;
        {   // queries of this kv head, RoPE at committed + i, F16, swizzled like K tiles.
            // Item u = (row, 4 consecutive pairs); every load is issued before any use.
            constexpr int kItems = kRows * (kHeadDim / 2) / 4;          // 512
            constexpr int kPer = kItems / SH::kConsumers;
            float4 xa[kPer], xb[kPer], ca[kPer], cb[kPer];
#pragma unroll
            for (int b = 0; b < kPer; ++b) {
                const int u = b * SH::kConsumers + tid;
                const int r = u >> 4, j0 = (u & 15) * 4;
                if (r < d.rows) {
                    const int hh = r / d.q_len, i = r - hh * d.q_len;
                    const float *qs = q + (((int64_t)s * d.q_len + i) * d.n_head + gk * d.group + hh) * kHeadDim;
                    xa[b] = *reinterpret_cast<const float4 *>(qs + j0);
                    xb[b] = *reinterpret_cast<const float4 *>(qs + j0 + half);
                    ca[b] = *reinterpret_cast<const float4 *>(csq + i * half + j0);
                    cb[b] = *reinterpret_cast<const float4 *>(csq + i * half + j0 + 2);
                } else {
                    xa[b] = xb[b] = ca[b] = cb[b] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
#pragma unroll
            for (int b = 0; b < kPer; ++b) {
                const int u = b * SH::kConsumers + tid;
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
        if (Q8 && owns_noise) {
            // q8_0 slots: the same items, quantised per 32-value block by the four lanes
            // that hold it (every thread runs every round, so the shuffles see full warps)
            const int64_t head = ((int64_t)s * d.n_layer + layer) * d.n_head_kv + gk;
            const int n_items = d.q_len * (half / 8);
            for (int u0 = 0; u0 < n_items; u0 += SH::kConsumers) {
                const int u = u0 + tid;
                const bool okn = u < n_items;
                const int uu = okn ? u : 0;
                const int i = uu / (half / 8), jc = uu - i * (half / 8);
                const uint16_t *ks = k_noise + ((int64_t)s * d.q_len + i) * d.kv_row + gk * kHeadDim + jc * 8;
                const uint16_t *vs = v_noise + ((int64_t)s * d.q_len + i) * d.kv_row + gk * kHeadDim + jc * 8;
                uint4 a = make_uint4(0, 0, 0, 0), bq = a, va = a, vb = a;
                if (okn) {
                    a = *reinterpret_cast<const uint4 *>(ks);
                    bq = *reinterpret_cast<const uint4 *>(ks + half);
                    va = *reinterpret_cast<const uint4 *>(vs);
                    vb = *reinterpret_cast<const uint4 *>(vs + half);
                }
                const uint16_t *a16 = reinterpret_cast<const uint16_t *>(&a);
                const uint16_t *b16 = reinterpret_cast<const uint16_t *>(&bq);
                const uint16_t *va16 = reinterpret_cast<const uint16_t *>(&va);
                const uint16_t *vb16 = reinterpret_cast<const uint16_t *>(&vb);
                float k1[8], k2[8], v1[8], v2[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float2 rr = rope_rotate(a16[e], b16[e], csq[i * half + jc * 8 + e]);
                    k1[e] = rr.x;
                    k2[e] = rr.y;
                    v1[e] = __half2float(__ushort_as_half(va16[e]));
                    v2[e] = __half2float(__ushort_as_half(vb16[e]));
                }
                float dk1, dk2, dv1, dv2;
                const uint2 ck1 = q8_quant8(k1, &dk1), ck2 = q8_quant8(k2, &dk2);
                const uint2 cv1 = q8_quant8(v1, &dv1), cv2 = q8_quant8(v2, &dv2);
                if (okn) {
                    const int64_t dst = (head * d.kv_total + d.cap + i) * kHeadDim + jc * 8;
                    *reinterpret_cast<uint2 *>(m.kq + dst) = ck1;
                    *reinterpret_cast<uint2 *>(m.kq + dst + half) = ck2;
                    *reinterpret_cast<uint2 *>(m.vq + dst) = cv1;
                    *reinterpret_cast<uint2 *>(m.vq + dst + half) = cv2;
                    if ((jc & 3) == 0) {
                        const int64_t sb = (head * d.kv_total + d.cap + i) * (kHeadDim / 32);
                        const int b1 = jc >> 2, b2 = 2 + (jc >> 2);
                        m.ks[sb + b1] = __half_as_ushort(__float2half_rn(dk1));
                        m.ks[sb + b2] = __half_as_ushort(__float2half_rn(dk2));
                        m.vs[sb + b1] = __half_as_ushort(__float2half_rn(dv1));
                        m.vs[sb + b2] = __half_as_ushort(__float2half_rn(dv2));
                    }
                }
            }
            asm volatile("fence.proxy.async.global;" ::: "memory");
        } else if (owns_noise) {
            // noise block of this head: K turned at committed + i, V copied.  Item u =
            // (noise row, 8 consecutive pairs); loads first, then stores.
            const int64_t head = ((int64_t)s * d.n_layer + layer) * d.n_head_kv + gk;
            const int n_items = d.q_len * (half / 8);
            for (int u = tid; u < n_items; u += SH::kConsumers) {
                const int i = u / (half / 8), jc = u - i * (half / 8);
                const uint16_t *ks = k_noise + ((int64_t)s * d.q_len + i) * d.kv_row + gk * kHeadDim + jc * 8;
                const uint16_t *vs = v_noise + ((int64_t)s * d.q_len + i) * d.kv_row + gk * kHeadDim + jc * 8;
                const uint4 a = *reinterpret_cast<const uint4 *>(ks);
                const uint4 bq = *reinterpret_cast<const uint4 *>(ks + half);
                const uint4 va = *reinterpret_cast<const uint4 *>(vs);
                const uint4 vb = *reinterpret_cast<const uint4 *>(vs + half);
                float2 cs8[8];
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    const float4 t = *reinterpret_cast<const float4 *>(csq + i * half + jc * 8 + e);
                    cs8[e] = make_float2(t.x, t.y);
                    cs8[e + 1] = make_float2(t.z, t.w);
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
            asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        bar_arrive(2, SH::kThreads);
        bar_sync(1, SH::kConsumers);

        const int mb = warp & 1, ksl = warp >> 1;
        const int g = lane >> 2, c = lane & 3;
        const int r0 = mb * 16 + g, r1 = r0 + 8;
        uint32_t qf[8][4];
        if constexpr (Q8) {
            // q8_0 K operands come four consecutive dimensions to a thread (4c .. 4c+3 of
            // each 16), which fill the MMA's k slots 2c, 2c+1, 2c+8, 2c+9; the query takes
            // the same order (a dot product does not care which slot holds which dimension)
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const int col = ks * 16 + 4 * c;
                const uint2 a = *reinterpret_cast<const uint2 *>(sq + swz(r0, col & ~7, kRows) + (col & 7) * 2);
                const uint2 b = *reinterpret_cast<const uint2 *>(sq + swz(r1, col & ~7, kRows) + (col & 7) * 2);
                qf[ks][0] = a.x;
                qf[ks][1] = b.x;
                qf[ks][2] = a.y;
                qf[ks][3] = b.y;
            }
        } else {
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
        const int i0 = r0 < d.rows ? r0 % d.q_len : 0;
        const int i1 = r1 < d.rows ? r1 % d.q_len : 0;
        const int key0 = ksl * SH::kKeys;

        // Visible tiles of this split, 32 at a time: one flags load per chunk, then the
        // set bits of two warp ballots (any visible / partly visible) give the tiles.
        int cbase = CLUSTER ? t0 + 32 : t0;
        uint32_t vis = CLUSTER ? __ballot_sync(0xffffffffu, f_first != 0) : 0u;
        uint32_t part = CLUSTER ? __ballot_sync(0xffffffffu, f_first == 2) : 0u;
        auto next_tile = [&](int &t, int &flag) -> bool {
            while (vis == 0u) {
                if (cbase >= t1) return false;
                const int u = cbase + lane;
                const int f = u < t1 ? (int)flags[u] : 0;
                vis = __ballot_sync(0xffffffffu, f != 0);
                part = __ballot_sync(0xffffffffu, f == 2);
                cbase += 32;
            }
            const int bit = __ffs(vis) - 1;
            vis &= vis - 1u;
            t = cbase - 32 + bit;
            flag = ((part >> bit) & 1u) ? 2 : 1;
            return true;
        };
        // every lane waits (each needs the barrier's acquire of the copied bytes); the
        // vote keeps the warp together if the bounded wait ever gives up
        auto wait_full = [&](int i) -> bool {
            if (__all_sync(0xffffffffu, mbar_wait(bar0 + 8 * (i % kStages), (uint32_t)(i / kStages) & 1u)))
                return true;
            if (lane == 0) atomicOr(m.err, kErrWaitFull);
            s_abort = 1;
            return false;
        };
        // S = Q K^T over this warp's keys of stage stg (F16 K tile at sk, or q8_0 codes and
        // scales), masked by the stage's per-row visibility bits when flag == 2 and, in the
        // plain online softmax, scaled to the log2 domain (the lazy one applies the scale in
        // the exponent).  nvalid: slots of the tile below kv_total.
        auto qk = [&](uint32_t sk, int flag, int stg, int nvalid, float (&sc)[SH::kNT][4]) {
#pragma unroll
            for (int n = 0; n < SH::kNT; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
            if constexpr (Q8) {
                // n-tile m holds keys key0 + 8m .. +7; this thread's key in it is key0 + 8m + g
                const uint2 *ksc = reinterpret_cast<const uint2 *>(smem + stg * kStageB + 2 * kTile * 128);
                uint2 kw[SH::kNT];
#pragma unroll
                for (int mt = 0; mt < SH::kNT; ++mt) {
                    const int key = key0 + 8 * mt + g;
                    kw[mt] = key < nvalid ? ksc[key] : make_uint2(0u, 0u);
                }
                // scale of block b of n-tile mt's key, in both halves
                auto kscale = [&](int mt, int b) {
                    return prmt((b >> 1) ? kw[mt].y : kw[mt].x, 0u, (b & 1) ? 0x3232u : 0x1010u);
                };
                if constexpr (SH::kNT == 4) {
                    // one ldmatrix.x4 per 16 dimensions: lane L addresses key key0 + L
                    const uint32_t rowa = sk + (uint32_t)(key0 + lane) * 128u;
                    const int xr = (key0 + lane) & 7;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        uint32_t w[4];
                        ldsm_x4(rowa + ((ks ^ xr) << 4), w[0], w[1], w[2], w[3]);
#pragma unroll
                        for (int mt = 0; mt < 4; ++mt) {
                            const uint32_t s2 = kscale(mt, ks >> 1);
                            const uint32_t wx = w[mt] ^ 0x80808080u;
                            mma16816(sc[mt], qf[ks], q8_pair(wx, 0x5140u, s2), q8_pair(wx, 0x7362u, s2));
                        }
                    }
                } else {
                    // 16 keys: one ldmatrix.x4 covers both n-tiles and two k steps (the 32
                    // dimensions of scale block kp)
                    const int lkey = key0 + 8 * ((lane >> 3) & 1) + (lane & 7);
                    const uint32_t rowa = sk + (uint32_t)lkey * 128u;
                    const int xr = lkey & 7;
#pragma unroll
                    for (int kp = 0; kp < 4; ++kp) {
                        uint32_t w[4];
                        ldsm_x4(rowa + (((2 * kp + (lane >> 4)) ^ xr) << 4), w[0], w[1], w[2], w[3]);
#pragma unroll
                        for (int mt = 0; mt < 2; ++mt) {
                            const uint32_t s2 = kscale(mt, kp);
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const uint32_t wx = w[2 * h + mt] ^ 0x80808080u;
                                mma16816(sc[mt], qf[2 * kp + h], q8_pair(wx, 0x5140u, s2),
                                         q8_pair(wx, 0x7362u, s2));
                            }
                        }
                    }
                }
            } else {
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
                    for (int np = 0; np < SH::kNT / 2; ++np) {
                        const int key = key0 + np * 16 + (lane & 7) + ((lane >> 4) << 3);
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(sk + swz(key, ks * 16 + (((lane >> 3) & 1) << 3), kTile), b0, b1, b2, b3);
                        mma16816(sc[np * 2], qf[ks], b0, b1);
                        mma16816(sc[np * 2 + 1], qf[ks], b2, b3);
                    }
                }
            }
            if constexpr (!SH::kLazy) {
#pragma unroll
                for (int n = 0; n < SH::kNT; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sc[n][e] *= scale_log2;
            }
            if (flag == 2) {
                const uint64_t w0 = sbits[stg * kMaxQWords + i0];
                const uint64_t w1 = sbits[stg * kMaxQWords + i1];
#pragma unroll
                for (int n = 0; n < SH::kNT; ++n)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int bit = key0 + n * 8 + 2 * c + e;
                        if (!((w0 >> bit) & 1ull)) sc[n][e] = -INFINITY;
                        if (!((w1 >> bit) & 1ull)) sc[n][2 + e] = -INFINITY;
                    }
            }
        };
        // online softmax (log2 domain) of rows r0 (j = 0) and r1 (j = 1), then O += P V
        // over the same keys of stage stg (F16 V tile at sv, or q8_0 codes and scales);
        // then the stage barrier `release` hands the stage back to the producer.
        // The reference maximum mrow may move lazily: P = 2^(scale S - mrow) may reach
        // 2^kLazyLog2 (exact in F16), and O and l are rescaled only when some row of the
        // warp outgrows its reference by more than that -- rarely after a row's first
        // visible tile.  O / l does not depend on the reference.
        auto softmax_pv = [&](uint32_t sv, uint32_t release, int stg, int nvalid,
                              float (&sc)[SH::kNT][4]) {
          if constexpr (!SH::kLazy) {
            float alpha[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float mx = -INFINITY;
#pragma unroll
                for (int n = 0; n < SH::kNT; ++n) mx = fmaxf(mx, fmaxf(sc[n][2 * j], sc[n][2 * j + 1]));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const float mnew = fmaxf(mrow[j], mx);
                const float muse = mnew == -INFINITY ? 0.f : mnew;
                alpha[j] = exp2f(mrow[j] - muse);
                mrow[j] = mnew;
                float rs = 0.f;
#pragma unroll
                for (int n = 0; n < SH::kNT; ++n) {
                    const float p0 = exp2f(sc[n][2 * j] - muse);
                    const float p1 = exp2f(sc[n][2 * j + 1] - muse);
                    sc[n][2 * j] = p0;
                    sc[n][2 * j + 1] = p1;
                    rs += p0 + p1;
                }
                lrow[j] = lrow[j] * alpha[j] + rs;
            }
            // rescale the numerators only when some row's maximum moved
            if (!__all_sync(0xffffffffu, alpha[0] == 1.f && alpha[1] == 1.f)) {
#pragma unroll
                for (int n = 0; n < 16; ++n) {
                    oacc[n][0] *= alpha[0];
                    oacc[n][1] *= alpha[0];
                    oacc[n][2] *= alpha[1];
                    oacc[n][3] *= alpha[1];
                }
            }
          } else {
            float mx[2];
            bool move = false;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float x = -INFINITY;
#pragma unroll
                for (int n = 0; n < SH::kNT; ++n) x = fmaxf(x, fmaxf(sc[n][2 * j], sc[n][2 * j + 1]));
                x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 1));
                x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 2));
                mx[j] = x * scale_log2;
                move |= mx[j] > mrow[j] + SH::kLazyLog2;
            }
            if (__any_sync(0xffffffffu, move)) {
                float alpha[2];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const float mnew = fmaxf(mrow[j], mx[j]);
                    alpha[j] = mnew == -INFINITY ? 1.f : exp2f(mrow[j] - mnew);
                    mrow[j] = mnew;
                    lrow[j] *= alpha[j];
                }
#pragma unroll
                for (int n = 0; n < 16; ++n) {
                    oacc[n][0] *= alpha[0];
                    oacc[n][1] *= alpha[0];
                    oacc[n][2] *= alpha[1];
                    oacc[n][3] *= alpha[1];
                }
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float muse = mrow[j] == -INFINITY ? 0.f : mrow[j];
                float rs = 0.f;
#pragma unroll
                for (int n = 0; n < SH::kNT; ++n) {
                    const float p0 = ex2_fast(fmaf(sc[n][2 * j], scale_log2, -muse));
                    const float p1 = ex2_fast(fmaf(sc[n][2 * j + 1], scale_log2, -muse));
                    sc[n][2 * j] = p0;
                    sc[n][2 * j + 1] = p1;
                    rs += p0 + p1;
                }
                lrow[j] += rs;
            }
          }
#pragma unroll
            for (int kk = 0; kk < SH::kKK; ++kk) {
                uint32_t pa[4];
                pa[0] = pack_half2(sc[2 * kk][0], sc[2 * kk][1]);
                pa[1] = pack_half2(sc[2 * kk][2], sc[2 * kk][3]);
                pa[2] = pack_half2(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
                pa[3] = pack_half2(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
                const int key = key0 + kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
                if constexpr (Q8) {
                    // keys kb + 2c, +1 (k slots 2c, 2c+1) and kb + 2c + 8, +9: their scales
                    const int kb = key0 + kk * 16;
                    const uint2 *vsc = reinterpret_cast<const uint2 *>(smem + stg * kStageB + 2 * kTile * 128 + kTile * 8);
                    const uint2 zero2 = make_uint2(0u, 0u);
                    const uint2 s0 = kb + 2 * c < nvalid ? vsc[kb + 2 * c] : zero2;
                    const uint2 s1 = kb + 2 * c + 1 < nvalid ? vsc[kb + 2 * c + 1] : zero2;
                    const uint2 s2 = kb + 2 * c + 8 < nvalid ? vsc[kb + 2 * c + 8] : zero2;
                    const uint2 s3 = kb + 2 * c + 9 < nvalid ? vsc[kb + 2 * c + 9] : zero2;
                    const uint32_t rowv = sv + (uint32_t)key * 128u;
#pragma unroll
                    for (int qp = 0; qp < 4; ++qp) {
                        // 16-byte chunks 2qp, 2qp+1 (dimensions 32qp .. 32qp+31, scale block
                        // qp) of keys kb..kb+15, transposed: a thread holds codes of keys
                        // (2c, 2c+1) at dimensions (2g, 2g+1) of each chunk
                        uint32_t r[4];
                        ldsm_x4_t(rowv + (((2 * qp + (lane >> 4)) ^ (key & 7)) << 4), r[0], r[1], r[2], r[3]);
                        const uint32_t hs = (qp & 1) ? 0x7632u : 0x5410u;
                        const uint32_t sA = prmt((qp >> 1) ? s0.y : s0.x, (qp >> 1) ? s1.y : s1.x, hs);
                        const uint32_t sB = prmt((qp >> 1) ? s2.y : s2.x, (qp >> 1) ? s3.y : s3.x, hs);
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            // chunk q = 2qp + h: n-tile 2q takes its even dimensions, 2q+1
                            // its odd ones (undone where O is written)
                            const uint32_t wa = r[2 * h] ^ 0x80808080u, wb = r[2 * h + 1] ^ 0x80808080u;
                            const int q = 2 * qp + h;
                            mma16816(oacc[2 * q], pa, q8_pair(wa, 0x6240u, sA), q8_pair(wb, 0x6240u, sB));
                            mma16816(oacc[2 * q + 1], pa, q8_pair(wa, 0x7351u, sA), q8_pair(wb, 0x7351u, sB));
                        }
                    }
                } else {
#pragma unroll
                    for (int dp = 0; dp < 8; ++dp) {
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_t(sv + swz(key, dp * 16 + ((lane >> 4) << 3), kTile), b0, b1, b2, b3);
                        mma16816(oacc[dp * 2], pa, b0, b1);
                        mma16816(oacc[dp * 2 + 1], pa, b2, b3);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(release);
        };
        int it = 0, t = 0, flag = 0;
        while (next_tile(t, flag)) {
            float sc[SH::kNT][4];
            if (!wait_full(it)) break;
            const int stg = it % kStages;
            const uint32_t sk = smem_u32(smem + stg * kStageB);
            const int nvalid = d.kv_total - t * kTile;      // >= 32: kv_total is a multiple of 32
            qk(sk, flag, stg, nvalid, sc);
            softmax_pv(sk + (Q8 ? kTile * 128 : kTileBytes), bar0 + 8 * (kStages + stg), stg, nvalid, sc);
            ++it;
        }

#pragma unroll
        for (int j = 0; j < 2; ++j) {
            lrow[j] += __shfl_xor_sync(0xffffffffu, lrow[j], 1);
            lrow[j] += __shfl_xor_sync(0xffffffffu, lrow[j], 2);
        }
        if constexpr (CLUSTER) {
            cluster_wait();     // every CTA of the cluster has started (see cluster_arrive_relaxed)
            // Merge the key slices of each row block inside this CTA, then push one partial
            // per row to the CTA of the cluster that finishes that row.  Every warp first
            // publishes its partial (in the idle stage buffers: per lane one float4 per
            // n-tile, then (max r0, max r1, sum r0, sum r1)); warp (mb, ksl) then merges
            // columns [32 ksl, 32 ksl + 32) of its row block and pushes them.
            bar_sync(1, SH::kConsumers);
            constexpr int kX4 = 17 * 32;                  // float4 per warp partial
            float4 *xs4 = reinterpret_cast<float4 *>(smem);
            {
                float4 *x = xs4 + (mb * SH::kSlices + ksl) * kX4;
#pragma unroll
                for (int n = 0; n < 16; ++n)
                    x[n * 32 + lane] = make_float4(oacc[n][0], oacc[n][1], oacc[n][2], oacc[n][3]);
                x[16 * 32 + lane] = make_float4(mrow[0], mrow[1], lrow[0], lrow[1]);
            }
            bar_sync(1, SH::kConsumers);
            const float4 *xb = xs4 + mb * SH::kSlices * kX4;
            float wk[2][SH::kSlices], mm[2], ll[2];
            {
                float4 ml[SH::kSlices];
#pragma unroll
                for (int k = 0; k < SH::kSlices; ++k) ml[k] = xb[k * kX4 + 16 * 32 + lane];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    float m = -INFINITY;
#pragma unroll
                    for (int k = 0; k < SH::kSlices; ++k) m = fmaxf(m, j ? ml[k].y : ml[k].x);
                    const float muse = m == -INFINITY ? 0.f : m;
                    float l = 0.f;
#pragma unroll
                    for (int k = 0; k < SH::kSlices; ++k) {
                        wk[j][k] = exp2f((j ? ml[k].y : ml[k].x) - muse);
                        l += wk[j][k] * (j ? ml[k].w : ml[k].z);
                    }
                    mm[j] = m;
                    ll[j] = l;
                }
            }
            const int rr[2] = {r0, r1};
            uint32_t a_row[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int r = rr[j];
                const int owner = r * (int)nct / kRows, lr = r - cluster_first_row(owner, (int)nct);
                a_row[j] = map_rank(smem_u32(recv_acc + ((int64_t)rank * rmax + lr) * kHeadDim), (uint32_t)owner);
                if (ksl == 0 && c == 0)
                    st_cluster_v2(map_rank(smem_u32(recv_ml + (int)rank * rmax + lr), (uint32_t)owner),
                                  mm[j], ll[j]);
            }
            if constexpr (Q8) {
                // n-tiles 2q / 2q+1 hold the even / odd dimensions of 16q .. 16q+15
#pragma unroll
                for (int qq = 0; qq < 8 / SH::kSlices; ++qq) {
                    const int q = ksl * (8 / SH::kSlices) + qq;
                    float v[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                    for (int k = 0; k < SH::kSlices; ++k) {
                        const float4 a = xb[k * kX4 + (2 * q) * 32 + lane];
                        const float4 b = xb[k * kX4 + (2 * q + 1) * 32 + lane];
                        v[0][0] += wk[0][k] * a.x; v[0][1] += wk[0][k] * b.x;
                        v[0][2] += wk[0][k] * a.y; v[0][3] += wk[0][k] * b.y;
                        v[1][0] += wk[1][k] * a.z; v[1][1] += wk[1][k] * b.z;
                        v[1][2] += wk[1][k] * a.w; v[1][3] += wk[1][k] * b.w;
                    }
#pragma unroll
                    for (int j = 0; j < 2; ++j)
                        st_cluster_v4(a_row[j] + 4u * (16 * q + 4 * c), v[j][0], v[j][1], v[j][2], v[j][3]);
                }
            } else {
#pragma unroll
                for (int nn = 0; nn < 16 / SH::kSlices; ++nn) {
                    const int n = ksl * (16 / SH::kSlices) + nn;
                    float v[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int k = 0; k < SH::kSlices; ++k) {
                        const float4 a = xb[k * kX4 + n * 32 + lane];
                        v[0] += wk[0][k] * a.x;
                        v[1] += wk[0][k] * a.y;
                        v[2] += wk[1][k] * a.z;
                        v[3] += wk[1][k] * a.w;
                    }
                    st_cluster_v2(a_row[0] + 4u * (n * 8 + 2 * c), v[0], v[1]);
                    st_cluster_v2(a_row[1] + 4u * (n * 8 + 2 * c), v[2], v[3]);
                }
            }
        } else {
            // merge the two key halves through stage buffer 0 (idle now), then write this
            // CTA's rows straight from registers
            bar_sync(1, SH::kConsumers);
            float *xo = reinterpret_cast<float *>(smem);          // [2 mb][64][32 lanes]
            float *xm = xo + 2 * 64 * 32;                          // [2 mb][2 j][32 lanes]
            float *xl = xm + 2 * 2 * 32;
            if (ksl == 1) {
#pragma unroll
                for (int n = 0; n < 16; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) xo[(mb * 64 + n * 4 + e) * 32 + lane] = oacc[n][e];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    xm[(mb * 2 + j) * 32 + lane] = mrow[j];
                    xl[(mb * 2 + j) * 32 + lane] = lrow[j];
                }
            }
            bar_sync(1, SH::kConsumers);
            if (ksl == 0) {
                const int rr[2] = {r0, r1};
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const float m1 = xm[(mb * 2 + j) * 32 + lane], l1 = xl[(mb * 2 + j) * 32 + lane];
                    const float mm = fmaxf(mrow[j], m1);
                    const float muse = mm == -INFINITY ? 0.f : mm;
                    const float a0 = exp2f(mrow[j] - muse), a1 = exp2f(m1 - muse);
                    const float ll = lrow[j] * a0 + l1 * a1;
                    const int r = rr[j];
                    if (d.groups == 1) {
                        // the only CTA of this (sequence, kv head): final output
                        if (r < d.rows) {
                            const int hh = r / d.q_len, i = r - hh * d.q_len;
                            const int h = gk * d.group + hh;
                            const float inv = ll > 0.f ? 1.f / ll : 0.f;
                            float *dst = o + (((int64_t)s * d.q_len + i) * d.n_head + h) * kHeadDim;
                            if constexpr (Q8) {
                                // n-tiles 2q / 2q+1: even / odd dimensions of 16q .. 16q+15
#pragma unroll
                                for (int q = 0; q < 8; ++q) {
                                    float v[4];
#pragma unroll
                                    for (int e = 0; e < 4; ++e) {
                                        const int n = 2 * q + (e & 1), x = 2 * j + (e >> 1);
                                        v[e] = (oacc[n][x] * a0 + xo[(mb * 64 + n * 4 + x) * 32 + lane] * a1) * inv;
                                    }
                                    *reinterpret_cast<float4 *>(dst + 16 * q + 4 * c) = make_float4(v[0], v[1], v[2], v[3]);
                                }
                            } else {
#pragma unroll
                                for (int n = 0; n < 16; ++n) {
                                    const float v0 = oacc[n][2 * j] * a0 + xo[(mb * 64 + n * 4 + 2 * j) * 32 + lane] * a1;
                                    const float v1 = oacc[n][2 * j + 1] * a0 + xo[(mb * 64 + n * 4 + 2 * j + 1) * 32 + lane] * a1;
                                    *reinterpret_cast<float2 *>(dst + n * 8 + 2 * c) = make_float2(v0 * inv, v1 * inv);
                                }
                            }
                        }
                    } else {
                        // one of several independent CTAs: partial for the combine kernel
                        const int64_t base = (((int64_t)s * d.n_head_kv + gk) * d.groups + sp) * kRows + r;
                        float *dst = m.part_acc + base * kHeadDim;
                        if constexpr (Q8) {
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                float v[4];
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const int n = 2 * q + (e & 1), x = 2 * j + (e >> 1);
                                    v[e] = oacc[n][x] * a0 + xo[(mb * 64 + n * 4 + x) * 32 + lane] * a1;
                                }
                                *reinterpret_cast<float4 *>(dst + 16 * q + 4 * c) = make_float4(v[0], v[1], v[2], v[3]);
                            }
                        } else {
#pragma unroll
                            for (int n = 0; n < 16; ++n) {
                                const float v0 = oacc[n][2 * j] * a0 + xo[(mb * 64 + n * 4 + 2 * j) * 32 + lane] * a1;
                                const float v1 = oacc[n][2 * j + 1] * a0 + xo[(mb * 64 + n * 4 + 2 * j + 1) * 32 + lane] * a1;
                                *reinterpret_cast<float2 *>(dst + n * 8 + 2 * c) = make_float2(v0, v1);
                            }
                        }
                        if (c == 0) m.part_ml[base] = make_float2(mm, ll);
                    }
                }
            }
        }
    }
    if constexpr (!CLUSTER) {
        if (m.clock) {
            __syncthreads();
            if (threadIdx.x == 0) clock_stop(m.clock, clk_slot);
        }
        return;
    }

    // ---------------- cluster merge: this CTA finishes its rows (cluster_first_row) ----
    cluster_sync();     // every partial of this CTA's rows is in its receive buffer
    const int n_part = (int)nct;
    const int row0 = cluster_first_row((int)rank, n_part);
    const int items = (min(kRows, cluster_first_row((int)rank + 1, n_part)) - row0) * (kHeadDim / 4);
    // one warp per row (items: 32 per row): lane p < n_part reads partial p's (max, sum)
    // and its weight; the warp's lanes then add the weighted numerators of their 4 columns
    for (int u = threadIdx.x; u < items; u += SH::kThreads) {
        const int lr = u / (kHeadDim / 4), c4 = (u % (kHeadDim / 4)) * 4;
        const float2 ml = lane < n_part ? recv_ml[lane * rmax + lr] : make_float2(-INFINITY, 0.f);
        float mm = ml.x;
#pragma unroll
        for (int o = 16; o; o >>= 1) mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, o));
        const float muse = mm == -INFINITY ? 0.f : mm;
        const float wp = lane < n_part ? exp2f(ml.x - muse) : 0.f;
        float l = wp * ml.y;
#pragma unroll
        for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int p = 0; p < n_part; ++p) {
            const float w = __shfl_sync(0xffffffffu, wp, p);
            const float4 v = *reinterpret_cast<const float4 *>(recv_acc + ((int64_t)p * rmax + lr) * kHeadDim + c4);
            acc.x += w * v.x;
            acc.y += w * v.y;
            acc.z += w * v.z;
            acc.w += w * v.w;
        }
        const int r = row0 + lr;
        if (d.groups == 1) {
            if (r < d.rows) {
                const int hh = r / d.q_len, i = r - hh * d.q_len;
                const int h = gk * d.group + hh;
                const float inv = l > 0.f ? 1.f / l : 0.f;
                *reinterpret_cast<float4 *>(o + (((int64_t)s * d.q_len + i) * d.n_head + h) * kHeadDim + c4) =
                    make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
            }
        } else {
            const int group = sp / (int)nct;
            const int64_t base = (((int64_t)s * d.n_head_kv + gk) * d.groups + group) * kRows + r;
            *reinterpret_cast<float4 *>(m.part_acc + base * kHeadDim + c4) = acc;
            if (c4 == 0) m.part_ml[base] = make_float2(mm, l);
        }
    }
    if (m.clock) {
        __syncthreads();
        if (threadIdx.x == 0) clock_stop(m.clock, clk_slot);
    }
}

// ---------------------------------------------------------------------------------
// Combine the per-group partials (log-sum-exp merge) of every (sequence, kv head).
// Grid (4, n_head_kv, n_seq) of 128 threads: block x covers rows 8x .. 8x+7, thread ->
// (row, 8 columns).  The group loop is unrolled so that its loads overlap.
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(128)
k_attend_combine(RingDims d, RingDev m, float *o) {
    const int gk = blockIdx.y, s = blockIdx.z;
    const int r = blockIdx.x * 8 + (threadIdx.x >> 4), c0 = (threadIdx.x & 15) * 8;
    if (r >= d.rows) return;
    const int64_t base = ((int64_t)s * d.n_head_kv + gk) * d.groups;
    float mm = -INFINITY;
#pragma unroll 4
    for (int g = 0; g < d.groups; ++g) mm = fmaxf(mm, m.part_ml[(base + g) * kRows + r].x);
    const float muse = mm == -INFINITY ? 0.f : mm;
    float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
    float l = 0.f;
#pragma unroll 4
    for (int g = 0; g < d.groups; ++g) {
        const float2 ml = m.part_ml[(base + g) * kRows + r];
        const float4 *src = reinterpret_cast<const float4 *>(m.part_acc + ((base + g) * kRows + r) * kHeadDim + c0);
        const float4 v0 = src[0], v1 = src[1];
        const float w = exp2f(ml.x - muse);
        l += w * ml.y;
        a0.x += w * v0.x; a0.y += w * v0.y; a0.z += w * v0.z; a0.w += w * v0.w;
        a1.x += w * v1.x; a1.y += w * v1.y; a1.z += w * v1.z; a1.w += w * v1.w;
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const int hh = r / d.q_len, i = r - hh * d.q_len;
    const int h = gk * d.group + hh;
    float4 *dst = reinterpret_cast<float4 *>(o + (((int64_t)s * d.q_len + i) * d.n_head + h) * kHeadDim + c0);
    dst[0] = make_float4(a0.x * inv, a0.y * inv, a0.z * inv, a0.w * inv);
    dst[1] = make_float4(a1.x * inv, a1.y * inv, a1.z * inv, a1.w * inv);
}

}  // namespace

size_t attend_smem_bytes() { return (size_t)Shape<true>::kSmem; }

cudaError_t attend_kernels_init() {
    cudaError_t e = cudaFuncSetAttribute(k_attend<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Shape<true>::kSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_attend<true, false>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_attend<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Shape<false>::kSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_attend<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Shape<false, true>::kSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_attend<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Shape<true, true>::kSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_attend<true, true>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
}

int attend_cluster_capacity(int cluster, bool q8) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cluster, 1, 1);
    cfg.blockDim = dim3(Shape<true>::kThreads);
    cfg.dynamicSmemBytes = q8 ? Shape<true, true>::kSmem : Shape<true>::kSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    const cudaError_t e = q8 ? cudaOccupancyMaxActiveClusters(&n, k_attend<true, true>, &cfg)
                             : cudaOccupancyMaxActiveClusters(&n, k_attend<true, false>, &cfg);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

cudaError_t launch_attend(const RingDims &d, const RingDev &m, const CUtensorMap *tm_k,
                          const CUtensorMap *tm_v, int layer, int kind, float scale_log2,
                          const float *q, const uint16_t *k_noise, const uint16_t *v_noise,
                          float *o, bool pdl, int early, cudaStream_t st) {
    if (!pdl) early = 0;
    const bool clustered = d.cluster > 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(d.n_splits, d.n_head_kv, d.n_seq);
    cfg.blockDim = dim3(clustered ? Shape<true>::kThreads : Shape<false>::kThreads);
    cfg.dynamicSmemBytes = clustered ? (d.kv_q8 ? Shape<true, true>::kSmem : Shape<true>::kSmem)
                                     : (d.kv_q8 ? Shape<false, true>::kSmem : Shape<false>::kSmem);
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (clustered) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = d.cluster;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    if (clustered && d.kv_q8)
        return cudaLaunchKernelEx(&cfg, k_attend<true, true>, *tm_k, *tm_v, d, m, layer, kind,
                                  scale_log2, q, k_noise, v_noise, o, early);
    if (clustered)
        return cudaLaunchKernelEx(&cfg, k_attend<true, false>, *tm_k, *tm_v, d, m, layer, kind,
                                  scale_log2, q, k_noise, v_noise, o, early);
    if (d.kv_q8)
        return cudaLaunchKernelEx(&cfg, k_attend<false, true>, *tm_k, *tm_v, d, m, layer, kind,
                                  scale_log2, q, k_noise, v_noise, o, 0);
    return cudaLaunchKernelEx(&cfg, k_attend<false, false>, *tm_k, *tm_v, d, m, layer, kind, scale_log2,
                              q, k_noise, v_noise, o, 0);
}

cudaError_t launch_attend_combine(const RingDims &d, const RingDev &m, float *o,
                                  cudaStream_t st) {
    k_attend_combine<<<dim3(kRows / 8, d.n_head_kv, d.n_seq), 128, 0, st>>>(d, m, o);
    return cudaGetLastError();
}

}  // namespace dflash
