// Context-row producer on the 5th-generation tensor cores, for steps with many new rows.
//
// Page "DFLASH2_RING_PORT.md", test 11 (point 4 of the refuted hypotheses) and section 1.6:
// the context K/V rows are W_k and W_v times the fused feature vector, then k_norm, then
// RoPE.  A decode step brings a handful of rows and streams the weights (k_produce); the
// legacy window recompute (section 1.6: the whole window produced again every step) and a
// bulk prefill bring thousands, and then the projection is a dense contraction -- 2 x
// rows x 2 kv_row x hidden flops per layer -- that belongs on tcgen05.
//
// Shape: persistent CTAs (one per SM), each taking a contiguous run of work items; an item
// is one (128-row tile, kv head, layer), items ordered tile by tile, so every CTA works on
// one or two row tiles and all CTAs move through the weights of the same layer and head
// at about the same time (L2 reuse).  Per item D[128 x 256] = X[128 x hidden] times
// [W_k head; W_v head]^T is accumulated in tensor memory (lanes = rows, 256 F32 columns:
// the K head, then the V head).  Warp 4 streams, by TMA into a 4-stage ring of 48 KiB
// stages, the tile's 64 feature columns (one 128 x 64 box, 128-byte swizzle) and the two
// packed 128 x 64 weight tiles (the layout ring_set_producer makes), item after item
// without a break; one thread of warp 5 issues four 128 x 256 x 16 MMAs per stage, commits
// each stage back to the copy warp and each finished item to the row warps; warps 0-3 own
// one row each (32 TMEM lanes per warp).  When a CTA reaches a new row tile, the row warps
// compute the RoPE cos/sin of their row's position once (64 pairs, float64 angle
// reduction) into TMEM columns 256-383, while the MMAs of the item run; per item they read
// the K head into registers, move the V head to columns 384-511 and release the
// accumulator (the next item's MMAs start), then finish in registers: RMS norm of the K head, k_norm weight, RoPE, F16 (or
// q8_0) stores into slot p % cap, V as F16 (or q8_0 of its F16 rounding), slot_pos.
// The feature rows of the step must be one contiguous run (row_off laid out back to back,
// as the legacy recompute and a prefill give them); otherwise k_produce serves the step.
#include "ring_internal.h"
#include "ptx.h"

#include <cuda_fp16.h>

#include <algorithm>

namespace dflash {
namespace {

constexpr int kTM = 128;                    // rows per tile = TMEM lanes
constexpr int kTN = 256;                    // the K head (0-127), then the V head (128-255)
constexpr int kTK = 64;                     // hidden columns per stage (128 bytes of F16)
constexpr int kTStages = 4;
constexpr int kTABytes = kTM * kTK * 2;     // 16 KiB feature tile
constexpr int kTBBytes = kTN * kTK * 2;     // 32 KiB: two packed weight tiles back to back
constexpr int kTStage = kTABytes + kTBBytes;
constexpr int kTOffBars = kTStages * kTStage;
constexpr int kTSmem = 1024 + kTOffBars + 128;
constexpr int kTThreads = 192;              // warps 0-3 rows, 4 copies, 5 MMA
constexpr int kTCols = 512;                 // TMEM columns allocated: accumulator 0-255,
constexpr int kTTab = 256;                  // RoPE cos/sin of the row's position 256-383,
constexpr int kTStash = 384;                // the V head, moved out of the accumulator 384-511
constexpr uint32_t kTIdesc = tc_idesc_f16(kTM, kTN);
static_assert(kTStage % 1024 == 0, "stages keep the 128-byte swizzle atoms aligned");
static_assert(kTSmem <= 227 * 1024, "one CTA per SM");

// One row's 128 values as q8_0 blocks: d = max|x| / 127, codes roundf(x * (1 / d)), d as F16.
__device__ __forceinline__ void q8_store_row(int8_t *codes, uint16_t *scales, int64_t base,
                                             const float *x) {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(x[32 * b + j]));
        const float dq = amax / 127.f;
        const float id = dq > 0.f ? 1.f / dq : 0.f;
        uint32_t w[8];
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
            uint32_t word = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                int c = (int)roundf(x[32 * b + 4 * j4 + e] * id);
                c = c > 127 ? 127 : (c < -127 ? -127 : c);
                word |= (uint32_t)(uint8_t)(int8_t)c << (8 * e);
            }
            w[j4] = word;
        }
        uint4 *dst = reinterpret_cast<uint4 *>(codes + base + 32 * b);
        __stcs(dst, make_uint4(w[0], w[1], w[2], w[3]));
        __stcs(dst + 1, make_uint4(w[4], w[5], w[6], w[7]));
        scales[base / 32 + b] = __half_as_ushort(__float2half_rn(dq));
    }
}

// 128 F32 values -> F16 row of 256 bytes.  Rows are written once and read by later
// kernels: streaming stores keep the weights and features in L2 rather than the output.
__device__ __forceinline__ void f16_store_row(uint16_t *dst, const float *x) {
    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int j = 0; j < 16; ++j)
        __stcs(d4 + j, make_uint4(pack_half2(x[8 * j], x[8 * j + 1]), pack_half2(x[8 * j + 2], x[8 * j + 3]),
                                  pack_half2(x[8 * j + 4], x[8 * j + 5]), pack_half2(x[8 * j + 6], x[8 * j + 7])));
}

// 128 TMEM columns of this warp's lanes starting at column col, as floats
__device__ __forceinline__ void tmem_row128(uint32_t taddr, float (&x)[128]) {
    uint32_t r[4][32];
#pragma unroll
    for (int q = 0; q < 4; ++q) tmem_ld32(taddr + 32 * q, r[q]);
    tmem_ld_wait();
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int j = 0; j < 32; ++j) x[32 * q + j] = __uint_as_float(r[q][j]);
}

// Work of CTA c: with at least as many row tiles as CTAs, tiles c, c + G, ... (G = grid
// size), each with all n_head_kv x n_layer units; otherwise (G = tiles x q) tile c % tiles
// with the q-th part c / tiles of its units.  Either way a CTA keeps a row tile across
// units (its RoPE table is computed once) and the CTAs move through the units together (the
// weights in flight at once stay few).  Rows of the step are packed over sequences by
// SeqStep::prod_base; packed row mr is feature row frow_base + mr.
struct TcWork {
    int64_t tile0, tile_step, tiles;
    int u0, u1;
    __device__ TcWork(int64_t n_tiles, int units) : tiles(n_tiles) {
        if (n_tiles >= (int64_t)gridDim.x) {
            tile0 = blockIdx.x;
            tile_step = gridDim.x;
            u0 = 0;
            u1 = units;
        } else {
            const int q = (int)(gridDim.x / n_tiles), j = (int)(blockIdx.x / n_tiles);
            tile0 = blockIdx.x % n_tiles;
            tile_step = n_tiles;                      // one tile
            u0 = j * units / q;
            u1 = (j + 1) * units / q;
        }
    }
};
__global__ void __launch_bounds__(kTThreads, 1)
k_produce_tc(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_feat,
             RingDims d, RingDev m, int hidden, int64_t m_total, int64_t frow_base, int out_heads,
             const float *__restrict__ k_norm, float eps,
             const __grid_constant__ ProduceSeqs seqs) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    // mbarriers: full[S], empty[S], then the accumulator's full and empty
    const uint32_t bar0 = smem_u32(smem + kTOffBars);
    const uint32_t acc_full = bar0 + 8 * 2 * kTStages, acc_empty = acc_full + 8;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kTOffBars + 8 * (2 * kTStages + 2));
    __shared__ int s_fail;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nkt = hidden / kTK;
    const int units = d.n_head_kv * d.n_layer;       // items per row tile
    const TcWork wk((m_total + kTM - 1) / kTM, units);

    if (threadIdx.x == 4 * 32) {
        prefetch_tensormap(&tm_w);
        prefetch_tensormap(&tm_feat);
        for (int k = 0; k < kTStages; ++k) {
            mbar_init(bar0 + 8 * k, 1);                  // the copy thread's expect_tx arrival
            mbar_init(bar0 + 8 * (kTStages + k), 1);     // the MMA thread's commit
        }
        mbar_init(acc_full, 1);                          // the MMA thread's commit per item
        mbar_init(acc_empty, 4);                         // one arrival per row warp
        s_fail = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), kTCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // features, step records and ring slots only after the previous kernel is done
    pdl_wait();
    int clk_slot = 0;
    if (threadIdx.x == 0 && m.clock) clk_slot = clock_start(m.clock, kClockProduce, 0);

    if (warp == 4) {
        // ---------------- copies: every item's k-tiles, back to back ----------------
        int it = 0;
        if (lane == 0) {
            bool alive = true;
            for (int64_t tile = wk.tile0; tile < wk.tiles && alive; tile += wk.tile_step)
            for (int unit = wk.u0; unit < wk.u1 && alive; ++unit) {
                const int layer = unit / d.n_head_kv, head = unit - layer * d.n_head_kv;
                const int kplane = (layer * out_heads + head) * nkt;
                const int vplane = (layer * out_heads + d.n_head_kv + head) * nkt;
                const int frow0 = (int)(frow_base + tile * kTM);
                for (int kt = 0; kt < nkt; ++kt, ++it) {
                    const int stg = it % kTStages;
                    const uint32_t ph = (uint32_t)(it / kTStages) & 1u;
                    if (!mbar_wait(bar0 + 8 * (kTStages + stg), ph ^ 1u)) {
                        atomicOr(m.err, kErrWaitEmpty);
                        s_fail = 1;
                        alive = false;
                        break;
                    }
                    const uint32_t sa = smem_u32(smem + stg * kTStage), sb = sa + kTABytes;
                    const uint32_t full = bar0 + 8 * stg;
                    mbar_expect_tx(full, kTStage);
                    tma_load_2d(sa, &tm_feat, kt * kTK, frow0, full);
                    tma_load_3d(sb, &tm_w, 0, 0, kplane + kt, full);
                    tma_load_3d(sb + kTBBytes / 2, &tm_w, 0, 0, vplane + kt, full);
                }
            }
            // no copy may land after the CTA exits: wait (bounded) for the last stages
            for (int k = max(0, it - kTStages); k < it; ++k)
                if (!mbar_wait(bar0 + 8 * (k % kTStages), (uint32_t)(k / kTStages) & 1u)) {
                    atomicOr(m.err, kErrDrain);
                    break;
                }
        }
        __syncwarp();
    } else if (warp == 5) {
        // ---------------- MMA issue (one thread) ----------------
        if (lane == 0) {
            int it = 0, j = 0;
            bool alive = true;
            for (int64_t tile = wk.tile0; tile < wk.tiles && alive; tile += wk.tile_step)
            for (int unit = wk.u0; unit < wk.u1 && alive; ++unit, ++j) {
                // the row warps have read the previous item's accumulator
                if (!mbar_wait(acc_empty, (uint32_t)(j & 1) ^ 1u)) {
                    atomicOr(m.err, kErrWaitEmpty);
                    s_fail = 1;
                    alive = false;
                    break;
                }
                tc_fence_after();
                for (int kt = 0; kt < nkt; ++kt, ++it) {
                    const int stg = it % kTStages;
                    if (!mbar_wait(bar0 + 8 * stg, (uint32_t)(it / kTStages) & 1u)) {
                        atomicOr(m.err, kErrWaitFull);
                        s_fail = 1;
                        alive = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + stg * kTStage), sb = sa + kTABytes;
#pragma unroll
                    for (int kk = 0; kk < kTK / 16; ++kk)
                        tc_mma_f16(tmem, tc_desc_sw128(sa + 32 * kk), tc_desc_sw128(sb + 32 * kk), kTIdesc,
                                   (kt | kk) != 0 ? 1u : 0u);
                    tc_commit(bar0 + 8 * (kTStages + stg));   // the stage is free once these finish
                }
                tc_commit(acc_full);                          // this item's accumulators are final
            }
        }
        __syncwarp();
    } else {
        // ---------------- rows: warp w, lane l -> tile row 32 w + l ----------------
        const int r = warp * 32 + lane;
        const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
        int64_t cur_tile = -1;
        int s = -1;
        int64_t p = 0;
        int j = 0;
        bool alive = true;
        for (int64_t tile = wk.tile0; tile < wk.tiles && alive; tile += wk.tile_step)
        for (int unit = wk.u0; unit < wk.u1; ++unit, ++j) {
            const int layer = unit / d.n_head_kv, head = unit - layer * d.n_head_kv;
            if (tile != cur_tile) {
                // this row's sequence and position, and the RoPE table of the position
                cur_tile = tile;
                const int64_t mr = tile * kTM + r;
                s = -1;
                p = 0;
                if (mr < m_total) {
                    if (seqs.n > 0) {
                        for (int q = 0; q < seqs.n; ++q)
                            if (mr >= seqs.base[q] && mr < seqs.base[q] + seqs.n_new[q]) {
                                s = q;
                                p = seqs.start[q] + (mr - seqs.base[q]);
                            }
                    } else {
                        int lo = 0, hi = d.n_seq - 1;
                        while (lo < hi) {               // last s with prod_base <= mr
                            const int mid = (lo + hi + 1) >> 1;
                            if (m.steps[mid].prod_base <= mr) lo = mid;
                            else hi = mid - 1;
                        }
                        const SeqStep st = m.steps[lo];
                        if (mr - st.prod_base < st.n_new) {
                            s = lo;
                            p = st.start + (mr - st.prod_base);
                        }
                    }
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t u[32];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float2 cs = rope_angle_cs(p, m.inv_freq[16 * c + e]);
                        u[2 * e] = __float_as_uint(cs.x);
                        u[2 * e + 1] = __float_as_uint(cs.y);
                    }
                    tmem_st32(trow + kTTab + 32 * c, u);
                }
                tmem_st_wait();
            }
            // warp-uniform, so the warp's TMEM loads stay converged
            const bool ok = __all_sync(0xffffffffu, mbar_wait(acc_full, (uint32_t)(j & 1)));
            if (!ok) {
                if (lane == 0) {
                    atomicOr(m.err, kErrWaitFull);
                    s_fail = 1;
                }
                alive = false;
                break;
            }
            tc_fence_after();
            const bool live = s >= 0 && !s_fail;
            const int slot = (int)(p % d.cap);
            const int64_t base =
                ((((int64_t)(s < 0 ? 0 : s) * d.n_layer + layer) * d.n_head_kv + head) * d.kv_total + slot) * kHeadDim;
            float x[128];
            // the K head into registers and the V head into spare columns: the accumulator
            // is free for the next item's MMAs before this item's rows are finished
            tmem_row128(trow, x);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t u[32];
                tmem_ld32(trow + 128 + 32 * c, u);
                tmem_ld_wait();
                tmem_st32(trow + kTStash + 32 * c, u);
                tmem_st_wait();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);
            // K head: RMS norm over the head, the per-layer weight, RoPE at p (pairs i, i + 64)
            if (live) {
                float ss = 0.f;
#pragma unroll
                for (int i = 0; i < 128; ++i) ss = fmaf(x[i], x[i], ss);
                const float inv = rsqrtf(ss / 128.f + eps);
                const float *wn = k_norm + (int64_t)layer * kHeadDim;
#pragma unroll
                for (int i = 0; i < 128; ++i) x[i] = x[i] * inv * wn[i];
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t u[32];
                tmem_ld32(trow + kTTab + 32 * c, u);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int i = 16 * c + e;
                    const float cn = __uint_as_float(u[2 * e]), sn = __uint_as_float(u[2 * e + 1]);
                    const float x1 = x[i], x2 = x[i + 64];
                    x[i] = fmaf(x1, cn, -x2 * sn);
                    x[i + 64] = fmaf(x1, sn, x2 * cn);
                }
            }
            if (live) {
                if (d.kv_q8) q8_store_row(m.kq, m.ks, base, x);
                else f16_store_row(m.k + base, x);
            }
            // V head
            tmem_row128(trow + kTStash, x);
            if (live) {
                if (d.kv_q8) {
#pragma unroll
                    for (int i = 0; i < 128; ++i) x[i] = __half2float(__float2half_rn(x[i]));
                    q8_store_row(m.vq, m.vs, base, x);
                } else {
                    f16_store_row(m.v + base, x);
                }
                // section 1.2: slot_pos[slot] = p
                if (layer == 0 && head == 0) m.slot_pos[(int64_t)s * d.cap + slot] = (int32_t)p;
            }
        }
        if (m.clock) {
            bar_sync(1, 128);
            if (threadIdx.x == 0) clock_stop(m.clock, clk_slot);
        }
    }
    // every TMEM access is complete (tcgen05.wait::ld / ::st) before the columns are freed
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTCols);
    }
}

}  // namespace

cudaError_t produce_tc_init() {
    return cudaFuncSetAttribute(k_produce_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, kTSmem);
}

cudaError_t launch_produce_tc(const RingDims &d, const RingDev &m, const CUtensorMap *tm_w,
                              const CUtensorMap *tm_feat, int hidden, int64_t m_total,
                              int64_t frow_base, int out_heads, const float *k_norm, float eps,
                              const ProduceSeqs &seqs, int sms, bool pdl, cudaStream_t st) {
    const int64_t tiles = (m_total + kTM - 1) / kTM;
    if (tiles <= 0 || hidden % kTK) return cudaErrorInvalidValue;
    // one CTA per SM: all of them on distinct tiles, or q CTAs per tile
    const int64_t g = std::max(sms, 1);
    const int64_t units = (int64_t)d.n_head_kv * d.n_layer;
    const int64_t grid = tiles >= g ? g : tiles * std::min<int64_t>(g / tiles, units);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kTThreads);
    cfg.dynamicSmemBytes = kTSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_produce_tc, *tm_w, *tm_feat, d, m, hidden, m_total, frow_base,
                              out_heads, k_norm, eps, seqs);
}

}  // namespace dflash
