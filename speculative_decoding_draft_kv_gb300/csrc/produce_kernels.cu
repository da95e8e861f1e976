// Context-row producer: fused target features -> ring K/V rows, one kernel.
//
// Page "DFLASH2_RING_PORT.md", test 11 (point 4 of the refuted hypotheses): the draft's
// context K/V rows are a shallow injection of the fused target features -- W_k and W_v
// times the feature vector, then k_norm, then RoPE -- and section 1.2 puts the row of
// position p into slot p % cap.  Here the projection, the per-head RMS norm, RoPE at p,
// the F16 rounding and the scatter into the ring are one kernel, so the pre-RoPE rows
// never make a round trip through HBM.
//
// Shape: a CTA owns 32 feature rows (the step's new positions, packed across sequences)
// and one 128-wide head of K or of V of one layer.  C = X W^T runs on the F16 tensor cores
// (m16n8k16, F32 accumulation).  The weights are repacked once (ring_set_producer) into
// contiguous 16 KiB tiles of 128 output rows x 64 hidden columns, so every W tile is one
// contiguous TMA box -- a row-major W read as 128-row x 128-byte boxes scatters each box
// over 128 DRAM rows and streamed at well under half of the HBM bandwidth.  W tiles
// arrive by TMA; the tile's feature rows
// (32 x 64) by one TMA box when they are consecutive rows of the caller's buffer (one
// sequence), else by one 128-byte bulk copy per row; both into a 4-stage shared-memory
// ring guarded by mbarriers.  With few rows the kernel streams weights, so the hidden dimension is split
// over a thread-block cluster of `ks` CTAs whose partial tiles are summed in the shared
// memory of the CTA that owns each row (distributed shared memory stores).  The owner then
// normalises, turns and stores its rows: one warp per row, lane l holding columns
// l, l+32, l+64, l+96, so both members of every rotary pair sit in one lane.
#include "ring_internal.h"
#include "ptx.h"

#include <cuda_fp16.h>

#include <type_traits>

namespace dflash {
namespace {

constexpr int kPM = 32;                    // feature rows per CTA
constexpr int kPN = 128;                   // output columns per CTA: one head of K or V
constexpr int kPK = 64;                    // hidden columns per stage
constexpr int kPStages = 4;
constexpr int kPBBytes = kPN * kPK * 2;    // W tile, 16 KiB (TMA box 64 x 128, 128B swizzle)
constexpr int kPAPitch = kPK * 2 + 16;     // feature row pitch: 16 bytes of padding keep
                                           // the row fragments of ldmatrix conflict-free
constexpr int kPABytes = kPM * kPAPitch;   // feature tile
constexpr int kPStage = (kPBBytes + kPABytes + 1023) / 1024 * 1024;   // W tiles 1024-aligned
constexpr int kPConsumers = 128;           // 4 warps, warp w -> columns [32 w, 32 w + 32)
constexpr int kPThreads = kPConsumers + 32;
constexpr int kPRecvRows = 40;             // >= ks * ceil(32 / ks) for ks = 1 .. 8
constexpr int kPOffRecv = kPStages * kPStage;                 // [ks][rows_per][128] f32
constexpr int kPOffBars = kPOffRecv + kPRecvRows * kPN * 4;
constexpr int kPOffMap = kPOffBars + 2 * kPStages * 8;
constexpr int kPSmem = 1024 + kPOffMap + kPM * 16;
static_assert(kPSmem <= 113 * 1024, "two producer CTAs per SM");

// byte offset of (row r, 16-byte chunk holding column dcol) in a 128-byte-swizzled tile of
// 64 columns
__device__ __forceinline__ uint32_t swz64(int r, int dcol) {
    return (uint32_t)(r * 128 + (((dcol >> 3) ^ (r & 7)) << 4));
}
// One head's row of a q8_0 slot from a warp: lane holds the values at lane + 32 q4, so
// 32-value block q4 is one value per lane.  Block maximum by a warp reduction, scale
// d = max|x| / 127, codes roundf(x * (1 / d)) (half away from zero), all in float32; the
// scale is stored as F16.  base: the slot's first value (codes and scales share it, the
// scales at base / 32).
__device__ __forceinline__ void q8_store_head(int8_t *codes, uint16_t *scales, int64_t base,
                                              const float (&x)[4], int lane) {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        float amax = fabsf(x[b]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float dq = amax / 127.f;
        const float id = dq > 0.f ? 1.f / dq : 0.f;
        int c = (int)roundf(x[b] * id);
        c = c > 127 ? 127 : (c < -127 ? -127 : c);
        codes[base + lane + 32 * b] = (int8_t)c;
        if (lane == 0) scales[base / 32 + b] = __half_as_ushort(__float2half_rn(dq));
    }
}

// Grid (units * ks): CTA x works on unit x / ks (the units of job 0, then those of job 1)
// as rank x % ks of a cluster of ks CTAs.  A unit is one 32-row tile of one output head of
// one layer: K head y (y < n_head_kv), V head y - n_head_kv (y < 2 n_head_kv), else query
// head y - 2 n_head_kv (noise rows only).
__global__ void __launch_bounds__(kPThreads, 2)
k_produce(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_feat0,
          const __grid_constant__ CUtensorMap tm_feat1, RingDims d, RingDev m,
          const uint16_t *__restrict__ feat0, const uint16_t *__restrict__ feat1, int hidden,
          const float *__restrict__ k_norm, float eps, const __grid_constant__ ProduceSeqs seqs,
          const __grid_constant__ ProduceLaunch L, NoiseOut nout) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *recv = reinterpret_cast<float *>(smem + kPOffRecv);
    const uint32_t bar0 = smem_u32(smem + kPOffBars);     // full[0..3], empty[0..3]
    int64_t *map_pos = reinterpret_cast<int64_t *>(smem + kPOffMap);
    int64_t *map_frow = map_pos + kPM;                    // -1: padding row
    __shared__ int map_seq[kPM];
    __shared__ int s_fail, s_valid, s_contig;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ks = L.ks;
    const uint32_t rank = ks > 1 ? cluster_rank() : 0u;
    const int64_t unit = (int64_t)blockIdx.x / ks;
    const int jb = L.n_jobs > 1 && unit >= L.job[0].units ? 1 : 0;
    const ProduceJob job = L.job[jb];
    const int64_t u = jb ? unit - L.job[0].units : unit;
    const int64_t m_total = job.m_total;
    const int64_t tiles = (m_total + kPM - 1) / kPM;
    const int64_t tile = u % tiles;
    int yk, layer;
    if (job.mode == 1) {
        yk = (int)(u / tiles);
        layer = job.layer;
    } else {
        const int64_t hl = u / tiles;
        yk = (int)(hl % (2 * d.n_head_kv));
        layer = (int)(hl / (2 * d.n_head_kv));
    }
    const CUtensorMap *tm_feat = jb ? &tm_feat1 : &tm_feat0;
    const uint16_t *__restrict__ feat = jb ? feat1 : feat0;
    const bool is_q = yk >= 2 * d.n_head_kv;
    const bool is_v = !is_q && yk >= d.n_head_kv;
    const int head = is_q ? yk - 2 * d.n_head_kv : (is_v ? yk - d.n_head_kv : yk);
    const int nkt = hidden / kPK;
    const int per = (nkt + ks - 1) / ks;
    const int kt0 = min(nkt, (int)rank * per), kt1 = min(nkt, kt0 + per);
    const int rows_per = (kPM + ks - 1) / ks;         // the last rank may own fewer

    // packed W tile (layer, K head y or V head y - n_head_kv, k-tile kt) is plane
    // wplane + kt of the packed weights
    const int wplane = (layer * L.out_heads + yk) * nkt;
    const int n_pre = min(kPStages, kt1 - kt0);
    if (threadIdx.x == kPConsumers) {
        prefetch_tensormap(&tm_w);
        prefetch_tensormap(tm_feat);
        for (int k = 0; k < kPStages; ++k) {
            mbar_init(bar0 + 8 * k, 1);          // the producer's expect_tx arrival
            mbar_init(bar0 + 8 * (kPStages + k), kPConsumers / 32);
        }
        s_fail = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        // the first weight tiles depend on nothing earlier in the stream: start them now
        // (expected bytes only: the stage's arrival comes with its feature rows)
        for (int k = 0; k < n_pre; ++k) {
            mbar_add_tx(bar0 + 8 * k, kPBBytes);
            tma_load_3d(smem_u32(smem + k * kPStage), &tm_w, 0, 0, wplane + kt0 + k, bar0 + 8 * k);
        }
    }
    // features, ring slots and step records are touched only after the previous kernel
    // is done
    pdl_wait();
    // kernel clock: the step counter is read before this grid releases its dependents (a
    // begin-step kernel that follows advances it)
    int clk_slot = 0;
    if (threadIdx.x == 0 && m.clock)
        clk_slot = job.mode == 1 ? clock_start(m.clock, kClockProject, job.layer)
                                 : clock_start(m.clock, kClockProduce, 0);
    if (warp == 0) {
        // row map: packed row index -> (sequence, position, feature row).  Sequence s owns
        // rows [prod_base, prod_base + n_new) of the packed list.
        const int64_t mr = tile * kPM + lane;
        int sq = -1;
        int64_t pos = 0, frow = -1;
        if (job.mode == 1) {                        // noise rows: (sequence, i) of layer
            if (mr < m_total) {
                sq = (int)(mr / d.q_len);
                pos = mr % d.q_len;
                frow = (int64_t)layer * m_total + mr;
            }
        } else if (mr < m_total && seqs.n > 0) {
            for (int s = 0; s < seqs.n; ++s)
                if (mr >= seqs.base[s] && mr < seqs.base[s] + seqs.n_new[s]) {
                    sq = s;
                    pos = seqs.start[s] + (mr - seqs.base[s]);
                    frow = seqs.src_row[s] + (mr - seqs.base[s]);
                }
        } else if (mr < m_total) {
            int lo = 0, hi = d.n_seq - 1;
            while (lo < hi) {                       // last s with prod_base <= mr
                const int mid = (lo + hi + 1) >> 1;
                if (m.steps[mid].prod_base <= mr) lo = mid;
                else hi = mid - 1;
            }
            const SeqStep st = m.steps[lo];
            const int64_t i = mr - st.prod_base;
            if (i < st.n_new) {
                sq = lo;
                pos = st.start + i;
                frow = st.src_row + i;
            }
        }
        map_seq[lane] = sq;
        map_pos[lane] = pos;
        map_frow[lane] = frow;
        const int nv = __popc(__ballot_sync(0xffffffffu, frow >= 0));
        const int64_t f0 = __shfl_sync(0xffffffffu, frow, 0);
        const bool seq_rows = __all_sync(0xffffffffu, frow < 0 || frow == f0 + lane);
        if (lane == 0) {
            s_valid = nv;
            s_contig = seq_rows ? 1 : 0;
        }
    }
    __syncthreads();
    // With every CTA of the grid resident, the next kernel's CTAs may settle onto idle SMs
    // now and do what does not depend on this grid while it finishes.
    if (L.single_wave) pdl_trigger();
    if (ks > 1) cluster_arrive_relaxed();

    if (warp == kPConsumers / 32) {
        // ---------------- producer warp ----------------
        int it = 0;
        for (int kt = kt0; kt < kt1; ++kt, ++it) {
            const int stg = it % kPStages;
            const uint32_t ph = (uint32_t)(it / kPStages) & 1u;
            if (!__all_sync(0xffffffffu, mbar_wait(bar0 + 8 * (kPStages + stg), ph ^ 1u))) {
                if (lane == 0) {
                    atomicOr(m.err, kErrWaitEmpty);
                    s_fail = 1;
                }
                break;
            }
            const uint32_t sb = smem_u32(smem + stg * kPStage);
            const uint32_t sa = sb + kPBBytes;
            const uint32_t full = bar0 + 8 * stg;
            const bool contig = s_contig != 0;
            if (lane == 0) {
                // one arrival for the stage, expecting the W tile (unless it went out at
                // start-up) and the feature rows: one box of 32 rows, or one 128-byte copy
                // per valid row
                const uint32_t a_bytes = contig ? (uint32_t)kPM * kPK * 2 : (uint32_t)s_valid * kPK * 2;
                mbar_expect_tx(full, (it >= n_pre ? kPBBytes : 0) + a_bytes);
                if (it >= n_pre) tma_load_3d(sb, &tm_w, 0, 0, wplane + kt, full);
                if (contig) tma_load_2d(sa, tm_feat, kt * kPK, (int)map_frow[0], full);
            }
            __syncwarp();
            const int64_t fr = map_frow[lane];      // row `lane` of the tile
            if (!contig && fr >= 0)
                bulk_g2s(sa + lane * kPAPitch, feat + fr * hidden + kt * kPK, kPK * 2, full);
        }
        // no copy may land after the CTA exits: wait (bounded) for the last stages' bytes
        if (lane == 0)
            for (int k = max(0, it - kPStages); k < it; ++k)
                if (!mbar_wait(bar0 + 8 * (k % kPStages), (uint32_t)(k / kPStages) & 1u)) {
                    atomicOr(m.err, kErrDrain);
                    break;
                }
        __syncwarp();
        if (ks > 1) cluster_wait();
    } else {
        // ---------------- consumer warps: C[32][32 w .. 32 w + 32) ----------------
        float acc[2][4][4];
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) acc[a][b][0] = acc[a][b][1] = acc[a][b][2] = acc[a][b][3] = 0.f;
        const bool two_blocks = m_total - tile * kPM > 16;
        const bool contig = s_contig != 0;        // feature tile swizzled (TMA) or padded
        int it = 0;
        for (int kt = kt0; kt < kt1; ++kt, ++it) {
            const int stg = it % kPStages;
            const uint32_t ph = (uint32_t)(it / kPStages) & 1u;
            if (!__all_sync(0xffffffffu, mbar_wait(bar0 + 8 * stg, ph))) {
                if (lane == 0) {
                    atomicOr(m.err, kErrWaitFull);
                    s_fail = 1;
                }
                break;
            }
            const uint32_t sb = smem_u32(smem + stg * kPStage);
            const uint32_t sa = sb + kPBBytes;
            // MT row blocks of 16: the second only when the tile has more than 16 rows
            auto mma_stage = [&](auto mtc) {
                constexpr int MT = decltype(mtc)::value;
#pragma unroll
                for (int ks16 = 0; ks16 < kPK / 16; ++ks16) {
                    uint32_t af[MT][4];
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt)
                        ldsm_x4(sa + (contig ? swz64(mt * 16 + (lane & 15), ks16 * 16 + ((lane >> 4) << 3))
                                             : (uint32_t)((mt * 16 + (lane & 15)) * kPAPitch +
                                                          (ks16 * 16 + ((lane >> 4) << 3)) * 2)),
                                af[mt][0], af[mt][1], af[mt][2], af[mt][3]);
#pragma unroll
                    for (int np = 0; np < 2; ++np) {
                        const int n = warp * 32 + np * 16 + (lane & 7) + ((lane >> 4) << 3);
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(sb + swz64(n, ks16 * 16 + (((lane >> 3) & 1) << 3)), b0, b1, b2, b3);
#pragma unroll
                        for (int mt = 0; mt < MT; ++mt) {
                            mma16816(acc[mt][np * 2], af[mt], b0, b1);
                            mma16816(acc[mt][np * 2 + 1], af[mt], b2, b3);
                        }
                    }
                }
            };
            if (two_blocks) mma_stage(std::integral_constant<int, 2>{});
            else mma_stage(std::integral_constant<int, 1>{});
            __syncwarp();
            if (lane == 0) mbar_arrive(bar0 + 8 * (kPStages + stg));
        }
        // partial tile -> the receive buffer of the CTA owning each row:
        // recv[src rank][local row][128]; only the tile's rows that hold a new row (a
        // prefix: rows are packed) -- a decode step fills a few of the 32
        if (ks > 1) cluster_wait();
        const int g = lane >> 2, c = lane & 3;
        const int64_t n_rows_tile = m_total - tile * kPM;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int h8 = 0; h8 < 2; ++h8) {
                const int r = mt * 16 + g + 8 * h8;
                if (r >= n_rows_tile) continue;
                const int owner = r / rows_per, lr = r - owner * rows_per;
                float *row = recv + ((int64_t)rank * rows_per + lr) * kPN;
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    const int col = warp * 32 + nt * 8 + 2 * c;
                    const float v0 = acc[mt][nt][2 * h8], v1 = acc[mt][nt][2 * h8 + 1];
                    if (ks > 1) {
                        st_cluster_v2(map_rank(smem_u32(row + col), (uint32_t)owner), v0, v1);
                    } else {
                        row[col] = v0;
                        row[col + 1] = v1;
                    }
                }
            }
    }
    if (ks > 1) cluster_sync();
    else __syncthreads();
    if (warp >= kPConsumers / 32 || s_fail) return;

    // ---------------- epilogue: rows [rank * rows_per, +rows_per) of the tile ----------
    for (int lr = warp; lr < rows_per; lr += kPConsumers / 32) {
        const int r = (int)rank * rows_per + lr;
        if (r >= kPM) break;
        const int s = map_seq[r];
        if (s < 0) continue;
        const int64_t p = map_pos[r];
        float v[4];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
            float a = 0.f;
            for (int src = 0; src < ks; ++src) a += recv[((int64_t)src * rows_per + lr) * kPN + lane + 32 * q4];
            v[q4] = a;
        }
        if (job.mode == 1) {
            // noise row i = p of sequence s: V as is, K and Q through their RMS norms
            const int64_t row = ((int64_t)layer * d.n_seq + s) * d.q_len + p;
            if (is_v) {
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                    nout.v[row * d.kv_row + head * kHeadDim + lane + 32 * q4] = __half_as_ushort(__float2half_rn(v[q4]));
                continue;
            }
            float ss = v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            const float inv = rsqrtf(ss / (float)kPN + eps);
            const float *w = (is_q ? nout.q_norm : k_norm) + (int64_t)layer * kPN;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const float y = v[q4] * inv * w[lane + 32 * q4];
                if (is_q) nout.q[(row * d.n_head + head) * kHeadDim + lane + 32 * q4] = y;
                else nout.k[row * d.kv_row + head * kHeadDim + lane + 32 * q4] = __half_as_ushort(__float2half_rn(y));
            }
            continue;
        }
        const int slot = (int)(p % d.cap);
        const int64_t base = ((((int64_t)s * d.n_layer + layer) * d.n_head_kv + head) * d.kv_total + slot) * kHeadDim;
        if (is_v) {
            if (d.kv_q8) {
                // q8_0 slots: V rounded to F16 first (it is an F16 row), then quantised
                float x[4];
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) x[q4] = __half2float(__float2half_rn(v[q4]));
                q8_store_head(m.vq, m.vs, base, x, lane);
                continue;
            }
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) m.v[base + lane + 32 * q4] = __half_as_ushort(__float2half_rn(v[q4]));
            continue;
        }
        // k_norm: RMS over the head, then the per-layer weight
        float ss = v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float inv = rsqrtf(ss / (float)kPN + eps);
        const float *w = k_norm + (int64_t)layer * kPN;
        float y[4];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) y[q4] = v[q4] * inv * w[lane + 32 * q4];
        // RoPE at p: pairs (i, i + 64) for i = lane and lane + 32
        float kr[4];                      // rotated values at lane + 32 q4
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2) {
            const int i = lane + 32 * q2;
            const float2 cs = rope_angle_cs(p, m.inv_freq[i]);
            const float x1 = y[q2], x2 = y[q2 + 2];
            kr[q2] = fmaf(x1, cs.x, -x2 * cs.y);
            kr[q2 + 2] = fmaf(x1, cs.y, x2 * cs.x);
        }
        if (d.kv_q8) {
            q8_store_head(m.kq, m.ks, base, kr, lane);   // quantised straight from the rotation
        } else {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) m.k[base + lane + 32 * q4] = __half_as_ushort(__float2half_rn(kr[q4]));
        }
        // section 1.2: slot_pos[slot] = p (the begin-step kernel that follows reads it)
        if (layer == 0 && head == 0 && lane == 0) m.slot_pos[(int64_t)s * d.cap + slot] = (int32_t)p;
    }
    if (m.clock) {
        bar_sync(1, kPConsumers);         // every consumer warp is past its stores
        if (threadIdx.x == 0) clock_stop(m.clock, clk_slot);
    }
}

}  // namespace

// Repack W_k, W_v [n_layer][kv_row][hidden] (and W_q [n_layer][n_q_heads * 128][hidden])
// into tiles: tile ((layer * out_heads + y) * nkt + kt), y = K head, n_head_kv + V head or
// 2 n_head_kv + Q head, holds rows head*128 .. +128 of that weight, columns kt*64 .. +64,
// row-major (128 x 64 F16 = 16 KiB).  16 bytes per item.
__global__ void k_pack_weights(const uint16_t *__restrict__ wk, const uint16_t *__restrict__ wv,
                               const uint16_t *__restrict__ wq, uint16_t *__restrict__ out,
                               int n_layer, int n_head_kv, int n_q_heads, int hidden) {
    const int nkt = hidden / kPK;
    const int out_heads = 2 * n_head_kv + n_q_heads;
    const int64_t total = (int64_t)n_layer * out_heads * nkt * kPN * (kPK / 8);
    for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < total;
         u += (int64_t)gridDim.x * blockDim.x) {
        const int c8 = (int)(u % (kPK / 8));
        int64_t t = u / (kPK / 8);
        const int row = (int)(t % kPN);
        t /= kPN;
        const int kt = (int)(t % nkt);
        t /= nkt;
        const int yk = (int)(t % out_heads);
        const int layer = (int)(t / out_heads);
        const bool is_q = yk >= 2 * n_head_kv;
        const bool is_v = !is_q && yk >= n_head_kv;
        const int head = is_q ? yk - 2 * n_head_kv : (is_v ? yk - n_head_kv : yk);
        const int src_heads = is_q ? n_q_heads : n_head_kv;
        const uint16_t *src = (is_q ? wq : (is_v ? wv : wk)) +
                              ((int64_t)layer * src_heads * kPN + head * kPN + row) * hidden + kt * kPK + c8 * 8;
        *reinterpret_cast<uint4 *>(out + u * 8) = *reinterpret_cast<const uint4 *>(src);
    }
}

size_t produce_smem_bytes() { return (size_t)kPSmem; }

cudaError_t launch_pack_weights(const uint16_t *wk, const uint16_t *wv, const uint16_t *wq,
                                uint16_t *out, int n_layer, int n_head_kv, int n_q_heads,
                                int hidden, cudaStream_t st) {
    k_pack_weights<<<1024, 256, 0, st>>>(wk, wv, wq, out, n_layer, n_head_kv, n_q_heads, hidden);
    return cudaGetLastError();
}

cudaError_t produce_kernels_init() {
    return cudaFuncSetAttribute(k_produce, cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmem);
}

int produce_capacity(int ks, int sms) {
    if (ks <= 1) {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_produce, kPThreads, kPSmem) !=
            cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        return per_sm * sms;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ks, 1, 1);
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = kPSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, k_produce, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n * ks;
}

int64_t produce_units(const RingDims &d, int mode, int64_t m_total, int out_heads) {
    const int64_t tiles = (m_total + kPM - 1) / kPM;
    return mode == 1 ? tiles * out_heads : tiles * 2 * d.n_head_kv * d.n_layer;
}

int produce_split(int64_t units, int hidden, const int *cap) {
    const int nkt = hidden / kPK;
    int best = 1;
    for (int ks = 2; ks <= kProduceMaxSplit && 2 * ks <= nkt; ++ks)
        if (units * ks * 20 <= (int64_t)cap[ks] * 17) best = ks;
    return best;
}

cudaError_t launch_produce(const RingDims &d, const RingDev &m, const CUtensorMap *tm_w,
                           const CUtensorMap *tm_feat0, const CUtensorMap *tm_feat1,
                           const uint16_t *feat0, const uint16_t *feat1, int hidden,
                           const ProduceLaunch &L, const float *k_norm, float eps,
                           const ProduceSeqs &seqs, const NoiseOut &nout, bool pdl, int resident,
                           cudaStream_t st) {
    int64_t units = 0;
    for (int j = 0; j < L.n_jobs; ++j) units += L.job[j].units;
    const int64_t ctas = units * L.ks;
    if (ctas <= 0 || ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
    ProduceLaunch lc = L;
    lc.single_wave = ctas <= resident ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas, 1, 1);
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = kPSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (L.ks > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = L.ks;
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
    return cudaLaunchKernelEx(&cfg, k_produce, *tm_w, *tm_feat0, *(tm_feat1 ? tm_feat1 : tm_feat0), d,
                              m, feat0, feat1, hidden, k_norm, eps, seqs, lc, nout);
}

}  // namespace dflash
