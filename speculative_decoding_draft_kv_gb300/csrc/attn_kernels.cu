// Masked GQA attention of the noise block over the ring (split-KV flash-decode).
//
// Page "DFLASH2_RING_PORT.md", sections 1.1 and 1.4: the q_len noise queries attend to
// all kv_total slots of the layer's F16 K/V tensors under mask_full or mask_swa.  The
// hot kernel streams each kv head's visible 64-slot tiles with 3-D TMA boxes into a
// 3-stage shared-memory ring (128-byte swizzle), guarded by mbarriers; one producer warp
// issues the copies and four consumer warps compute S = Q K^T and O += P V on the F16
// tensor cores (m16n8k16, F32 accumulation) with an online softmax in F32 registers.
// All 32 query rows that share a kv head (4 heads x 8 queries) ride in one CTA, so each
// K/V byte is read from HBM once per step and layer.  Tiles whose mask flag says "no
// visible slot" are never fetched.
#include "ring_internal.h"

#include <cuda_fp16.h>

namespace dflash {
namespace {

constexpr int kStages = 3;              // 3 x 32 KiB + Q: two CTAs fit on one SM
constexpr int kTileBytes = kTile * kHeadDim * 2;   // one 64-slot tile of one head, K or V
constexpr int kHalfBox = kTileBytes / 2;           // TMA box: 64 slots x 64 columns
constexpr int kStageBytes = 2 * kTileBytes;        // K + V
constexpr int kQBytes = kRows * kHeadDim * 2;
constexpr int kComputeWarps = 4;
constexpr int kThreads = (kComputeWarps + 1) * 32;
constexpr int kBarBytes = 2 * kStages * 8;
constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kQBytes + kBarBytes;
constexpr uint64_t kWaitNs = 2000000000ull;        // bounded waits give up after 2 s

static_assert(kComputeWarps * 32 == 128, "named barrier below assumes 128 consumers");
static_assert(2 * 64 * 32 * 4 + 2 * 2 * 2 * 32 * 4 <= kStages * kStageBytes,
              "merge scratch must fit in the stage buffers");

// ---------------------------------------------------------------------------------
// PTX helpers
// ---------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase of `parity` to complete; false once kWaitNs have passed (or after a
// hard iteration cap), never an unbounded spin.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t it = 1; it < (1u << 30); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0 && global_ns() - t0 > kWaitNs) return false;
    }
    return false;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *tm, int x, int y,
                                            int z, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D += A(16x16, row) * B(16x8, col), F16 inputs, F32 accumulation.
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Byte offset of the 16-byte chunk holding (row r, columns dcol..dcol+7) in a
// [rows][128] F16 tile kept as two halves (columns 0-63 and 64-127) of `rows_half` rows
// of 128 bytes each, in the TMA 128-byte swizzle (chunk index xor row mod 8).  The
// tile base must be 1024-byte aligned.
__device__ __forceinline__ uint32_t swz(int r, int dcol, int rows_half) {
    return (uint32_t)((dcol >> 6) * rows_half * 128 + r * 128 +
                      ((((dcol & 63) >> 3) ^ (r & 7)) << 4));
}

// ---------------------------------------------------------------------------------
// Prologue: RoPE of the queries (to F16, GQA-grouped rows) and of the noise-block keys
// (stored to slots cap + j), noise values copied.  Grid (q_len, n_seq).
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
k_attend_prologue(RingDims d, RingDev m, int layer, const float *q, const uint16_t *k_noise,
                  const uint16_t *v_noise) {
    __shared__ double cs_cos[kHeadDim / 2], cs_sin[kHeadDim / 2];
    const int i = blockIdx.x, s = blockIdx.y;
    const int hd = kHeadDim, half = kHeadDim / 2;
    const int64_t pos = m.steps[s].committed + i;
    for (int j = threadIdx.x; j < half; j += blockDim.x) {
        double sn, c;
        sincos((double)pos * m.inv_freq[j], &sn, &c);
        cs_cos[j] = c;
        cs_sin[j] = sn;
    }
    __syncthreads();

    const float *qs = q + ((int64_t)s * d.q_len + i) * d.n_head * hd;
    for (int idx = threadIdx.x; idx < d.n_head * half; idx += blockDim.x) {
        const int h = idx / half, j = idx - h * half;
        const double x1 = qs[h * hd + j], x2 = qs[h * hd + j + half];
        const double c = cs_cos[j], sn = cs_sin[j];
        const double y1 = __dsub_rn(__dmul_rn(x1, c), __dmul_rn(x2, sn));
        const double y2 = __dadd_rn(__dmul_rn(x1, sn), __dmul_rn(x2, c));
        const int gk = h / d.group, r = (h - gk * d.group) * d.q_len + i;
        uint16_t *dst = m.q16 + (((int64_t)s * d.n_head_kv + gk) * kRows + r) * hd;
        dst[j] = __half_as_ushort(__double2half(y1));
        dst[j + half] = __half_as_ushort(__double2half(y2));
    }

    const uint16_t *ks = k_noise + ((int64_t)s * d.q_len + i) * d.kv_row;
    const int64_t head0 = ((int64_t)s * d.n_layer + layer) * d.n_head_kv;
    const int slot = d.cap + i;
    for (int idx = threadIdx.x; idx < d.n_head_kv * half; idx += blockDim.x) {
        const int g = idx / half, j = idx - g * half;
        const double x1 = (double)__half2float(__ushort_as_half(ks[g * hd + j]));
        const double x2 = (double)__half2float(__ushort_as_half(ks[g * hd + j + half]));
        const double c = cs_cos[j], sn = cs_sin[j];
        const double y1 = __dsub_rn(__dmul_rn(x1, c), __dmul_rn(x2, sn));
        const double y2 = __dadd_rn(__dmul_rn(x1, sn), __dmul_rn(x2, c));
        uint16_t *dst = m.k + ((head0 + g) * d.kv_total + slot) * hd;
        dst[j] = __half_as_ushort(__double2half(y1));
        dst[j + half] = __half_as_ushort(__double2half(y2));
    }
    const uint4 *vs = reinterpret_cast<const uint4 *>(v_noise + ((int64_t)s * d.q_len + i) * d.kv_row);
    for (int idx = threadIdx.x; idx < d.n_head_kv * (hd / 8); idx += blockDim.x) {
        const int g = idx / (hd / 8), c = idx - g * (hd / 8);
        reinterpret_cast<uint4 *>(m.v + ((head0 + g) * d.kv_total + slot) * hd)[c] = vs[idx];
    }
}

// ---------------------------------------------------------------------------------
// Split-KV attention.  Grid (n_splits, n_head_kv, n_seq); 5 warps: warps 0-3 compute,
// warp 4 produces.  Compute warp w owns query rows 16*(w & 1) .. +16 and the key half
// (w >> 1) of every 64-slot tile; the two key halves are merged at the end.
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 2)
k_attend_split(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
               RingDims d, RingDev m, int layer, int kind, float scale_log2, float *o) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sq = smem + kStages * kStageBytes;
    const uint32_t bar0 = smem_u32(sq + kQBytes);   // full[0..S-1], then empty[0..S-1]
    __shared__ volatile int s_abort;

    const int sp = blockIdx.x, gk = blockIdx.y, s = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = sp * d.tiles_per_split;
    const int t1 = min(d.n_tiles, t0 + d.tiles_per_split);
    const uint8_t *flags = m.flags + ((int64_t)s * d.n_kinds + kind) * d.n_tiles;
    const float *maskp = m.mask + ((int64_t)s * d.n_kinds + kind) * d.q_len * d.kv_total;

    if (threadIdx.x == 0) {
        for (int k = 0; k < kStages; ++k) {
            mbar_init(bar0 + 8 * k, 1);
            mbar_init(bar0 + 8 * (kStages + k), kComputeWarps);
        }
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();

    if (warp == kComputeWarps) {
        // ---------------- producer ----------------
        if (lane != 0) return;
        const int zrow = (s * d.n_layer + layer) * d.n_head_kv + gk;
        int it = 0;
        for (int t = t0; t < t1; ++t) {
            if (flags[t] == 0) continue;
            const int stg = it % kStages;
            const uint32_t ph = (uint32_t)(it / kStages) & 1u;
            if (!mbar_wait(bar0 + 8 * (kStages + stg), ph ^ 1u)) {
                atomicOr(m.err, kErrWaitEmpty);
                s_abort = 1;
                break;
            }
            if (s_abort) break;
            const uint32_t full = bar0 + 8 * stg;
            const uint32_t dk = smem_u32(smem + stg * kStageBytes);
            const uint32_t dv = dk + kTileBytes;
            mbar_expect_tx(full, kStageBytes);
            tma_load_3d(dk, &tm_k, 0, t * kTile, zrow, full);
            tma_load_3d(dk + kHalfBox, &tm_k, 64, t * kTile, zrow, full);
            tma_load_3d(dv, &tm_v, 0, t * kTile, zrow, full);
            tma_load_3d(dv + kHalfBox, &tm_v, 64, t * kTile, zrow, full);
            ++it;
        }
        // No copy may land after the CTA exits: wait for the last load of every stage.
        for (int k = max(0, it - kStages); k < it; ++k) {
            if (!mbar_wait(bar0 + 8 * (k % kStages), (uint32_t)(k / kStages) & 1u)) {
                atomicOr(m.err, kErrDrain);
                break;
            }
        }
        return;
    }

    // ---------------- consumers ----------------
    const int mb = warp & 1, kh = warp >> 1;
    const int g = lane >> 2, c = lane & 3;

    {   // stage this kv head's 32 F16 query rows into shared memory (swizzled like K)
        const uint4 *qsrc = reinterpret_cast<const uint4 *>(
            m.q16 + ((int64_t)s * d.n_head_kv + gk) * kRows * kHeadDim);
        for (int idx = threadIdx.x; idx < kRows * kHeadDim / 8; idx += kComputeWarps * 32) {
            const int r = idx >> 4, ch = idx & 15;
            *reinterpret_cast<uint4 *>(sq + swz(r, ch * 8, kRows)) = qsrc[idx];
        }
    }
    named_bar_sync(1, kComputeWarps * 32);

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

    const int r0 = mb * 16 + g, r1 = r0 + 8;
    const int i0 = r0 < d.rows ? r0 % d.q_len : 0;
    const int i1 = r1 < d.rows ? r1 % d.q_len : 0;
    const float *mrow0 = maskp + (int64_t)i0 * d.kv_total;
    const float *mrow1 = maskp + (int64_t)i1 * d.kv_total;

    int it = 0;
    for (int t = t0; t < t1; ++t) {
        const int flag = flags[t];
        if (flag == 0) continue;
        const int stg = it % kStages;
        const uint32_t ph = (uint32_t)(it / kStages) & 1u;
        if (!mbar_wait(bar0 + 8 * stg, ph)) {
            atomicOr(m.err, kErrWaitFull);
            s_abort = 1;
            break;
        }
        const uint32_t sk = smem_u32(smem + stg * kStageBytes);
        const uint32_t sv = sk + kTileBytes;

        // S = Q K^T over this warp's 32 keys (4 n-tiles of 8)
        float sc[4][4];
#pragma unroll
        for (int n = 0; n < 4; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
            for (int np = 0; np < 2; ++np) {
                const int key = kh * 32 + np * 16 + (lane & 7) + ((lane >> 4) << 3);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(sk + swz(key, ks * 16 + (((lane >> 3) & 1) << 3), kTile), b0, b1, b2, b3);
                mma16816(sc[np * 2], qf[ks], b0, b1);
                mma16816(sc[np * 2 + 1], qf[ks], b2, b3);
            }
        }
#pragma unroll
        for (int n = 0; n < 4; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) sc[n][e] *= scale_log2;
        if (flag == 2) {
#pragma unroll
            for (int n = 0; n < 4; ++n)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int slot = t * kTile + kh * 32 + n * 8 + 2 * c + e;
                    const bool ok = slot < d.kv_total;
                    sc[n][e] += ok ? __ldg(mrow0 + slot) : -INFINITY;
                    sc[n][2 + e] += ok ? __ldg(mrow1 + slot) : -INFINITY;
                }
        }

        // online softmax (log2 domain), rows r0 (j = 0) and r1 (j = 1)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float mx = fmaxf(fmaxf(sc[0][2 * j], sc[0][2 * j + 1]), fmaxf(sc[1][2 * j], sc[1][2 * j + 1]));
            mx = fmaxf(mx, fmaxf(fmaxf(sc[2][2 * j], sc[2][2 * j + 1]), fmaxf(sc[3][2 * j], sc[3][2 * j + 1])));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float mnew = fmaxf(mrow[j], mx);
            const float muse = mnew == -INFINITY ? 0.f : mnew;
            const float alpha = exp2f(mrow[j] - muse);
            mrow[j] = mnew;
            float rs = 0.f;
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                const float p0 = exp2f(sc[n][2 * j] - muse);
                const float p1 = exp2f(sc[n][2 * j + 1] - muse);
                sc[n][2 * j] = p0;
                sc[n][2 * j + 1] = p1;
                rs += p0 + p1;
            }
            lrow[j] = lrow[j] * alpha + rs;
#pragma unroll
            for (int n = 0; n < 16; ++n) {
                oacc[n][2 * j] *= alpha;
                oacc[n][2 * j + 1] *= alpha;
            }
        }

        // O += P V over the same 32 keys (2 k-steps of 16)
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            uint32_t pa[4];
            pa[0] = pack_half2(sc[2 * kk][0], sc[2 * kk][1]);
            pa[1] = pack_half2(sc[2 * kk][2], sc[2 * kk][3]);
            pa[2] = pack_half2(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
            pa[3] = pack_half2(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
            const int key = kh * 32 + kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
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
        ++it;
    }

#pragma unroll
    for (int j = 0; j < 2; ++j) {
        lrow[j] += __shfl_xor_sync(0xffffffffu, lrow[j], 1);
        lrow[j] += __shfl_xor_sync(0xffffffffu, lrow[j], 2);
    }

    // merge the two key halves through the (now idle) stage buffers
    named_bar_sync(1, kComputeWarps * 32);
    float *xo = reinterpret_cast<float *>(smem);          // [2 mb][64][32 lanes]
    float *xm = xo + 2 * 64 * 32;                          // [2 mb][2 j][32 lanes]
    float *xl = xm + 2 * 2 * 32;
    if (kh == 1) {
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
    named_bar_sync(1, kComputeWarps * 32);
    if (kh == 1) return;

#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const float m1 = xm[(mb * 2 + j) * 32 + lane], l1 = xl[(mb * 2 + j) * 32 + lane];
        const float mm = fmaxf(mrow[j], m1);
        const float muse = mm == -INFINITY ? 0.f : mm;
        const float a0 = exp2f(mrow[j] - muse), a1 = exp2f(m1 - muse);
        lrow[j] = lrow[j] * a0 + l1 * a1;
        mrow[j] = mm;
#pragma unroll
        for (int n = 0; n < 16; ++n)
#pragma unroll
            for (int e = 0; e < 2; ++e)
                oacc[n][2 * j + e] = oacc[n][2 * j + e] * a0 + xo[(mb * 64 + n * 4 + 2 * j + e) * 32 + lane] * a1;
    }

    const int rr[2] = {r0, r1};
    if (d.n_splits == 1) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int r = rr[j];
            if (r >= d.rows) continue;
            const int hh = r / d.q_len, i = r - hh * d.q_len;
            const int h = gk * d.group + hh;
            const float inv = lrow[j] > 0.f ? 1.f / lrow[j] : 0.f;
            float *dst = o + (((int64_t)s * d.q_len + i) * d.n_head + h) * kHeadDim;
#pragma unroll
            for (int n = 0; n < 16; ++n)
                *reinterpret_cast<float2 *>(dst + n * 8 + 2 * c) =
                    make_float2(oacc[n][2 * j] * inv, oacc[n][2 * j + 1] * inv);
        }
    } else {
        const int64_t base = (((int64_t)s * d.n_head_kv + gk) * d.n_splits + sp) * kRows;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int r = rr[j];
            float *dst = m.part_acc + (base + r) * kHeadDim;
#pragma unroll
            for (int n = 0; n < 16; ++n)
                *reinterpret_cast<float2 *>(dst + n * 8 + 2 * c) =
                    make_float2(oacc[n][2 * j], oacc[n][2 * j + 1]);
            if (c == 0) m.part_ml[base + r] = make_float2(mrow[j], lrow[j]);
        }
    }
}

// ---------------------------------------------------------------------------------
// Combine the per-split partials (log-sum-exp merge).  Grid (n_head_kv, n_seq), 256
// threads: thread -> (row r = tid / 8, 16 columns).
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
k_attend_combine(RingDims d, RingDev m, float *o) {
    const int gk = blockIdx.x, s = blockIdx.y;
    const int r = threadIdx.x >> 3, c0 = (threadIdx.x & 7) * 16;
    if (r >= d.rows) return;
    const int64_t base = ((int64_t)s * d.n_head_kv + gk) * d.n_splits;
    float mm = -INFINITY;
    for (int sp = 0; sp < d.n_splits; ++sp) mm = fmaxf(mm, m.part_ml[(base + sp) * kRows + r].x);
    const float muse = mm == -INFINITY ? 0.f : mm;
    float acc[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) acc[k] = 0.f;
    float l = 0.f;
    for (int sp = 0; sp < d.n_splits; ++sp) {
        const float2 ml = m.part_ml[(base + sp) * kRows + r];
        const float w = exp2f(ml.x - muse);
        l += w * ml.y;
        const float4 *src = reinterpret_cast<const float4 *>(m.part_acc + ((base + sp) * kRows + r) * kHeadDim + c0);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float4 v = src[k];
            acc[4 * k + 0] += w * v.x;
            acc[4 * k + 1] += w * v.y;
            acc[4 * k + 2] += w * v.z;
            acc[4 * k + 3] += w * v.w;
        }
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const int hh = r / d.q_len, i = r - hh * d.q_len;
    const int h = gk * d.group + hh;
    float4 *dst = reinterpret_cast<float4 *>(o + (((int64_t)s * d.q_len + i) * d.n_head + h) * kHeadDim + c0);
#pragma unroll
    for (int k = 0; k < 4; ++k)
        dst[k] = make_float4(acc[4 * k] * inv, acc[4 * k + 1] * inv, acc[4 * k + 2] * inv,
                             acc[4 * k + 3] * inv);
}

}  // namespace

size_t attend_split_smem_bytes() { return (size_t)kSmemBytes; }

cudaError_t launch_attend_prologue(const RingDims &d, const RingDev &m, int layer,
                                   const float *q, const uint16_t *k_noise,
                                   const uint16_t *v_noise, cudaStream_t st) {
    k_attend_prologue<<<dim3(d.q_len, d.n_seq), 256, 0, st>>>(d, m, layer, q, k_noise, v_noise);
    return cudaGetLastError();
}

cudaError_t attend_kernels_init() {
    return cudaFuncSetAttribute(k_attend_split, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmemBytes);
}

cudaError_t launch_attend_split(const RingDims &d, const RingDev &m, const CUtensorMap *tm_k,
                                const CUtensorMap *tm_v, int layer, int kind, float scale_log2,
                                float *o, cudaStream_t st) {
    k_attend_split<<<dim3(d.n_splits, d.n_head_kv, d.n_seq), kThreads, kSmemBytes, st>>>(
        *tm_k, *tm_v, d, m, layer, kind, scale_log2, o);
    return cudaGetLastError();
}

cudaError_t launch_attend_combine(const RingDims &d, const RingDev &m, float *o,
                                  cudaStream_t st) {
    k_attend_combine<<<dim3(d.n_head_kv, d.n_seq), 256, 0, st>>>(d, m, o);
    return cudaGetLastError();
}

}  // namespace dflash
