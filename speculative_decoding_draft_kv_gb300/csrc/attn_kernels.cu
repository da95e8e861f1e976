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
static_assert(2 * 64 * 32 * 4 + 2 * 2 * 2 * 32 * 4 <= kStageBytes,
              "key-half merge scratch must fit in stage buffer 0");
static_assert(kStages >= 2 && kRows * 132 * 4 + kRows * 8 <= kStageBytes,
              "cluster-merge partial must fit in stage buffer 1");

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

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ float ld_cluster(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// Named barrier 2: the consumer warps arrive (non-blocking) once the noise rows are in
// global memory; the producer warp waits on it before fetching a tile that holds noise
// slots.  Both are always executed by whole, converged warps.
__device__ __forceinline__ void noise_bar_arrive() {
    asm volatile("barrier.arrive 2, %0;" ::"r"(kThreads) : "memory");
}
__device__ __forceinline__ void noise_bar_sync() {
    asm volatile("barrier.sync 2, %0;" ::"r"(kThreads) : "memory");
}

constexpr int kPartStride = 132;   // floats per row of a CTA's merged partial in smem

// ---------------------------------------------------------------------------------
// Split-KV attention of one layer.  Grid (n_splits, n_head_kv, n_seq) in clusters of
// `cluster` CTAs along x; 5 warps: warps 0-3 compute, warp 4 produces.
//
//   prologue   consumers turn this kv head's 32 query rows by RoPE at committed + i
//              (float32, the step's cos/sin table) into F16 shared memory; the CTA whose
//              tiles hold the noise slots writes the noise block's K (RoPE at
//              committed + j) and V rows of this head to slots cap + j.  Meanwhile the
//              producer already streams the context tiles.
//   main loop  compute warp w owns query rows 16*(w & 1) .. +16 and key half (w >> 1) of
//              every 64-slot tile: S = Q K^T, online softmax, O += P V.
//   merge      the two key halves merge through shared memory; then the CTAs of the
//              cluster merge their (max, sum, numerator) rows through distributed shared
//              memory, each CTA finishing 32 / cluster rows.
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 2)
k_attend(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
         RingDims d, RingDev m, int layer, int kind, float scale_log2,
         const float *__restrict__ q, const uint16_t *__restrict__ k_noise,
         const uint16_t *__restrict__ v_noise, float *__restrict__ o) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sq = smem + kStages * kStageBytes;
    const uint32_t bar0 = smem_u32(sq + kQBytes);   // full[0..S-1], then empty[0..S-1]
    __shared__ volatile int s_abort;
    // merged partial of this CTA (rows x head_dim numerators, then max and sum per row);
    // lives in stage buffer 1, which is idle once the main loop is over
    float *pacc = reinterpret_cast<float *>(smem + kStageBytes);
    float *pml = pacc + kRows * kPartStride;

    const int sp = blockIdx.x, gk = blockIdx.y, s = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = sp * d.tiles_per_split;
    const int t1 = min(d.n_tiles, t0 + d.tiles_per_split);
    const int tn0 = d.cap / kTile, tn1 = (d.cap + d.q_len - 1) / kTile;
    const bool owns_noise = t0 < t1 && t0 <= tn1 && t1 > tn0;
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
    pdl_wait();   // ring state written by begin_step (and earlier kernels) is visible
    // A grid that fits in one wave lets the next kernel's CTAs settle onto idle SMs now;
    // a multi-wave grid must not, or they would take slots its own later CTAs need.
    if (d.single_wave) pdl_trigger();

    const int mb = warp & 1, kh = warp >> 1;
    const int g = lane >> 2, c = lane & 3;
    const int r0 = mb * 16 + g, r1 = r0 + 8;
    float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};

    if (warp == kComputeWarps) {
        // ---------------- producer ----------------
        // The whole warp walks the tile list (so every barrier it meets is met by all 32
        // lanes together); lane 0 alone waits on the stage barriers and issues the copies.
        const int zrow = (s * d.n_layer + layer) * d.n_head_kv + gk;
        bool noise_ready = false;
        int it = 0;
        for (int t = t0; t < t1; ++t) {
            if (flags[t] == 0) continue;
            if (!noise_ready && t >= tn0 && t <= tn1) {
                __syncwarp();
                noise_bar_sync();
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
                    const uint32_t full = bar0 + 8 * stg;
                    const uint32_t dk = smem_u32(smem + stg * kStageBytes);
                    const uint32_t dv = dk + kTileBytes;
                    mbar_expect_tx(full, kStageBytes);
                    tma_load_3d(dk, &tm_k, 0, t * kTile, zrow, full);
                    tma_load_3d(dk + kHalfBox, &tm_k, 64, t * kTile, zrow, full);
                    tma_load_3d(dv, &tm_v, 0, t * kTile, zrow, full);
                    tma_load_3d(dv + kHalfBox, &tm_v, 64, t * kTile, zrow, full);
                }
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            ++it;
        }
        __syncwarp();
        if (!noise_ready) noise_bar_sync();
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
    } else {
        // ---------------- consumers ----------------
        const int tid = threadIdx.x;    // 0..127
        const int half = kHeadDim / 2;
        const float2 *csq = m.rope32 + (int64_t)s * d.q_len * half;
        {   // queries of this kv head, RoPE at committed + i, F16, swizzled like K tiles.
            // Item u = (row, 4 consecutive pairs); every load is issued before any use.
            constexpr int kItems = kRows * (kHeadDim / 2) / 4;          // 512
            constexpr int kPer = kItems / (kComputeWarps * 32);         // 4
            float4 xa[kPer], xb[kPer], ca[kPer], cb[kPer];
#pragma unroll
            for (int b = 0; b < kPer; ++b) {
                const int u = b * kComputeWarps * 32 + tid;
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
                const int u = b * kComputeWarps * 32 + tid;
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
            // noise block of this head: K turned at committed + i, V copied.  Item u =
            // (noise row, 8 consecutive pairs); loads first, then stores.
            const int64_t head = ((int64_t)s * d.n_layer + layer) * d.n_head_kv + gk;
            const int n_items = d.q_len * (half / 8);
            for (int u = tid; u < n_items; u += kComputeWarps * 32) {
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
        noise_bar_arrive();
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
            // every lane waits (each needs the barrier's acquire of the copied bytes); the
            // vote keeps the warp together if the bounded wait ever gives up
            if (!__all_sync(0xffffffffu, mbar_wait(bar0 + 8 * stg, ph))) {
                if (lane == 0) atomicOr(m.err, kErrWaitFull);
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

        // merge the two key halves through stage buffer 0 (idle now)
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
        if (kh == 0) {
            const int rr[2] = {r0, r1};
            const bool clustered = cluster_size() > 1;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float m1 = xm[(mb * 2 + j) * 32 + lane], l1 = xl[(mb * 2 + j) * 32 + lane];
                const float mm = fmaxf(mrow[j], m1);
                const float muse = mm == -INFINITY ? 0.f : mm;
                const float a0 = exp2f(mrow[j] - muse), a1 = exp2f(m1 - muse);
                const float ll = lrow[j] * a0 + l1 * a1;
                float vals[32];
#pragma unroll
                for (int n = 0; n < 16; ++n) {
                    vals[2 * n] = oacc[n][2 * j] * a0 + xo[(mb * 64 + n * 4 + 2 * j) * 32 + lane] * a1;
                    vals[2 * n + 1] = oacc[n][2 * j + 1] * a0 + xo[(mb * 64 + n * 4 + 2 * j + 1) * 32 + lane] * a1;
                }
                const int r = rr[j];
                if (clustered) {
                    // to this CTA's shared memory; the cluster merges below
                    float *dst = pacc + r * kPartStride;
#pragma unroll
                    for (int n = 0; n < 16; ++n)
                        *reinterpret_cast<float2 *>(dst + n * 8 + 2 * c) = make_float2(vals[2 * n], vals[2 * n + 1]);
                    if (c == 0) {
                        pml[2 * r] = mm;
                        pml[2 * r + 1] = ll;
                    }
                } else if (d.groups == 1) {
                    // the only CTA of this (sequence, kv head): final output
                    if (r < d.rows) {
                        const int hh = r / d.q_len, i = r - hh * d.q_len;
                        const int h = gk * d.group + hh;
                        const float inv = ll > 0.f ? 1.f / ll : 0.f;
                        float *dst = o + (((int64_t)s * d.q_len + i) * d.n_head + h) * kHeadDim;
#pragma unroll
                        for (int n = 0; n < 16; ++n)
                            *reinterpret_cast<float2 *>(dst + n * 8 + 2 * c) =
                                make_float2(vals[2 * n] * inv, vals[2 * n + 1] * inv);
                    }
                } else {
                    // one of several independent CTAs: partial for the combine kernel
                    const int64_t base = (((int64_t)s * d.n_head_kv + gk) * d.groups + sp) * kRows + r;
                    float *dst = m.part_acc + base * kHeadDim;
#pragma unroll
                    for (int n = 0; n < 16; ++n)
                        *reinterpret_cast<float2 *>(dst + n * 8 + 2 * c) = make_float2(vals[2 * n], vals[2 * n + 1]);
                    if (c == 0) m.part_ml[base] = make_float2(mm, ll);
                }
            }
        }
    }

    const uint32_t nct = cluster_size();
    if (nct == 1) return;
    cluster_sync();     // every CTA's merged partial is in its shared memory

    // ---------------- cluster merge: this CTA finishes 32 / cluster rows ----------------
    const uint32_t rank = cluster_rank();
    const int rows_per = kRows / (int)nct;
    if (threadIdx.x < kHeadDim) {
        const int col = threadIdx.x;
        const uint32_t pacc_a = smem_u32(pacc), pml_a = smem_u32(pml);
        const int group = sp / (int)nct;
        for (int rr = (int)rank * rows_per; rr < ((int)rank + 1) * rows_per; ++rr) {
            float mv[16], lv[16], av[16];
#pragma unroll
            for (int cr = 0; cr < 16; ++cr) {
                if (cr < (int)nct) {
                    mv[cr] = ld_cluster(map_rank(pml_a + 8 * rr, cr));
                    lv[cr] = ld_cluster(map_rank(pml_a + 8 * rr + 4, cr));
                    av[cr] = ld_cluster(map_rank(pacc_a + 4 * (rr * kPartStride + col), cr));
                }
            }
            float mm = -INFINITY;
#pragma unroll
            for (int cr = 0; cr < 16; ++cr)
                if (cr < (int)nct) mm = fmaxf(mm, mv[cr]);
            const float muse = mm == -INFINITY ? 0.f : mm;
            float l = 0.f, acc = 0.f;
#pragma unroll
            for (int cr = 0; cr < 16; ++cr) {
                if (cr < (int)nct) {
                    const float w = exp2f(mv[cr] - muse);
                    l += w * lv[cr];
                    acc += w * av[cr];
                }
            }
            if (d.groups == 1) {
                if (rr < d.rows) {
                    const int hh = rr / d.q_len, i = rr - hh * d.q_len;
                    const int h = gk * d.group + hh;
                    o[(((int64_t)s * d.q_len + i) * d.n_head + h) * kHeadDim + col] = l > 0.f ? acc / l : 0.f;
                }
            } else {
                const int64_t base = (((int64_t)s * d.n_head_kv + gk) * d.groups + group) * kRows + rr;
                m.part_acc[base * kHeadDim + col] = acc;
                if (col == 0) m.part_ml[base] = make_float2(mm, l);
            }
        }
    }
    cluster_sync();     // keep this CTA's shared memory alive until the cluster has read it
}

// ---------------------------------------------------------------------------------
// Combine the per-group partials (log-sum-exp merge) when one cluster does not cover a
// (sequence, kv head).  Grid (n_head_kv, n_seq), 256 threads: thread -> (row r = tid / 8,
// 16 columns).
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
k_attend_combine(RingDims d, RingDev m, float *o) {
    const int gk = blockIdx.x, s = blockIdx.y;
    const int r = threadIdx.x >> 3, c0 = (threadIdx.x & 7) * 16;
    if (r >= d.rows) return;
    const int64_t base = ((int64_t)s * d.n_head_kv + gk) * d.groups;
    float mm = -INFINITY;
    for (int sp = 0; sp < d.groups; ++sp) mm = fmaxf(mm, m.part_ml[(base + sp) * kRows + r].x);
    const float muse = mm == -INFINITY ? 0.f : mm;
    float acc[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) acc[k] = 0.f;
    float l = 0.f;
    for (int sp = 0; sp < d.groups; ++sp) {
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

size_t attend_smem_bytes() { return (size_t)kSmemBytes; }

cudaError_t attend_kernels_init() {
    cudaError_t e = cudaFuncSetAttribute(k_attend, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_attend, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
}

int attend_max_cluster() {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(16, 1, 1);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    int n = 1;
    if (cudaOccupancyMaxPotentialClusterSize(&n, k_attend, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 1;
    }
    return n;
}

cudaError_t launch_attend(const RingDims &d, const RingDev &m, const CUtensorMap *tm_k,
                          const CUtensorMap *tm_v, int layer, int kind, float scale_log2,
                          const float *q, const uint16_t *k_noise, const uint16_t *v_noise,
                          float *o, bool pdl, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(d.n_splits, d.n_head_kv, d.n_seq);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = d.cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, k_attend, *tm_k, *tm_v, d, m, layer, kind, scale_log2, q,
                              k_noise, v_noise, o);
}

cudaError_t launch_attend_combine(const RingDims &d, const RingDev &m, float *o,
                                  cudaStream_t st) {
    k_attend_combine<<<dim3(d.n_head_kv, d.n_seq), 256, 0, st>>>(d, m, o);
    return cudaGetLastError();
}

}  // namespace dflash
