// Ring append (fold-in and bulk) and device-side mask construction.
//
// Page "DFLASH2_RING_PORT.md": section 1.2 (slot = p % cap, slot_pos[slot] = p, RoPE at
// absolute positions), section 1.3 (fold-in of a_step rows with pad rows routed to
// trash_slot; bulk append in chunks when n_new > a_step; noise positions committed + i)
// and section 1.4 (mask_full, mask_swa).  These kernels move a few KiB per step: they are
// latency-bound, so one kernel does the whole fold-in step (append, slot_pos, masks, tile
// flags and the RoPE table of the noise positions) instead of a chain of small launches.
#include "ring_internal.h"

#include <cuda_fp16.h>

namespace dflash {
namespace {

constexpr int kBeginThreads = 128;

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// cos/sin of position `pos` for every rotary pair (see rope_angle_cs).
__device__ __forceinline__ void rope_table(float2 *cs, int64_t pos, const double *inv_freq,
                                           int half) {
    for (int j = threadIdx.x; j < half; j += blockDim.x) cs[j] = rope_angle_cs(pos, inv_freq[j]);
}

// Write context row `row` (position p) into slot p % cap of every layer of sequence s:
// K turned by RoPE at p (NeoX pairs j, j + head_dim/2, float32 products, one rounding to
// F16), V copied.  Called by a whole block after rope_table() for p.  Work item u is
// (layer, kv head, 8 consecutive pairs); all of a thread's loads are issued before any of
// its stores, so a row costs one memory round trip instead of one per item.
// q8_0 slots: the same items; the four items of one 32-value block sit on four
// consecutive lanes (item u and thread index agree modulo 8), which quantise it together
// (q8_quant8).  Every thread runs every round so that the shuffles see full warps.
__device__ void append_row_q8(const RingDims &d, const RingDev &m, int s, int64_t p,
                              int64_t row, const uint16_t *__restrict__ k_rows,
                              const uint16_t *__restrict__ v_rows, int64_t n_rows,
                              const float2 *cs) {
    const int slot = (int)(p % d.cap);
    const int hd = d.head_dim, half = hd / 2;
    const int chunks = half / 8;
    const int n_items = d.n_layer * d.n_head_kv * chunks;
    for (int base = 0; base < n_items; base += (int)blockDim.x) {
        const int u = base + (int)threadIdx.x;
        const bool ok = u < n_items;
        const int uu = ok ? u : 0;
        const int layer = uu / (d.n_head_kv * chunks);
        const int g = (uu / chunks) % d.n_head_kv, jc = uu % chunks;
        const int64_t src = ((int64_t)layer * n_rows + row) * d.kv_row + g * hd + jc * 8;
        uint4 xa = make_uint4(0, 0, 0, 0), xb = xa, va = xa, vb = xa;
        if (ok) {
            xa = *reinterpret_cast<const uint4 *>(k_rows + src);
            xb = *reinterpret_cast<const uint4 *>(k_rows + src + half);
            va = *reinterpret_cast<const uint4 *>(v_rows + src);
            vb = *reinterpret_cast<const uint4 *>(v_rows + src + half);
        }
        const uint16_t *a16 = reinterpret_cast<const uint16_t *>(&xa);
        const uint16_t *b16 = reinterpret_cast<const uint16_t *>(&xb);
        const uint16_t *va16 = reinterpret_cast<const uint16_t *>(&va);
        const uint16_t *vb16 = reinterpret_cast<const uint16_t *>(&vb);
        float k1[8], k2[8], v1[8], v2[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float2 r = rope_rotate(a16[e], b16[e], cs[jc * 8 + e]);
            k1[e] = r.x;
            k2[e] = r.y;
            v1[e] = __half2float(__ushort_as_half(va16[e]));
            v2[e] = __half2float(__ushort_as_half(vb16[e]));
        }
        float dk1, dk2, dv1, dv2;
        const uint2 ck1 = q8_quant8(k1, &dk1), ck2 = q8_quant8(k2, &dk2);
        const uint2 cv1 = q8_quant8(v1, &dv1), cv2 = q8_quant8(v2, &dv2);
        if (!ok) continue;
        const int64_t head = ((int64_t)s * d.n_layer + layer) * d.n_head_kv + g;
        const int64_t dst = (head * d.kv_total + slot) * hd + jc * 8;
        *reinterpret_cast<uint2 *>(m.kq + dst) = ck1;
        *reinterpret_cast<uint2 *>(m.kq + dst + half) = ck2;
        *reinterpret_cast<uint2 *>(m.vq + dst) = cv1;
        *reinterpret_cast<uint2 *>(m.vq + dst + half) = cv2;
        if ((jc & 3) == 0) {
            const int64_t sb = (head * d.kv_total + slot) * (hd / 32);
            const int b1 = jc >> 2, b2 = (half >> 5) + (jc >> 2);
            m.ks[sb + b1] = __half_as_ushort(__float2half_rn(dk1));
            m.ks[sb + b2] = __half_as_ushort(__float2half_rn(dk2));
            m.vs[sb + b1] = __half_as_ushort(__float2half_rn(dv1));
            m.vs[sb + b2] = __half_as_ushort(__float2half_rn(dv2));
        }
    }
    if (threadIdx.x == 0) m.slot_pos[(int64_t)s * d.cap + slot] = (int32_t)p;
}

__device__ void append_row(const RingDims &d, const RingDev &m, int s, int64_t p,
                           int64_t row, const uint16_t *__restrict__ k_rows,
                           const uint16_t *__restrict__ v_rows, int64_t n_rows,
                           const float2 *cs) {
    if (d.kv_q8) {
        append_row_q8(d, m, s, p, row, k_rows, v_rows, n_rows, cs);
        return;
    }
    constexpr int kBatch = 4;
    const int slot = (int)(p % d.cap);
    const int hd = d.head_dim, half = hd / 2;
    const int chunks = half / 8;                          // 8-pair chunks per head
    const int n_items = d.n_layer * d.n_head_kv * chunks;
    for (int base = 0; base < n_items; base += kBatch * (int)blockDim.x) {
        uint4 xa[kBatch], xb[kBatch], xv[kBatch][2];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int u = base + b * (int)blockDim.x + (int)threadIdx.x;
            if (u < n_items) {
                const int layer = u / (d.n_head_kv * chunks);
                const int g = (u / chunks) % d.n_head_kv, jc = u % chunks;
                const int64_t src = ((int64_t)layer * n_rows + row) * d.kv_row + g * hd + jc * 8;
                xa[b] = *reinterpret_cast<const uint4 *>(k_rows + src);
                xb[b] = *reinterpret_cast<const uint4 *>(k_rows + src + half);
                xv[b][0] = *reinterpret_cast<const uint4 *>(v_rows + src);
                xv[b][1] = *reinterpret_cast<const uint4 *>(v_rows + src + half);
            }
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int u = base + b * (int)blockDim.x + (int)threadIdx.x;
            if (u < n_items) {
                const int layer = u / (d.n_head_kv * chunks);
                const int g = (u / chunks) % d.n_head_kv, jc = u % chunks;
                const int64_t head = ((int64_t)s * d.n_layer + layer) * d.n_head_kv + g;
                const int64_t dst = (head * d.kv_total + slot) * hd + jc * 8;
                const uint16_t *a16 = reinterpret_cast<const uint16_t *>(&xa[b]);
                const uint16_t *b16 = reinterpret_cast<const uint16_t *>(&xb[b]);
                uint4 ya, yb;
                uint16_t *ya16 = reinterpret_cast<uint16_t *>(&ya);
                uint16_t *yb16 = reinterpret_cast<uint16_t *>(&yb);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float2 r = rope_rotate(a16[e], b16[e], cs[jc * 8 + e]);
                    ya16[e] = __half_as_ushort(__float2half_rn(r.x));
                    yb16[e] = __half_as_ushort(__float2half_rn(r.y));
                }
                *reinterpret_cast<uint4 *>(m.k + dst) = ya;
                *reinterpret_cast<uint4 *>(m.k + dst + half) = yb;
                *reinterpret_cast<uint4 *>(m.v + dst) = xv[b][0];
                *reinterpret_cast<uint4 *>(m.v + dst + half) = xv[b][1];
            }
        }
    }
    if (threadIdx.x == 0) m.slot_pos[(int64_t)s * d.cap + slot] = (int32_t)p;
}

// Pad row of the fold-in path: zeros to trash_slot of every layer (reading: pad rows are
// zeros, so concurrent pad writers agree and the slot stays finite).
__device__ void pad_row(const RingDims &d, const RingDev &m, int s) {
    const int vec_per_head = d.head_dim / 8;
    const uint4 zero = make_uint4(0, 0, 0, 0);
    if (d.kv_q8) {                       // all-zero blocks: codes 0, scales 0
        for (int layer = 0; layer < d.n_layer; ++layer) {
            const int64_t head0 = ((int64_t)s * d.n_layer + layer) * d.n_head_kv;
            for (int idx = threadIdx.x; idx < d.n_head_kv * (d.head_dim / 16); idx += blockDim.x) {
                const int g = idx / (d.head_dim / 16), c = idx % (d.head_dim / 16);
                const int64_t off = ((head0 + g) * d.kv_total + d.trash_slot) * d.head_dim;
                reinterpret_cast<uint4 *>(m.kq + off)[c] = zero;
                reinterpret_cast<uint4 *>(m.vq + off)[c] = zero;
                if (c == 0) {
                    const int64_t so = ((head0 + g) * d.kv_total + d.trash_slot) * (d.head_dim / 32);
                    *reinterpret_cast<uint2 *>(m.ks + so) = make_uint2(0, 0);
                    *reinterpret_cast<uint2 *>(m.vs + so) = make_uint2(0, 0);
                }
            }
        }
        return;
    }
    for (int layer = 0; layer < d.n_layer; ++layer) {
        const int64_t head0 = ((int64_t)s * d.n_layer + layer) * d.n_head_kv;
        for (int idx = threadIdx.x; idx < d.n_head_kv * vec_per_head; idx += blockDim.x) {
            const int g = idx / vec_per_head, cidx = idx - g * vec_per_head;
            const int64_t off = ((head0 + g) * d.kv_total + d.trash_slot) * d.head_dim;
            reinterpret_cast<uint4 *>(m.k + off)[cidx] = zero;
            reinterpret_cast<uint4 *>(m.v + off)[cidx] = zero;
        }
    }
}

// Masks, visibility bits and flags of one 64-slot tile.  The slot_pos a slot holds after
// this step is computed here rather than read back: a slot written by this step's rows
// holds start + k with k = (slot - start) mod cap < n_new (whichever kernel writes it: the
// fold-in blocks of this grid, the bulk kernels before it, or the producer, which may run
// after it); any other slot keeps its value.
// Threads 0-63 own one slot each (warps 0 and 1); warps 2 and 3 only join the barriers.
__device__ void mask_tile(const RingDims &d, const RingDev &m, int s, int tile, const SeqStep &st) {
    const int slot = tile * kTile + (int)threadIdx.x;
    const bool active = threadIdx.x < kTile;
    const bool in_range = active && slot < d.kv_total;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qw = (d.q_len + 1) & ~1;
    bool ctx_full = false, ctx_swa = false;
    int noise_j = -1;
    if (active && slot < d.cap) {
        const int64_t k = ((int64_t)slot - st.start % d.cap + d.cap) % d.cap;
        const int64_t p = k < st.n_new ? st.start + k
                                           : (int64_t)m.slot_pos[(int64_t)s * d.cap + slot];
        ctx_full = p >= st.lo && p < st.committed;
        ctx_swa = p >= st.swa_lo && p < st.committed;
    } else if (active && slot < d.cap + d.q_len) {
        noise_j = slot - d.cap;
    }
    const float ninf = __int_as_float(0xff800000);
    for (int kind = 0; kind < d.n_kinds; ++kind) {
        const int64_t fi = ((int64_t)s * d.n_kinds + kind) * d.n_tiles + tile;
        float *mk = m.mask + ((int64_t)s * d.n_kinds + kind) * d.q_len * d.kv_total;
        uint32_t *bits = reinterpret_cast<uint32_t *>(m.maskbits + fi * qw);
        bool all_rows = true, any_row = false;
        for (int i = 0; i < qw; ++i) {
            // mask_full: window [lo, c), noise bidirectional; mask_swa: window anchored at
            // committed for every row, noise causal (j <= i)
            bool vis = false;
            if (i < d.q_len)
                vis = kind == 0 ? (ctx_full || noise_j >= 0)
                                : (ctx_swa || (noise_j >= 0 && noise_j <= i));
            vis = vis && in_range;
            if (in_range && i < d.q_len) mk[(int64_t)i * d.kv_total + slot] = vis ? 0.f : ninf;
            if (warp < 2) {
                const uint32_t b = __ballot_sync(0xffffffffu, vis);
                if (lane == 0) bits[2 * i + warp] = b;
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
}

// One begin_step for every sequence: grid (a_step + n_tiles + 1, n_seq).
//   blocks [0, a_step)                 fold-in row i (real row, or pad row to trash)
//   blocks [a_step, a_step + n_tiles)  mask rows and flags of one tile
//   block  a_step + n_tiles            cos/sin of the noise positions committed + i
// The work of one block of the begin-step kernel.
__device__ __forceinline__ void begin_block(const RingDims &d, const RingDev &m,
                                            const uint16_t *__restrict__ k_rows,
                                            const uint16_t *__restrict__ v_rows, int64_t n_rows,
                                            const SeqStep *host_steps, float2 *cs) {
    const int b = blockIdx.x, s = blockIdx.y;
    // the step's records: straight from the host's pinned staging slot when given (no
    // copy ahead of the launch), else from the device copy
    const SeqStep st = host_steps ? host_steps[s] : m.steps[s];
    if (b < d.a_step) {
        if (b < st.fold_rows) {
            if (!k_rows) return;        // the producer kernel writes the row and slot_pos
            const int64_t p = st.start + b;
            rope_table(cs, p, m.inv_freq, d.head_dim / 2);
            __syncthreads();
            append_row(d, m, s, p, st.src_row + b, k_rows, v_rows, n_rows, cs);
        } else {
            pad_row(d, m, s);
        }
        return;
    }
    if (b < d.a_step + d.n_tiles) {
        mask_tile(d, m, s, b - d.a_step, st);
        return;
    }
    const int half = d.head_dim / 2;
    for (int idx = threadIdx.x; idx < d.q_len * half; idx += blockDim.x) {
        const int i = idx / half, j = idx - i * half;
        m.rope32[((int64_t)s * d.q_len + i) * half + j] = rope_angle_cs(st.committed + i, m.inv_freq[j]);
    }
    // the whole-step attention kernel's counters start every step at zero (the previous
    // step's kernel has finished: this grid, or the producer before it, waited for it)
    if (s == 0)
        for (int idx = threadIdx.x; idx < d.step_sync_words; idx += blockDim.x) m.step_sync[idx] = 0u;
}

// wait_end = 0: the previous kernel may still read the ring state -- wait for it first.
// wait_end = 1: the previous kernel is the producer of this step's rows, which waited for
// everything before it and writes none of what this grid reads or writes (the new rows'
// slot_pos is computed here, not read): run alongside it, and wait for it only before
// exiting, so that the kernels after this grid see its rows too.
__global__ void __launch_bounds__(kBeginThreads)
k_begin_step(RingDims d, RingDev m, const uint16_t *__restrict__ k_rows,
             const uint16_t *__restrict__ v_rows, int64_t n_rows, const SeqStep *host_steps,
             int wait_end) {
    __shared__ float2 cs[kHeadDim / 2];
    if (!wait_end) pdl_wait();
    // one small wave: the first attention kernel may settle its CTAs right away (it waits
    // for this grid to finish before reading anything)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // kernel clock: a new step (the attention launches read the counter after this grid;
    // a producer before it read it before it let this grid start)
    if (m.clock && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
        unsigned int *step = reinterpret_cast<unsigned int *>(m.clock + 2 * kClockKinds * kClockSlots);
        *step = *step + 1u;
    }
    begin_block(d, m, k_rows, v_rows, n_rows, host_steps, cs);
    if (wait_end) pdl_wait();
}

// Bulk append, one chunk of bulk_chunk rows: grid (bulk_chunk, n_seq).  Only sequences
// that took the bulk path (n_new > a_step) do anything.
__global__ void __launch_bounds__(kBeginThreads)
k_bulk_append(RingDims d, RingDev m, const uint16_t *__restrict__ k_rows,
              const uint16_t *__restrict__ v_rows, int64_t n_rows, int chunk) {
    __shared__ float2 cs[kHeadDim / 2];
    const int s = blockIdx.y;
    const SeqStep st = m.steps[s];
    if (st.n_new <= d.a_step) return;
    const int64_t i = (int64_t)chunk * d.bulk_chunk + blockIdx.x;
    if (i >= st.n_new) return;
    const int64_t p = st.start + i;
    rope_table(cs, p, m.inv_freq, d.head_dim / 2);
    __syncthreads();
    append_row(d, m, s, p, st.src_row + i, k_rows, v_rows, n_rows, cs);
}

}  // namespace

cudaError_t launch_bulk_append(const RingDims &d, const RingDev &m, const uint16_t *k_rows,
                               const uint16_t *v_rows, int64_t n_rows, int chunk,
                               cudaStream_t st) {
    k_bulk_append<<<dim3(d.bulk_chunk, d.n_seq), kBeginThreads, 0, st>>>(d, m, k_rows, v_rows,
                                                                        n_rows, chunk);
    return cudaGetLastError();
}

cudaError_t launch_begin_step(const RingDims &d, const RingDev &m, const uint16_t *k_rows,
                              const uint16_t *v_rows, int64_t n_rows, bool pdl,
                              const SeqStep *host_steps, cudaStream_t st, bool after_producer) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(d.a_step + d.n_tiles + 1, d.n_seq);
    cfg.blockDim = dim3(kBeginThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_begin_step, d, m, k_rows, v_rows, n_rows, host_steps,
                              after_producer ? 1 : 0);
}

}  // namespace dflash
