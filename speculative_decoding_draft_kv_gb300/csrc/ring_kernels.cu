// Ring append (fold-in and bulk) and device-side mask construction.
//
// Page "DFLASH2_RING_PORT.md": section 1.2 (slot = p % cap, slot_pos[slot] = p, RoPE at
// absolute positions), section 1.3 (fold-in of a_step rows with pad rows routed to
// trash_slot; bulk append in chunks when n_new > a_step) and section 1.4 (mask_full,
// mask_swa).  These kernels move a few KiB per step; they are latency-bound, so they
// are written for few instructions per row rather than for bandwidth.
#include "ring_internal.h"

#include <cuda_fp16.h>

namespace dflash {
namespace {

constexpr int kAppendThreads = 128;
constexpr int kMaskThreads = kTile;   // one thread per slot of a tile

__device__ __forceinline__ double h2d(uint16_t bits) {
    return (double)__half2float(__ushort_as_half(bits));
}

__device__ __forceinline__ uint16_t d2h(double x) {
    return __half_as_ushort(__double2half(x));   // round to nearest even
}

// cos/sin of position `pos` for every rotary pair, float64 (inv_freq from the host).
__device__ __forceinline__ void rope_table(double *cs_cos, double *cs_sin, int64_t pos,
                                           const double *inv_freq, int half) {
    for (int j = threadIdx.x; j < half; j += blockDim.x) {
        double s, c;
        sincos((double)pos * inv_freq[j], &s, &c);
        cs_cos[j] = c;
        cs_sin[j] = s;
    }
}

// Write context row `row` (position p) into slot p % cap of every layer of sequence s:
// K turned by RoPE at p (NeoX pairs j, j + head_dim/2; float64 products rounded once to
// F16), V copied.  Called by a whole block after rope_table() for p.
__device__ void append_row(const RingDims &d, const RingDev &m, int s, int64_t p,
                           int64_t row, const uint16_t *k_rows, const uint16_t *v_rows,
                           int64_t n_rows, const double *cs_cos, const double *cs_sin) {
    const int slot = (int)(p % d.cap);
    const int hd = d.head_dim, half = hd / 2;
    for (int layer = 0; layer < d.n_layer; ++layer) {
        const uint16_t *ks = k_rows + ((int64_t)layer * n_rows + row) * d.kv_row;
        const uint4 *vs = reinterpret_cast<const uint4 *>(v_rows + ((int64_t)layer * n_rows + row) * d.kv_row);
        const int64_t head0 = ((int64_t)s * d.n_layer + layer) * d.n_head_kv;
        for (int idx = threadIdx.x; idx < d.n_head_kv * half; idx += blockDim.x) {
            const int g = idx / half, j = idx - g * half;
            const double x1 = h2d(ks[g * hd + j]);
            const double x2 = h2d(ks[g * hd + j + half]);
            const double c = cs_cos[j], sn = cs_sin[j];
            const double y1 = __dsub_rn(__dmul_rn(x1, c), __dmul_rn(x2, sn));
            const double y2 = __dadd_rn(__dmul_rn(x1, sn), __dmul_rn(x2, c));
            uint16_t *dst = m.k + ((head0 + g) * d.kv_total + slot) * hd;
            dst[j] = d2h(y1);
            dst[j + half] = d2h(y2);
        }
        const int vec_per_head = hd / 8;
        for (int idx = threadIdx.x; idx < d.n_head_kv * vec_per_head; idx += blockDim.x) {
            const int g = idx / vec_per_head, cidx = idx - g * vec_per_head;
            uint4 *dst = reinterpret_cast<uint4 *>(m.v + ((head0 + g) * d.kv_total + slot) * hd);
            dst[cidx] = vs[g * vec_per_head + cidx];
        }
    }
    if (threadIdx.x == 0) m.slot_pos[(int64_t)s * d.cap + slot] = (int32_t)p;
}

// Fold-in append: grid (a_step, n_seq).  Block i appends real row i of the step when
// i < fold_rows, otherwise it is a pad row and writes zeros to trash_slot.
__global__ void __launch_bounds__(kAppendThreads)
k_fold_append(RingDims d, RingDev m, const uint16_t *k_rows, const uint16_t *v_rows,
              int64_t n_rows) {
    __shared__ double cs_cos[kHeadDim / 2], cs_sin[kHeadDim / 2];
    const int i = blockIdx.x, s = blockIdx.y;
    const SeqStep st = m.steps[s];
    if (i < st.fold_rows) {
        const int64_t p = st.start + i;
        rope_table(cs_cos, cs_sin, p, m.inv_freq, d.head_dim / 2);
        __syncthreads();
        append_row(d, m, s, p, st.src_row + i, k_rows, v_rows, n_rows, cs_cos, cs_sin);
        return;
    }
    const int vec_per_head = d.head_dim / 8;
    const uint4 zero = make_uint4(0, 0, 0, 0);
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

// Bulk append, one chunk of bulk_chunk rows: grid (bulk_chunk, n_seq).  Only sequences
// that took the bulk path (n_new > a_step) do anything.
__global__ void __launch_bounds__(kAppendThreads)
k_bulk_append(RingDims d, RingDev m, const uint16_t *k_rows, const uint16_t *v_rows,
              int64_t n_rows, int chunk) {
    __shared__ double cs_cos[kHeadDim / 2], cs_sin[kHeadDim / 2];
    const int s = blockIdx.y;
    const SeqStep st = m.steps[s];
    if (st.n_new <= d.a_step) return;
    const int64_t i = (int64_t)chunk * d.bulk_chunk + blockIdx.x;
    if (i >= st.n_new) return;
    const int64_t p = st.start + i;
    rope_table(cs_cos, cs_sin, p, m.inv_freq, d.head_dim / 2);
    __syncthreads();
    append_row(d, m, s, p, st.src_row + i, k_rows, v_rows, n_rows, cs_cos, cs_sin);
}

// Masks from slot_pos: grid (n_tiles, n_seq), one thread per slot.  Writes the F32 mask
// rows of every kind and one visibility flag per tile and kind.
__global__ void __launch_bounds__(kMaskThreads)
k_build_mask(RingDims d, RingDev m) {
    const int tile = blockIdx.x, s = blockIdx.y;
    const int slot = tile * kTile + threadIdx.x;
    const SeqStep st = m.steps[s];
    const bool in_range = slot < d.kv_total;
    bool ctx_full = false, ctx_swa = false;
    int noise_j = -1;
    if (slot < d.cap) {
        const int64_t p = m.slot_pos[(int64_t)s * d.cap + slot];
        ctx_full = p >= st.lo && p < st.committed;
        ctx_swa = p >= st.swa_lo && p < st.committed;
    } else if (slot < d.cap + d.q_len) {
        noise_j = slot - d.cap;
    }
    const float ninf = __int_as_float(0xff800000);

    // mask_full: the same row for every query (noise block bidirectional)
    {
        float *mk = m.mask + (int64_t)s * d.n_kinds * d.q_len * d.kv_total;
        const bool vis = ctx_full || noise_j >= 0;
        if (in_range)
            for (int i = 0; i < d.q_len; ++i) mk[(int64_t)i * d.kv_total + slot] = vis ? 0.f : ninf;
        const int all = __syncthreads_and(in_range && vis);
        const int any = __syncthreads_or(in_range && vis);
        if (threadIdx.x == 0)
            m.flags[((int64_t)s * d.n_kinds) * d.n_tiles + tile] = any ? (all ? 1 : 2) : 0;
    }
    if (d.n_kinds > 1) {
        // mask_swa: window anchored at committed for every row; noise causal (j <= i)
        float *mk = m.mask + ((int64_t)s * d.n_kinds + 1) * d.q_len * d.kv_total;
        bool all_rows = true, any_row = false;
        for (int i = 0; i < d.q_len; ++i) {
            const bool vis = ctx_swa || (noise_j >= 0 && noise_j <= i);
            if (in_range) mk[(int64_t)i * d.kv_total + slot] = vis ? 0.f : ninf;
            all_rows = all_rows && vis;
            any_row = any_row || vis;
        }
        const int all = __syncthreads_and(in_range && all_rows);
        const int any = __syncthreads_or(in_range && any_row);
        if (threadIdx.x == 0)
            m.flags[((int64_t)s * d.n_kinds + 1) * d.n_tiles + tile] = any ? (all ? 1 : 2) : 0;
    }
}

}  // namespace

cudaError_t launch_fold_append(const RingDims &d, const RingDev &m, const uint16_t *k_rows,
                               const uint16_t *v_rows, int64_t n_rows, cudaStream_t st) {
    k_fold_append<<<dim3(d.a_step, d.n_seq), kAppendThreads, 0, st>>>(d, m, k_rows, v_rows, n_rows);
    return cudaGetLastError();
}

cudaError_t launch_bulk_append(const RingDims &d, const RingDev &m, const uint16_t *k_rows,
                               const uint16_t *v_rows, int64_t n_rows, int chunk,
                               cudaStream_t st) {
    k_bulk_append<<<dim3(d.bulk_chunk, d.n_seq), kAppendThreads, 0, st>>>(d, m, k_rows, v_rows,
                                                                         n_rows, chunk);
    return cudaGetLastError();
}

cudaError_t launch_build_mask(const RingDims &d, const RingDev &m, cudaStream_t st) {
    k_build_mask<<<dim3(d.n_tiles, d.n_seq), kMaskThreads, 0, st>>>(d, m);
    return cudaGetLastError();
}

}  // namespace dflash
