// Internal declarations shared by the ring's CUDA translation units.
//
// Device layout of one ring set (n_seq sequences), all allocated once in ring_init:
//   K, V      F16  [n_seq][n_layer][n_head_kv][kv_total][head_dim]
//             (each kv head's slots are contiguous: one 64-slot tile of one head is a
//              16 KiB block that a single 3-D TMA box pair fetches)
//   slot_pos  I32  [n_seq][cap]                         -1 = never written
//   mask      F32  [n_seq][n_kinds][q_len][kv_total]    0 or -inf
//   flags     U8   [n_seq][n_kinds][n_tiles]            0 none / 1 all / 2 mixed visible
//   steps     SeqStep[n_seq]                            this step's window, per sequence
//   q16       F16  [n_seq][n_head_kv][32][head_dim]     RoPE'd queries, GQA-grouped rows
//   part_acc  F32  [n_seq][n_head_kv][n_splits][32][head_dim]  split partial numerators
//   part_ml   F32x2[n_seq][n_head_kv][n_splits][32]            split (max, sum), log2 units
//   err       U32  device error word (bounded waits that ran out)
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda.h>

namespace dflash {

constexpr int kHeadDim = 128;     // head_dim supported by the attention kernel
constexpr int kTile = 64;         // slots per attention tile
constexpr int kRows = 32;         // query rows per kv head held by one CTA (G * q_len, padded)
constexpr int kMaxKinds = 2;      // mask_full, mask_swa

// Device error bits.
constexpr uint32_t kErrWaitFull = 1u;     // consumer timed out on a stage's load
constexpr uint32_t kErrWaitEmpty = 2u;    // producer timed out on a free stage
constexpr uint32_t kErrDrain = 4u;        // producer timed out draining loads on abort

struct SeqStep {
    int64_t committed;   // c
    int64_t lo;          // c - min(c, cap)
    int64_t swa_lo;      // c - min(swa_window, min(c, cap)); equals lo without SWA
    int64_t start;       // first position appended by this step
    int64_t src_row;     // row (within the caller's k_rows/v_rows) of position `start`
    int32_t n_new;       // rows appended by this step
    int32_t fold_rows;   // n_new on the fold-in path, 0 on the bulk path
};

struct RingDims {
    int cap, q_len, head_dim, n_head_kv, n_head, n_layer, n_seq, swa_window;
    int a_step, trash_slot, kv_total, kv_row, group, rows;
    int n_tiles, tiles_per_split, n_splits, n_kinds, bulk_chunk;
};

struct RingDev {
    uint16_t *k, *v;
    int32_t *slot_pos;
    float *mask;
    uint8_t *flags;
    SeqStep *steps;
    uint16_t *q16;
    float *part_acc;
    float2 *part_ml;
    uint32_t *err;
    double *inv_freq;     // [head_dim / 2] theta^(-2i/head_dim), computed on the host
};

// ---- launchers (ring_kernels.cu) ----
cudaError_t launch_fold_append(const RingDims &d, const RingDev &m, const uint16_t *k_rows,
                               const uint16_t *v_rows, int64_t n_rows, cudaStream_t st);
cudaError_t launch_bulk_append(const RingDims &d, const RingDev &m, const uint16_t *k_rows,
                               const uint16_t *v_rows, int64_t n_rows, int chunk,
                               cudaStream_t st);
cudaError_t launch_build_mask(const RingDims &d, const RingDev &m, cudaStream_t st);

// ---- launchers (attn_kernels.cu) ----
cudaError_t launch_attend_prologue(const RingDims &d, const RingDev &m, int layer,
                                   const float *q, const uint16_t *k_noise,
                                   const uint16_t *v_noise, cudaStream_t st);
cudaError_t attend_kernels_init();   // per device, before the first launch
// scale_log2 = log2(e) / sqrt(head_dim): the softmax runs in base 2.
cudaError_t launch_attend_split(const RingDims &d, const RingDev &m, const CUtensorMap *tm_k,
                                const CUtensorMap *tm_v, int layer, int kind, float scale_log2,
                                float *o, cudaStream_t st);
cudaError_t launch_attend_combine(const RingDims &d, const RingDev &m, float *o,
                                  cudaStream_t st);
size_t attend_split_smem_bytes();

}  // namespace dflash
