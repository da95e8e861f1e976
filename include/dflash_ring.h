/*
 * dflash_ring.h -- C ABI of the DFlash draft-KV ring step for one GB300 GPU (sm_103a).
 *
 * The draft model of DFlash block-diffusion speculative decoding keeps the K/V rows of
 * its context in a fixed ring of `cap` slots instead of a cache that grows with the
 * prompt.  Source: the page "DFLASH2_RING_PORT.md" (DFlash2 draft KV-ring port to
 * llama.cpp), sections 1.1-1.7.  One step is
 *
 *   ring_begin_step   append the newly committed rows (slot = p % cap, RoPE at p),
 *                     route fold-in pad rows to trash_slot, update slot_pos and
 *                     build mask_full / mask_swa on the device          (sections 1.2-1.4)
 *   ring_attend       per layer: write the noise block to slots cap..cap+q_len-1 and
 *                     run masked GQA attention of the q_len noise queries over the
 *                     kv_total slots                                       (sections 1.3-1.4)
 *
 * Conventions shared by every call
 *   - Every function returns a status (RING_OK or a negative RING_E* code) and never
 *     aborts.  ring_last_error() gives a one-line message for the last failure.
 *   - Argument checks happen on the host before anything is launched; a call that
 *     fails a check changes no state.
 *   - "device pointer" means memory the GPU can read or write directly (cudaMalloc or a
 *     PyTorch CUDA tensor); the caller owns it and keeps it alive until the work queued
 *     on `stream` has finished.  The ring owns only what ring_init allocated.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *     Calls that take a stream only enqueue work and return without synchronising.
 *     Issue all calls on one stream (or order the streams yourself): begin_step
 *     rewrites per-step state that the previous step's attend kernels read.
 *   - Read-back calls (ring_get_*) synchronise the device and copy to host memory.
 *   - Layouts are row-major, innermost index last.  A K/V "row" is kv_row = head_dim *
 *     n_head_kv F16 values, head-major (the page's [kv_row, kv_total] ggml tensor,
 *     section 1.1).  F16 values travel as uint16_t bit patterns.
 *   - Shape limits of the kernels: head_dim == 128 and (n_head / n_head_kv) * q_len
 *     <= 32; other shapes are rejected with RING_EINVAL.
 */
#ifndef DFLASH_RING_H
#define DFLASH_RING_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct dflash_ring ring_t;

enum ring_status {
    RING_OK = 0,
    RING_EINVAL = -1,   /* a bad argument: dimension, kind, layer, sequence, NULL pointer   */
    RING_ERANGE = -2,   /* committed went backwards, exceeds the position range, or the rows
                           passed do not cover [start, committed)                        */
    RING_ENOMEM = -3,   /* a device or pinned-host allocation failed                       */
    RING_ECUDA = -4,    /* a CUDA runtime call failed (message in ring_last_error)         */
    RING_ESTATE = -5,   /* call out of order, e.g. ring_attend before any ring_begin_step  */
    RING_EDEVICE = -6   /* a kernel raised its device-side error flag (a bounded wait ran
                           out); see ring_device_error                                    */
};

enum ring_mask_kind {
    RING_MASK_FULL = 0, /* section 1.4 mask_full: window [lo, committed), noise bidirectional */
    RING_MASK_SWA = 1   /* section 1.4 mask_swa: window [committed - min(swa_window, win),
                           committed), noise causal within the block                      */
};

/* Extended construction parameters.  Zero in an optional field selects its default. */
typedef struct ring_params {
    int32_t cap;             /* ring capacity in context slots (section 1.1)                 */
    int32_t q_len;           /* noise-block length = draft block size (section 1.1)          */
    int32_t head_dim;        /* 128 (the only head size the kernels take)                    */
    int32_t n_head_kv;       /* K/V heads                                                    */
    int32_t n_head;          /* query heads, a multiple of n_head_kv (GQA)                   */
    int32_t n_layer;         /* draft layers sharing the slot map                            */
    float rope_theta;        /* RoPE base; NeoX pairing (i, i + head_dim/2)                  */
    int32_t n_seq;           /* independent rings (sequences); default 1                     */
    int32_t swa_window;      /* SWA window for RING_MASK_SWA; 0 = no SWA mask                */
    int32_t bulk_chunk;      /* rows per bulk-append chunk; default 1024 (section 1.3)       */
    int32_t tiles_per_split; /* attention split length in 64-slot tiles; 0 = chosen from the
                                SM count and the number of (sequence, kv head) pairs          */
    int32_t max_cluster;     /* upper bound on the attention cluster size (1 = no clusters);
                                0 = the largest the device can co-schedule, at most 16        */
    int32_t kv_format;       /* RING_KV_F16 (default) or RING_KV_Q8_0: slots hold q8_0 blocks
                                of 32 values (int8 codes, one F16 scale d = max|x| / 127,
                                codes round(x / d) half away from zero, decided in float32);
                                K is quantised straight from its rotated value, V from its
                                input; pad rows are all-zero blocks.  (Page
                                "DFLASH2_RING_PORT.md", section 1.7: the port's draft-KV
                                size is that of a q8_0 cache.)  A q8_0 ring attends with
                                independent CTAs (no clusters), turning codes into F16 MMA
                                operands on the fly; the producer quantises the rows it makes
                                the same way (V after its F16 rounding).                     */
    int32_t step_split;      /* ring_step's attention: 0 = one launch per layer (default);
                                > 0 = every layer of the step in one persistent kernel, one
                                thread-block cluster of this many CTAs per sequence x kv
                                head pair, one CTA per SM (F16 slots, n_layer <= 16, at most
                                16 CTAs with c * ceil(32 / c) <= 40; refused with EINVAL
                                when that is not met or a cluster per pair does not fit on
                                the GPU at once); -1 = that kernel with the widest such
                                cluster when the pairs are few (else one launch per layer)  */
} ring_params;

enum { RING_KV_F16 = 0, RING_KV_Q8_0 = 1 };

/* Geometry and sizes of an initialised ring (all counts, no pointers). */
typedef struct ring_geometry {
    int32_t cap, q_len, a_step, trash_slot, kv_total, kv_row;
    int32_t head_dim, n_head_kv, n_head, n_layer, n_seq, swa_window, bulk_chunk;
    int32_t tile_slots;      /* slots per attention tile (64)                                */
    int32_t n_tiles;         /* ceil(kv_total / tile_slots)                                  */
    int32_t tiles_per_split; /* tiles streamed by one attention CTA                          */
    int32_t n_splits;        /* CTAs per (sequence, kv head) = cluster * groups              */
    int32_t cluster;         /* CTAs per thread-block cluster; they merge their partial
                                softmax states through distributed shared memory            */
    int32_t groups;          /* clusters per (sequence, kv head); > 1 adds a combine kernel  */
    int64_t cache_bytes;     /* F16 K+V of one sequence: 2 * n_layer * kv_row * kv_total * 2
                                (section 1.7)                                                */
    int64_t device_bytes;    /* everything ring_init allocated on the device                 */
    int32_t step_split;      /* CTAs per (sequence, kv head) -- one cluster -- of ring_step's
                                persistent attention kernel; 0 = ring_step launches each
                                layer                                                        */
    int32_t step_ctas;       /* CTAs of that kernel (step_split * n_seq * n_head_kv)         */
} ring_geometry;

/* Per-kernel timing collected while profiling is on (CUDA events on the launch stream). */
typedef struct ring_profile {
    int64_t launches[6];     /* 0 bulk append chunk, 1 begin-step kernel (fold-in append,
                                slot_pos, masks, flags, RoPE table), 2 attention, 3 group
                                combine, 4 whole-step graph replay (ring_step), 5 context-
                                row producer (ring_begin_step_features)                     */
    double total_ms[6];      /* summed event time per kernel class                          */
} ring_profile;

/*
 * ring_init -- allocate one ring (n_seq = 1, no SWA) on the current CUDA device.
 * Section 1.1: a_step = 2*q_len + 2, trash_slot = cap + q_len,
 * kv_total = align_up(cap + q_len + 1, 32), kv_row = head_dim * n_head_kv; separate F16
 * K and V tensors per layer, zeroed once; slot_pos[] = -1; next position 0.
 * *out receives the handle (NULL on failure).  Errors: EINVAL, ENOMEM, ECUDA.
 */
int ring_init(ring_t **out, int32_t cap, int32_t q_len, int32_t head_dim, int32_t n_head_kv,
              int32_t n_head, int32_t n_layer, float rope_theta);

/* ring_init_ex -- as ring_init with n_seq rings, an SWA window, bulk chunk and split size. */
int ring_init_ex(ring_t **out, const ring_params *params);

/* ring_destroy -- synchronise the device, free everything the ring owns.  NULL is a no-op. */
int ring_destroy(ring_t *r);

/* ring_get_geometry -- fill *g.  Errors: EINVAL (NULL). */
int ring_get_geometry(const ring_t *r, ring_geometry *g);

/*
 * ring_rows_needed -- section 1.3 window arithmetic for sequence `seq` if `committed`
 * were passed to the next begin_step: win = min(c, cap), lo = c - win,
 * start = max(next_pos, lo), n_new = c - start.  Tells a caller which rows to produce.
 * Errors: EINVAL, ERANGE (committed below the ring's next position).
 */
int ring_rows_needed(const ring_t *r, int32_t seq, int64_t committed, int64_t *start,
                     int32_t *n_new);

/*
 * ring_begin_step -- sections 1.2-1.4 for every sequence, enqueued on `stream`.
 *
 *   committed  host int64[n_seq]: tokens committed so far per sequence; never decreases.
 *   k_rows     device F16 [n_layer][n_rows][kv_row]: pre-RoPE context K rows.
 *   v_rows     device F16 [n_layer][n_rows][kv_row]: context V rows.
 *   row_off    host int64[n_seq]: row (within n_rows) holding position first_pos[s].
 *   first_pos  host int64[n_seq]: position of that row; rows of sequence s cover
 *              [first_pos[s], committed[s]) contiguously.
 *   n_rows     rows per layer in k_rows / v_rows (the layer stride).
 *
 * For each sequence with n_new rows to append (see ring_rows_needed): when
 * n_new <= a_step the fold-in path writes a_step rows -- the n_new real rows to slot
 * p % cap with RoPE at p, and the rest as pad rows of zeros to trash_slot; otherwise
 * the bulk path appends all n_new rows in chunks of bulk_chunk rows.  slot_pos[p % cap]
 * = p.  Then mask_full (and mask_swa when swa_window > 0) and their per-tile flags are
 * rebuilt from slot_pos on the device.  Rows below `start` are ignored; k_rows/v_rows
 * may be NULL when no sequence appends.  Positions must stay below 2^31 - q_len.
 * Errors: EINVAL, ERANGE (state unchanged), ECUDA.
 */
int ring_begin_step(ring_t *r, const int64_t *committed, const void *k_rows,
                    const void *v_rows, const int64_t *row_off, const int64_t *first_pos,
                    int64_t n_rows, void *stream);

/*
 * Context-row producer -- page "DFLASH2_RING_PORT.md", test 11, point 4 of the refuted
 * hypotheses: the draft's context K/V rows come from the fused target features by
 * W_k / W_v times the feature vector, then k_norm, then RoPE.  Readings: k_norm is an RMS
 * norm over each kv head's head_dim slice, x / sqrt(mean(x^2) + eps) times one learned
 * weight [head_dim] per layer; V is not normalised; both round once to F16.
 *
 *   hidden   width of one fused feature row; a positive multiple of 64.
 *   eps      k_norm epsilon (>= 0; 1e-6 for the drafts on the page).
 *   wk, wv   device F16 [n_layer][kv_row][hidden], row-major, 16-byte aligned.
 *   k_norm   device F32 [n_layer][head_dim].
 *
 * Synchronous: the weights are copied into ring-owned device memory (W_k and W_v
 * repacked into contiguous 128 x 64 tiles, 2 * n_layer * kv_row * hidden F16 in all; k_norm
 * as is), so the caller's buffers may be freed or changed afterwards -- call again after
 * changing them.  Waits for the device to go idle before replacing earlier weights.
 * p == NULL detaches the producer and frees the copy.  Errors: EINVAL, ENOMEM, ECUDA.
 */
typedef struct ring_producer {
    int32_t hidden;
    float eps;
    const void *wk;
    const void *wv;
    const float *k_norm;
    const void *wq;          /* optional (with q_norm), for ring_draft_step: device F16
                                [n_layer][n_head * head_dim][hidden]                        */
    const float *q_norm;     /* optional: device F32 [n_layer][head_dim], the query heads'
                                RMS-norm weight                                              */
} ring_producer;
int ring_set_producer(ring_t *r, const ring_producer *p);

/*
 * ring_begin_step_features -- ring_begin_step with the context rows made on the device
 * from fused features: for every new position p of every sequence (the same window
 * arithmetic, fold-in and bulk), K = RoPE_p(k_norm(W_k x_p)) and V = W_v x_p of every
 * layer are computed on the tensor cores and written straight into slot p % cap
 * (F16, round to nearest even), with slot_pos; pad rows of the fold-in path still go to
 * trash_slot as zeros; masks and flags as in ring_begin_step.
 *
 *   feat       device F16 [n_rows][hidden], 16-byte aligned: one fused feature row per
 *              position, shared by every layer.
 *   row_off, first_pos, n_rows  as in ring_begin_step (rows of sequence s cover
 *              [first_pos[s], committed[s]) from row row_off[s]).
 *
 * Errors: ESTATE (no producer set), EINVAL, ERANGE (state unchanged), ECUDA.
 */
int ring_begin_step_features(ring_t *r, const int64_t *committed, const void *feat,
                             const int64_t *row_off, const int64_t *first_pos, int64_t n_rows,
                             void *stream);

/*
 * ring_recompute_window -- the page's legacy path (section 1.6: with the ring disabled
 * the draft recomputes the whole window every step; section 1.7: the ring gives the
 * same result): like ring_begin_step_features, but every position of [lo, committed) of
 * every sequence is produced and written again, not only the new ones, so the rows must
 * cover [lo, committed) (first_pos[s] <= lo).  The ring state afterwards is that of
 * ring_begin_step_features up to the rounding order of the projection.  A comparison
 * workload: it costs a projection of min(committed, cap) rows per sequence and layer.
 * Errors: as ring_begin_step_features.
 */
int ring_recompute_window(ring_t *r, const int64_t *committed, const void *feat,
                          const int64_t *row_off, const int64_t *first_pos, int64_t n_rows,
                          void *stream);

/*
 * ring_draft_step -- one whole draft step of the page's one-graph draft forward (section
 * 1.5; the noise block fed in per layer, section 1.6): ring_begin_step_features for the
 * new context rows, then for every layer l in order
 *   the noise-block projections of its hidden states h_l:  Q = q_norm(W_q h),
 *   K = k_norm(W_k h), V = W_v h (the same W_k, W_v, k_norm as the context rows; pre-RoPE),
 *   and the layer's attention with mask kind mask_kinds[l] (a per-layer full / SWA
 *   pattern, as the Luce draft's sliding-window layers), output o[l].
 * Layer 0's hidden states (the noise block's embeddings) are there from the start: its
 * projection shares one launch with the context rows.  Layer l > 0's are read only after
 * layer l - 1's attention has finished (in a draft model they are computed from its
 * output).
 * Needs ring_set_producer with wq and q_norm.
 *
 *   feat, row_off, first_pos, n_rows   as in ring_begin_step_features.
 *   noise_h     device F16 [n_layer][n_seq][q_len][hidden], 16-byte aligned.
 *   mask_kinds  host int32[n_layer]: RING_MASK_FULL or RING_MASK_SWA.
 *   o           host array of n_layer device F32 [n_seq][q_len][n_head][head_dim].
 *
 * Launches in stream order with programmatic serialization between them (each kernel
 * streams its first weight or K/V tiles while its predecessor finishes).
 * Errors: ESTATE (no producer with W_q, or no step yet), EINVAL, ERANGE, ECUDA.
 */
int ring_draft_step(ring_t *r, const int64_t *committed, const void *feat,
                    const int64_t *row_off, const int64_t *first_pos, int64_t n_rows,
                    const void *noise_h, const int32_t *mask_kinds, float *const *o, void *stream);

/*
 * ring_attend -- one draft layer's masked attention, enqueued on `stream`.
 *
 *   q        device F32 [n_seq][q_len][n_head][head_dim]: pre-RoPE noise-block queries.
 *   k_noise  device F16 [n_seq][q_len][kv_row]: pre-RoPE noise-block K rows.
 *   v_noise  device F16 [n_seq][q_len][kv_row]: noise-block V rows.
 *   o        device F32 [n_seq][q_len][n_head][head_dim]: output (overwritten).
 *
 * Noise row j is stored in slot cap + j of this layer with RoPE at committed + j; query
 * i is rotated to committed + i (section 1.3).  Then, per query head h (kv head
 * h / (n_head / n_head_kv)) and row i:
 *   o[i,h] = sum_s softmax_s(q_i . k_s / sqrt(head_dim) + mask[i,s]) v_s,
 * over the kv_total slots with the mask of `mask_kind` built by the last begin_step
 * (section 1.4).  Computed by a split-KV flash-decode kernel (F16 tensor-core products,
 * F32 softmax and accumulation) that skips slot tiles with no visible slot.
 * Errors: EINVAL (layer, kind, NULL, SWA without a window), ESTATE (no begin_step yet),
 * ECUDA.
 */
int ring_attend(ring_t *r, int32_t layer, int32_t mask_kind, const float *q,
                const void *k_noise, const void *v_noise, float *o, void *stream);

/*
 * ring_step -- one whole step as a fixed-topology CUDA graph: ring_begin_step followed by
 * ring_attend for layers 0 .. n_layer-1 with mask `mask_kind`, the layer inputs and
 * outputs given by host arrays of n_layer device pointers (q[l], k_noise[l], v_noise[l],
 * o[l], layouts as for ring_attend).  The page builds its step graph once and replays it
 * every step, feeding new inputs through dedicated buffers (section 1.5); here the graph
 * is captured on the first call and replayed on later ones as long as k_rows, v_rows,
 * n_rows, mask_kind, the layer pointers and the kernel clock setting stay the same (a
 * change re-captures it).  The per-step values (committed counts, row offsets) are staged
 * to the device before the replay; bulk-append chunks, when a sequence needs them, run
 * just before it.
 *
 * The layers run in order: layer l reads its queries and noise rows only after every
 * output of layer l-1 is written, so o[l] may serve as a later layer's q.  With few
 * (sequence, kv head) pairs (ring_geometry.step_split > 0) the attention of all layers is
 * one persistent kernel (one CTA per SM, launched cooperatively): its CTAs stream every
 * layer's context K/V tiles ahead while the layers run, and hand over from layer to layer
 * through counters in device memory with bounded waits (a wait that runs out sets
 * ring_device_error's bits).  Otherwise each layer is its own launch.  The ring state
 * afterwards equals that of the separate calls bit for bit; the outputs equal them up to
 * the order of the softmax merges (the persistent kernel splits the slots differently).
 * Errors: as ring_begin_step and ring_attend.
 */
int ring_step(ring_t *r, const int64_t *committed, const void *k_rows, const void *v_rows,
              const int64_t *row_off, const int64_t *first_pos, int64_t n_rows,
              int32_t mask_kind, const float *const *q, const void *const *k_noise,
              const void *const *v_noise, float *const *o, void *stream);

/* ring_get_slot_pos -- host int32[cap] of sequence `seq` (-1 = never written).  Syncs. */
int ring_get_slot_pos(ring_t *r, int32_t seq, int32_t *out);

/* ring_get_mask -- host F32 [q_len][kv_total] (0 or -inf) of the last begin_step.  Syncs. */
int ring_get_mask(ring_t *r, int32_t seq, int32_t mask_kind, float *out);

/* ring_get_tile_flags -- host uint8[n_tiles]: 0 = no visible slot, 1 = every slot visible
 * to every row, 2 = mixed.  Syncs. */
int ring_get_tile_flags(ring_t *r, int32_t seq, int32_t mask_kind, uint8_t *out);

/* ring_get_kv -- host F16 bits [kv_total][kv_row] of K and V of (seq, layer), in the
 * page's row layout (either pointer may be NULL).  F16 rings only (ESTATE otherwise).
 * Syncs. */
int ring_get_kv(ring_t *r, int32_t seq, int32_t layer, uint16_t *k, uint16_t *v);

/* ring_get_kv_q8 -- q8_0 rings: host int8 codes [kv_total][kv_row] and F16 scale bits
 * [kv_total][kv_row / 32] of K and V of (seq, layer), page row layout (any pointer may be
 * NULL).  ESTATE on an F16 ring.  Syncs. */
int ring_get_kv_q8(ring_t *r, int32_t seq, int32_t layer, int8_t *k_codes, uint16_t *k_scales,
                   int8_t *v_codes, uint16_t *v_scales);

/* ring_device_error -- synchronise, read and clear the device-side error word.  Returns
 * RING_OK, or RING_EDEVICE with the word's bits stored in *bits (may be NULL).  Bits: 1 a
 * consumer's wait for a stage's K/V load ran out, 2 the copy warp's wait for a free stage,
 * 4 draining the copies in flight, 8 the wait for a layer's noise rows, 16 a wait on other
 * CTAs of the persistent whole-step kernel.  Every such wait gives up after 2 s; the
 * kernel then stops its CTA (and, in the whole-step kernel, every other CTA) and returns,
 * and the outputs of that launch are not valid. */
int ring_device_error(ring_t *r, uint32_t *bits);

/* ring_describe -- the geometry line the Luce server logs (section 11, Test 4), e.g.
 * "[draft-kv] ctx-KV ring active: cap=4096 kv_total=4128 a_step=18 layers=5 f16 cache
 * 80.6 MiB", written NUL-terminated into buf[len]. */
int ring_describe(const ring_t *r, char *buf, size_t len);

/* ring_profile_enable -- on != 0 starts recording CUDA events around every kernel the ring
 * launches (not allowed while a stream capture is in progress); 0 stops. */
int ring_profile_enable(ring_t *r, int32_t on);

/* ring_profile_read -- synchronise on the recorded events, add them into *out (which the
 * caller zeroes first) and forget them. */
int ring_profile_read(ring_t *r, ring_profile *out);

/* ring_launch_count -- kernels this ring has launched since ring_init. */
int64_t ring_launch_count(const ring_t *r);

/*
 * Kernel clock -- the duration of the ring's kernels measured on the device, inside CUDA
 * graphs too: each launch records, with the GPU's global nanosecond timer, the earliest
 * moment any of its CTAs passed its grid dependency and the latest moment any CTA was
 * done, in a slot for its kind and layer of that step (every begin-step call starts a
 * step).  Kinds: RING_CLOCK_ATTEND, the attention kernel (one launch per layer, or the
 * persistent whole-step kernel in slot 0); RING_CLOCK_PRODUCE, the context-row producer
 * of ring_begin_step_features, ring_recompute_window and ring_draft_step (one launch per
 * step, slot 0); RING_CLOCK_PROJECT, the noise-block projections of ring_draft_step (one
 * per layer).  The stamps are reductions nobody waits for, so the clock does not slow the
 * launches it times.  A launch that starts before its predecessor ends (programmatic
 * serialization) counts from the moment its dependency resolved: the bytes it fetched
 * before that -- the first weight or K/V stages -- overlap the previous kernel.  (No
 * counterpart on the page: it is how the throughput of a kernel inside a pipelined or
 * replayed step is measured.)
 *
 * ring_clock_enable -- on != 0 starts recording with the next launch (ring_step re-captures
 *   its graph); 0 stops.  Errors: EINVAL.
 * ring_clock_read -- synchronise, return the summed milliseconds of the recorded launches
 *   of kind `kind` and their number, and clear them.  Slots cover the last 2048 steps:
 *   read at least that often; two launches of one kind and layer within one step share a
 *   slot (their joint span).  Either pointer may be NULL.  Errors: EINVAL (kind), ECUDA.
 */
enum { RING_CLOCK_ATTEND = 0, RING_CLOCK_PRODUCE = 1, RING_CLOCK_PROJECT = 2 };
int ring_clock_enable(ring_t *r, int32_t on);
int ring_clock_read(ring_t *r, int32_t kind, double *total_ms, int64_t *launches);

/*
 * ring_check_bounded_wait -- self-test of the kernels' bounded waits (no counterpart on the
 * page; the page's code has no device waits).  Launches one small kernel that waits on
 * something nothing will ever complete -- which = 0: an mbarrier phase no thread arrives
 * at (the wait the attention kernels use for their TMA stages); which = 1: a device
 * counter no CTA raises (the wait the persistent whole-step kernel uses between layers)
 * -- giving up after limit_us microseconds (1 .. 2,000,000).  The kernel then sets the
 * device error word's bit (1 = a stage load timed out, 16 = a wait on other CTAs timed
 * out) and returns; read it with ring_device_error.  Enqueued on `stream`.
 * Errors: EINVAL, ECUDA.
 */
int ring_check_bounded_wait(ring_t *r, int32_t which, int32_t limit_us, void *stream);

/*
 * ring_attend_static -- the attention of ring_attend for callers that cannot allocate
 * device memory (no counterpart on the page: it exists for hosts whose framework owns
 * every device allocation, or that run where a runtime allocation is not allowed, and
 * so cannot create a ring).  Every buffer comes from the caller; nothing is allocated.
 *
 *   k, v       device F16 [n_seq][n_head_kv][kv_total][head_dim]: one layer's ring K/V,
 *              kv_total = align_up(cap + q_len + 1, 32).  In/out: the noise block's rows
 *              are written to slots cap .. cap+q_len-1 exactly as ring_attend writes them.
 *   mask       device F32 [n_seq][q_len][kv_total]: 0 = visible, -inf = hidden (the
 *              layout ring_get_mask returns).
 *   committed  host int64[n_seq]: queries and noise keys turn by RoPE at committed + i.
 *   q, k_noise, v_noise, o   as for ring_attend.
 *
 * Scratch (tile flags, visibility bits, the RoPE table, split partials) lives in one
 * static device array of 16 MiB, which every GPU that loads this library holds until the
 * process exits.  The first call on a device looks up that array's device address (with
 * that device current); make that first call before any stream capture.  Every call on a
 * device shares the array, so calls that overlap on the GPU race: issue them on one
 * stream.  Shapes whose scratch exceeds 16 MiB, or n_seq above 256, fail with
 * RING_ERANGE: the scratch holds 4 bytes of error word, the RoPE table (n_seq * q_len *
 * head_dim * 4 bytes), one flag byte and q_len (rounded up to even) 8-byte visibility
 * words per 64-slot tile and sequence, and -- only when the call splits a (sequence, kv
 * head) over several CTAs, which it does when there are few pairs and halves until the
 * rest fits -- n_seq * n_head_kv * splits * 16.25 KiB of partial states.  A wait that runs
 * out inside the kernel is reported by ring_attend_static_device_error.
 * Errors: EINVAL, ERANGE, ECUDA (message in ring_last_error(NULL)).
 */
typedef struct ring_attend_static_args {
    int32_t cap, q_len, head_dim, n_head_kv, n_head, n_seq;
    float rope_theta;
    const int64_t *committed;
    void *k, *v;
    const float *mask;
    const float *q;
    const void *k_noise, *v_noise;
    float *o;
} ring_attend_static_args;

int ring_attend_static(const ring_attend_static_args *args, void *stream);

/*
 * ring_attend_static_device_error -- the device error word of ring_attend_static on the
 * current device (no counterpart on the page).  The attention kernel gives up a wait that
 * runs out (2 s) and sets a bit instead of hanging; without a ring handle, this is where a
 * caller of ring_attend_static learns of it.  Synchronises the device, reads the word --
 * the bits every call since the last read has set (the same bits as ring_device_error) --
 * and clears it.  Returns RING_OK, or RING_EDEVICE with the bits in *bits (may be NULL);
 * ECUDA if the device could not be read.  Allocates nothing.
 */
int ring_attend_static_device_error(uint32_t *bits);

/* ring_last_error -- message of the last failing call on r (or of the last failed
 * ring_init or ring_attend_static when r is NULL).  Never NULL. */
const char *ring_last_error(const ring_t *r);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH_RING_H */
