// Internal declarations shared by the ring's CUDA translation units.
//
// Device layout of one ring set (n_seq sequences), all allocated once in ring_init:
//   K, V      F16  [n_seq][n_layer][n_head_kv][kv_total][head_dim]
//             (each kv head's slots are contiguous: one 64-slot tile of one head is a
//              16 KiB block that a single 3-D TMA box pair fetches)
//   slot_pos  I32  [n_seq][cap]                         -1 = never written
//   mask      F32  [n_seq][n_kinds][q_len][kv_total]    0 or -inf
//   flags     U8   [n_seq][n_kinds][n_tiles]            0 none / 1 all / 2 mixed visible
//   maskbits  U64  [n_seq][n_kinds][n_tiles][qw]        bit b of row i: slot 64*tile + b
//                                                       visible to query i (qw = q_len
//                                                       rounded up to even)
//   steps     SeqStep[n_seq]                            this step's window, per sequence
//   rope32    F32x2[n_seq][q_len][head_dim/2]           cos, sin of the noise positions
//   part_acc  F32  [n_seq][n_head_kv][groups][32][head_dim]  cluster-group partial numerators
//   part_ml   F32x2[n_seq][n_head_kv][groups][32]            their (max, sum), log2 units
//   err       U32  device error word (bounded waits that ran out)
//   step_sync U32  [n_layer] + 1: the whole-step attention kernel's layer counters and
//             abort word (few sequences, ring_step), zeroed by every begin_step
//   clock     U64  kernel clock while enabled: earliest start [kClockKinds][kClockSlots],
//             latest end [kClockKinds][kClockSlots], then the step counter the begin-step
//             kernel advances
//
// Attention work split: n_splits = cluster * groups CTAs per (sequence, kv head), each
// streaming tiles_per_split consecutive 64-slot tiles.  The `cluster` CTAs of a group are
// one thread-block cluster and merge their partial softmax states through distributed
// shared memory; with groups > 1 a combine kernel merges the group partials.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda.h>
#include <cuda_fp16.h>

namespace dflash {

constexpr int kHeadDim = 128;     // head_dim supported by the attention kernel
constexpr int kTile = 64;         // slots per attention tile
constexpr int kRows = 32;         // query rows per kv head held by one CTA (G * q_len, padded)
constexpr int kMaxKinds = 2;      // mask_full, mask_swa
constexpr int kMaxQWords = 32;    // visibility words per tile (q_len <= 32, rounded to even)

// Device error bits.
constexpr uint32_t kErrWaitFull = 1u;     // consumer timed out on a stage's load
constexpr uint32_t kErrWaitEmpty = 2u;    // producer timed out on a free stage
constexpr uint32_t kErrDrain = 4u;        // producer timed out draining loads on abort
constexpr uint32_t kErrWaitNoise = 8u;    // producer timed out on the layer's noise rows
constexpr uint32_t kErrWaitPeer = 16u;    // a CTA timed out waiting on other CTAs

// Whole-step attention kernel (every layer in one launch, few sequences).
constexpr int kMaxStepLayers = 16;   // layers one launch takes
constexpr int kMaxStepTiles = 2048;  // slot tiles per (sequence, kv head): flags staged in smem
// Each of the c CTAs of a pair's cluster owns ceil(32 / c) or fewer query rows and receives
// one state per row from every CTA of the cluster: c * ceil(32 / c) receive slots.
constexpr int kMaxRecvSlots = 40;
constexpr int kMaxStepCluster = 16;

// The 32 query rows of a (sequence, kv head) split over the c CTAs of a cluster: rank k
// finishes rows [cluster_first_row(k, c), cluster_first_row(k + 1, c)), at most
// ceil(32 / c) of them; row r belongs to rank r * c / 32.
__host__ __device__ __forceinline__ int cluster_first_row(int k, int c) { return (k * kRows + c - 1) / c; }

// Kernel clock: one (earliest start, latest end) pair per launch of each kind -- per layer
// of each of the last kClockSteps steps, slot (step % kClockSteps) * kMaxStepLayers + layer
// within the kind's bank: attention (ring_attend, ring_step, ring_draft_step), the
// context-row producer (layer 0: one launch per step), the noise-block projections.
constexpr int kClockSteps = 2048;
constexpr int kClockSlots = kClockSteps * kMaxStepLayers;
constexpr int kClockAttend = 0, kClockProduce = 1, kClockProject = 2, kClockKinds = 3;
constexpr size_t kClockWords = 2 * (size_t)kClockKinds * kClockSlots + 1;

// Per-layer inputs and outputs of one step (layouts as for ring_attend).
struct StepIO {
    const float *q[kMaxStepLayers];
    const uint16_t *k_noise[kMaxStepLayers];
    const uint16_t *v_noise[kMaxStepLayers];
    float *o[kMaxStepLayers];
};

struct SeqStep {
    int64_t committed;   // c
    int64_t lo;          // c - min(c, cap)
    int64_t swa_lo;      // c - min(swa_window, min(c, cap)); equals lo without SWA
    int64_t start;       // first position appended by this step
    int64_t src_row;     // row (within the caller's k_rows/v_rows) of position `start`
    int32_t n_new;       // rows appended by this step
    int32_t fold_rows;   // n_new on the fold-in path, 0 on the bulk path
    int64_t prod_base;   // rows of earlier sequences in the producer's packed row list
};

struct RingDims {
    int cap, q_len, head_dim, n_head_kv, n_head, n_layer, n_seq, swa_window;
    int a_step, trash_slot, kv_total, kv_row, group, rows;
    int n_tiles, tiles_per_split, n_splits, n_kinds, bulk_chunk;
    int cluster, groups;
    int kv_q8;            // slots hold q8_0 blocks (codes + F16 scales) instead of F16
    int single_wave;      // attention grid fits in one wave (all its CTAs resident at once)
    int step_sync_words;  // words of RingDev::step_sync that begin_step zeroes (0: none)
};

struct RingDev {
    uint16_t *k, *v;          // F16 slots [S][L][Hkv][kv_total][128] (F16 rings)
    int8_t *kq, *vq;          // q8_0 codes, same layout (q8_0 rings)
    uint16_t *ks, *vs;        // q8_0 F16 scales [S][L][Hkv][kv_total][4]
    int32_t *slot_pos;
    float *mask;
    uint8_t *flags;
    uint64_t *maskbits;
    SeqStep *steps;
    float2 *rope32;
    float *part_acc;
    float2 *part_ml;
    uint32_t *err;
    double *inv_freq;     // [head_dim / 2] theta^(-2i/head_dim), computed on the host
    uint32_t *step_sync;  // whole-step kernel: layer counters + abort word
    unsigned long long *clock;   // kernel clock while enabled (else NULL)
    uint32_t *probe;      // two words nothing ever writes (bounded-wait self-test)
};

// RoPE angle of position p for the pair with inverse frequency f (= theta^(-2i/d)):
// the angle p * f is formed in float64 (one rounding, as a float64 reference does),
// reduced to [-pi, pi] with a two-part 2*pi, and only then handed to float32 sincosf.
// float64 work per angle is a multiply and two FMAs: this GPU's float64 rate is far
// below its float32 rate, so float64 sin/cos would dominate the small kernels.
__device__ __forceinline__ float2 rope_angle_cs(int64_t p, double f) {
    const double kTwoPiHi = 6.283185307179586;            // nearest double to 2*pi
    const double kTwoPiLo = 2.4492935982947064e-16;        // 2*pi - kTwoPiHi
    const double kInvTwoPi = 0.15915494309189535;
    const double a = (double)p * f;
    const double k = rint(a * kInvTwoPi);
    double r = fma(-k, kTwoPiHi, a);
    r = fma(-k, kTwoPiLo, r);
    float sn, c;
    sincosf((float)r, &sn, &c);
    return make_float2(c, sn);
}

// NeoX rotation of one F16 pair (x1, x2) by (cos, sin): float32 FMAs.
__device__ __forceinline__ float2 rope_rotate(uint16_t x1b, uint16_t x2b, float2 cs) {
    const float x1 = __half2float(__ushort_as_half(x1b));
    const float x2 = __half2float(__ushort_as_half(x2b));
    return make_float2(fmaf(x1, cs.x, -x2 * cs.y), fmaf(x1, cs.y, x2 * cs.x));
}

// q8_0 quantisation of 8 values that are one quarter of a 32-value block, the block's
// four quarters held by lanes 4k .. 4k+3 of a warp: the block maximum by two butterfly
// shuffles (every lane of the warp calls this, lanes without data pass zeros), scale
// d = max|x| / 127, codes roundf(x * (1 / d)) (half away from zero), all in float32.
// Returns the 8 codes packed little-endian and the scale in *d_out.
__device__ __forceinline__ uint2 q8_quant8(const float (&x)[8], float *d_out) {
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[e]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const float d = amax / 127.f;
    const float id = d > 0.f ? 1.f / d : 0.f;
    uint32_t w[2] = {0u, 0u};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        int c = (int)roundf(x[e] * id);
        c = c > 127 ? 127 : (c < -127 ? -127 : c);
        w[e >> 2] |= ((uint32_t)c & 0xffu) << (8 * (e & 3));
    }
    *d_out = d;
    return make_uint2(w[0], w[1]);
}

// ---- launchers (ring_kernels.cu) ----
// Bulk append of one chunk (rows chunk*bulk_chunk ...) for sequences on the bulk path.
cudaError_t launch_bulk_append(const RingDims &d, const RingDev &m, const uint16_t *k_rows,
                               const uint16_t *v_rows, int64_t n_rows, int chunk,
                               cudaStream_t st);
// Fold-in append + slot_pos + masks + tile flags + the step's RoPE table, one kernel.
// pdl: launch with programmatic stream serialization (the kernel waits on its
// predecessor before touching ring state).  host_steps: the step records in pinned host
// memory, read by the kernel directly (NULL: read m.steps, copied to the device before).
// after_producer: the predecessor is the producer of this step's rows (k_rows NULL): the
// kernel runs alongside it and waits for it only before exiting.
cudaError_t launch_begin_step(const RingDims &d, const RingDev &m, const uint16_t *k_rows,
                              const uint16_t *v_rows, int64_t n_rows, bool pdl,
                              const SeqStep *host_steps, cudaStream_t st,
                              bool after_producer = false);

// Row ranges of the producer's packed row list, passed by value (no copy to the device
// before the launch, so the launch can overlap the previous kernel) when n_seq is small.
constexpr int kProduceParamSeqs = 16;
struct ProduceSeqs {
    int n;                                   // sequences described here; 0: use RingDev::steps
    int64_t base[kProduceParamSeqs];         // first packed row of each sequence
    int64_t n_new[kProduceParamSeqs];
    int64_t start[kProduceParamSeqs];        // position of that row
    int64_t src_row[kProduceParamSeqs];      // its feature row
};

// Where the noise-block projection (ProduceJob::mode 1) puts a layer's rows: Q F32
// [n_layer][n_seq][q_len][n_head][128] after q_norm, K and V F16 [n_layer][n_seq][q_len]
// [kv_row] (K after k_norm), all pre-RoPE, as ring_attend takes them.
struct NoiseOut {
    float *q;
    uint16_t *k, *v;
    const float *q_norm;      // [n_layer][128]
};

// One kind of rows in a projection launch.
//   mode 0: the step's new context rows (m_total, packed over sequences), every layer, K and
//           V heads, written into the ring with RoPE at their positions (feat: the fused
//           target features);
//   mode 1: the noise-block rows of layer `layer` (m_total = n_seq * q_len rows of its
//           hidden states; feat: every layer's hidden states, layer-major), Q, K and V
//           heads, written to NoiseOut.
struct ProduceJob {
    int mode;
    int layer;
    int64_t m_total;
    int64_t units;            // 32-row tiles x heads (x layers in mode 0)
};

// One launch of the projection kernel: one or two jobs (a draft step's context rows and
// its first layer's noise rows share a launch), their work units numbered job after job,
// each unit's hidden dimension split over a cluster of ks CTAs.
struct ProduceLaunch {
    ProduceJob job[2];
    int n_jobs;
    int ks;
    int out_heads;            // heads in the packed weights per layer: 2 n_head_kv (+ n_head)
    int single_wave;          // set by launch_produce: every CTA of the grid is resident at
                              // once, so the kernel may release its dependents early
};

// ---- launchers (produce_kernels.cu) ----
cudaError_t produce_kernels_init();   // per device, before the first launch
// W_k, W_v [n_layer][n_head_kv * 128][hidden] (and W_q [n_layer][n_q_heads * 128][hidden]
// when n_q_heads > 0) -> tiles of 128 rows x 64 columns, ordered (layer, K heads, V heads,
// Q heads, k-tile); out holds (2 n_head_kv + n_q_heads) * n_layer * 128 * hidden values.
cudaError_t launch_pack_weights(const uint16_t *wk, const uint16_t *wv, const uint16_t *wq,
                                uint16_t *out, int n_layer, int n_head_kv, int n_q_heads,
                                int hidden, cudaStream_t st);
size_t produce_smem_bytes();
// Split of the hidden dimension over a cluster of 1 .. kProduceMaxSplit CTAs for `units`
// work units: the widest that keeps the grid within 85% of the CTAs resident at once
// (cap[ks], produce_capacity) -- one wave even while the previous kernel still holds some
// SMs -- with at least two 64-column k-tiles per CTA.
constexpr int kProduceMaxSplit = 8;
int produce_split(int64_t units, int hidden, const int *cap);
// CTAs of a producer grid with clusters of ks that are resident at once on sms SMs (0 if
// the occupancy query fails)
int produce_capacity(int ks, int sms);
// Units of a job: 32-row tiles x (2 n_head_kv x n_layer) in mode 0, x out_heads in mode 1.
int64_t produce_units(const RingDims &d, int mode, int64_t m_total, int out_heads);
// The projection launch.  tm_w: 3-D TMA map over the packed weights (launch_pack_weights):
// 64 x 128 x 1 boxes, 128-byte swizzle.  tm_feat[j], feat[j]: job j's input rows, F16
// [rows][hidden], 16-byte aligned, with a 2-D TMA map of 64 x 32 boxes, 128-byte swizzle.
// Mode 0: K = RoPE(k_norm(W_k x)), V = W_v x, rounded to F16 (or quantised to q8_0) and
// stored in their ring slots, with slot_pos; seqs.n == 0: the row ranges are read from
// m.steps (staged before the launch).  Mode 1: Q = q_norm(W_q h), K = k_norm(W_k h),
// V = W_v h into nout.  pdl: launch with programmatic stream serialization; the kernel
// streams its first weight tiles at once (weights are constant while steps run) and waits
// for its predecessor before it reads rows or step records or writes anything; it reads
// the kernel clock's step counter before it releases its dependents.  resident:
// produce_capacity(L.ks).
cudaError_t launch_produce(const RingDims &d, const RingDev &m, const CUtensorMap *tm_w,
                           const CUtensorMap *tm_feat0, const CUtensorMap *tm_feat1,
                           const uint16_t *feat0, const uint16_t *feat1, int hidden,
                           const ProduceLaunch &L, const float *k_norm, float eps,
                           const ProduceSeqs &seqs, const NoiseOut &nout, bool pdl, int resident,
                           cudaStream_t st);

// ---- tensor-core producer (produce_tc.cu): context rows of steps with many new rows ----
// Used from kProduceTcMinRows rows on, when packed row mr is feature row frow_base + mr
// for every new row (one contiguous run).  tm_feat: 2-D TMA map over the features with
// 64 x 128 boxes, 128-byte swizzle.  Same outputs as launch_produce in mode 0.
constexpr int64_t kProduceTcMinRows = 256;
cudaError_t produce_tc_init();        // per device, before the first launch
cudaError_t launch_produce_tc(const RingDims &d, const RingDev &m, const CUtensorMap *tm_w,
                              const CUtensorMap *tm_feat, int hidden, int64_t m_total,
                              int64_t frow_base, int out_heads, const float *k_norm, float eps,
                              const ProduceSeqs &seqs, int sms, bool pdl, cudaStream_t st);

// ---- shared host helpers (ring_host.cu) ----
// 3-D TMA map over F16 K or V laid out [n_seq * n_layer * n_head_kv][kv_total][head_dim],
// 64 x 64 boxes, 128-byte swizzle.
bool encode_kv_tensor_map(CUtensorMap *tm, void *base, const RingDims &d);
// Message returned by ring_last_error(NULL) on this thread.
void set_global_error(const char *msg);

// ---- launchers (attn_kernels.cu) ----
cudaError_t attend_kernels_init();   // per device, before the first launch
// clusters of `cluster` CTAs that can be resident at once (0 if none)
int attend_cluster_capacity(int cluster, bool q8);
// scale_log2 = log2(e) / sqrt(head_dim): the softmax runs in base 2.
// early (bit mask, with pdl only): kAttendPreload -- the kernel may fill its first
// pipeline stages before its grid dependency resolves, valid when the kernel launched just
// before it (if it overlaps at all) writes none of this layer's context K/V, flags or
// visibility bits (so: not right after the begin-step kernel); kAttendInputsReady -- the
// queries, the noise rows and the step's RoPE table were complete before the previous
// kernel started, so the query prologue and the noise-row stores may run before the grid
// dependency too.
constexpr int kAttendPreload = 1, kAttendInputsReady = 2;
cudaError_t launch_attend(const RingDims &d, const RingDev &m, const CUtensorMap *tm_k,
                          const CUtensorMap *tm_v, int layer, int kind, float scale_log2,
                          const float *q, const uint16_t *k_noise, const uint16_t *v_noise,
                          float *o, bool pdl, int early, cudaStream_t st);
cudaError_t launch_attend_combine(const RingDims &d, const RingDev &m, float *o,
                                  cudaStream_t st);
size_t attend_smem_bytes();

// ---- launchers (step_kernels.cu) ----
cudaError_t attend_step_init();      // per device, before the first launch
// clusters of `cluster` CTAs of the whole-step kernel resident at once (0 if none)
int attend_step_capacity(int cluster);
size_t attend_step_smem_bytes();
// Every layer's attention of one step: one cluster of `cluster` CTAs per (sequence, kv
// head), launched cooperatively (CTAs wait on each other, boundedly).  pdl: programmatic
// serialization after the begin-step kernel.
cudaError_t launch_attend_step(const RingDims &d, const RingDev &m, const CUtensorMap *tm_k,
                               const CUtensorMap *tm_v, int kind, float scale_log2,
                               const StepIO &io, int cluster, bool pdl, cudaStream_t st);
// which 0: an mbarrier wait, 1: a wait on another CTA's counter, each given limit_ns and
// bound to run out; the kernel sets kErrWaitFull / kErrWaitPeer and returns.
cudaError_t launch_wait_probe(const RingDev &m, int which, unsigned long long limit_ns,
                              cudaStream_t st);

}  // namespace dflash
