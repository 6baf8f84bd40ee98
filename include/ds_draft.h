/*
 * ds_draft.h -- C ABI of the draft-block sampling, confidence scheduling and
 * lossless verification hot path (one GPU, NVIDIA GB300 / sm_103a).
 *
 * Method sources (cited by page and section):
 *   [DSpark]  "DSpark: 반자기회귀 생성과 신뢰도 기반 검증으로 speculative decoding
 *             가속하기" -- sections 배경 (background: draft/verify cycle, lossless
 *             rejection rule), 방법론 › 반자기회귀 생성 (semi-autoregressive
 *             generation, Markov head), 방법론 › 신뢰도 기반 검증 (confidence head,
 *             STS, survival, hardware-aware prefix scheduler).
 *   [DFlash]  "[vLLM] MTP & DFlash" -- section DFlashProposer 초기화 (one bonus
 *             token plus K drafted tokens per request and cycle).
 *   [Philox]  Salmon et al., "Parallel random numbers: as easy as 1, 2, 3", SC'11.
 *
 * Conventions shared by every call:
 *   - Ownership: the caller allocates every buffer, including the workspace;
 *     the library never allocates, frees or keeps a pointer after returning.
 *   - Asynchrony: compute calls enqueue kernels on `stream` and return; no call
 *     synchronises except ds_check_status.
 *   - Errors: arguments the host can check are validated before anything is
 *     launched; a failing check returns a non-zero ds_status and launches
 *     nothing. Conditions only the device can see (token id out of range, a
 *     NaN or +inf logit, a bad temperature) are written to the caller's
 *     device word `status` (first error wins) and leave the outputs undefined.
 *     The caller zeroes `status` before the cycle and reads it with
 *     ds_check_status afterwards.
 *   - Layout: row-major, the last index contiguous; token ids are int32.
 *     Device pointers must be 16-byte aligned.
 *   - Limits: 1 <= B, 1 <= K <= 64, B*K <= 16384, 8 <= V, V % 8 == 0,
 *     16 <= r <= 1024, r % 16 == 0, d % 8 == 0. A logit of -inf has zero
 *     probability; NaN and +inf are errors. Sampling temperatures are 0
 *     (greedy) or in [1e-3, 1e3].
 *   - Randomness: one uniform per decision, u = (w0 + 0.5) * 2^-32 where w0 is
 *     word 0 of Philox4x32-10 with key (seed & 0xffffffff, seed >> 32) and
 *     counter (request, position, stage, 0); positions are 1-based. The draft
 *     and verify calls take the key by value, or from a device word
 *     (`seed_ptr`) read when the kernels run.
 *   - CUDA graphs: no call synchronises, allocates or reads device memory on
 *     the host, so a whole cycle can be captured on a stream and replayed.
 *     Per-replay state lives on the device: the Philox key behind `seed_ptr`
 *     and the asynchronous scheduler's ring (budgets and cycle counter).
 *   - Reentrancy: stateless; calls with distinct outputs and workspaces may run
 *     concurrently on different streams.
 */
#ifndef DS_DRAFT_H
#define DS_DRAFT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* ds_stream_t; /* a cudaStream_t; NULL is the legacy default stream */

typedef enum {
  DS_OK = 0,
  DS_ERR_INVALID_ARG = 1, /* a size, pointer, alignment or mode is out of its range */
  DS_ERR_UNSUPPORTED = 2, /* no device of compute capability 10.3, or a dtype not supported */
  DS_ERR_WORKSPACE = 3,   /* workspace pointer missing or smaller than *_workspace_bytes */
  DS_ERR_CUDA = 4,        /* a CUDA runtime call failed (launch or query) */
  DS_ERR_TIMEOUT = 5,     /* a bounded device-side wait gave up */
  DS_ERR_BOUNDS = 6,      /* a token id read from device memory is outside [0, V) */
  DS_ERR_NONFINITE = 7    /* a NaN or +inf logit, or a row with no finite logit */
} ds_status;

typedef enum { DS_F32 = 0, DS_BF16 = 1 } ds_dtype;

enum { DS_STAGE_DRAFT = 0, DS_STAGE_ACCEPT = 1, DS_STAGE_RESAMPLE = 2 };

enum {
  DS_SCHED_GREEDY_EARLYSTOP = 0, /* [DSpark] 신뢰도 기반 검증: global greedy + early stop */
  DS_SCHED_FIXED_K = 1,          /* verify every drafted token (scheduler off) */
  DS_SCHED_THRESHOLD = 2,        /* static survival threshold (the page's threshold sweep) */
  DS_SCHED_ASYNC = 3             /* [DSpark] 프로덕션 배포 결과: budget from two cycles back,
                                    dynamic top-k on the current survivals */
};

/*
 * Per-position statistics of a draft distribution, written by ds_draft_block
 * for every sampled (T > 0) position and read back by ds_verify. With
 * t_i = (z_i + bias_i) * log2(e) / T, the draft probability of token i is
 *     q_i = 2^(t_i - ref) / (sum_hi + sum_lo).
 * For greedy positions sum_hi = 1, sum_lo = 0, ref = 0 and `argmax` holds the
 * chosen token; for sampled positions argmax = -1.
 */
typedef struct {
  float sum_hi;
  float sum_lo;
  int32_t ref;
  int32_t argmax;
} ds_row_stats;

/* ------------------------------------------------------------------------ */
/* Randomness                                                                */
/* ------------------------------------------------------------------------ */

/* [Philox] Philox4x32-10: ten rounds of two 32x32->64 multiplies (constants
 * 0xD2511F53, 0xCD9E8D57) with a Weyl key schedule (0x9E3779B9, 0xBB67AE85).
 * Host function; `ctr`, `key`, `out` are host arrays of 4, 2 and 4 words. */
void ds_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);

/* The cycle's uniform for (seed, request, position, stage), exact in double,
 * strictly inside (0, 1). Host function. */
double ds_uniform(uint64_t seed, uint32_t request, uint32_t position, uint32_t stage);

/* Device evaluation of the same generator, for checking the kernels' copy:
 * ctr is a device array [n][4], out a device array [n][4]; key as above. */
ds_status ds_philox_fill(const uint32_t* ctr, uint32_t key0, uint32_t key1, uint32_t* out,
                         int32_t n, ds_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Draft block: sequential head (Markov or RNN) + sequential sampling        */
/* ------------------------------------------------------------------------ */

/*
 * [DSpark] 방법론 › 반자기회귀 생성. For k = 1..K, with x_0 = anchor[b]:
 *     l_k = z_k + E[x_{k-1}] . P             (Markov head: low-rank first-order bias)
 *     x_k ~ softmax(l_k / T_b)                (T_b = 0: argmax, lowest index on ties)
 * The draw is the inverse CDF in token order: x = min{i : u * S < C_i} with
 * u = U(seed, b, k, DS_STAGE_DRAFT). The loop is sequential over k and
 * parallel over requests and vocabulary; the V-wide logits are never stored.
 *
 * RNN head (head = DS_HEAD_RNN; same section: a recurrent state over the
 * whole drafted prefix, updated from the state, the previous token's
 * embedding and the backbone hidden state by a gated update). The state s_k
 * (size r) replaces E[x_{k-1}] as the input of P:  l_k = z_k + s_k . P, with
 *     g_i = W_ih [E[x_{k-1}] ; h_k] + b_ih,  g_h = W_hh s_{k-1} + b_hh  (rows:
 *           reset, update, new; the cuDNN GRU cell),  s_0 = 0,
 *     r = sigmoid(g_i^r + g_h^r), u = sigmoid(g_i^u + g_h^u),
 *     n = tanh(g_i^n + r * g_h^n), s_k = (1 - u) * n + u * s_{k-1},
 * each s_k rounded to bfloat16 (nearest even), the storage type. bfloat16
 * only, 64 <= r <= 256 with r % 64 == 0, d % 64 == 0 (DS_ERR_UNSUPPORTED
 * otherwise); the workspace is
 * ds_draft_workspace_bytes(B, K, V, r) + ds_rnn_workspace_bytes(B, K, r)
 * bytes. The states are returned for ds_verify.
 */
typedef enum { DS_HEAD_MARKOV = 0, DS_HEAD_RNN = 1 } ds_head;

typedef struct {
  int32_t B, K, V, r;
  int32_t dtype;              /* ds_dtype of base_logits, E and P */
  const void* base_logits;    /* [B][K][V]  z_k, the parallel backbone's logits */
  const void* E;              /* [V][r]     Markov embedding table */
  const void* P;              /* [r][V]     Markov projection */
  const void* P_t;            /* [V][r]     optional token-major copy of P written by
                                            ds_transpose_projection, or NULL */
  const int32_t* anchor;      /* [B]        x_0, the last verified token */
  const float* temperature;   /* [B]        sampling temperature, 0 = greedy */
  uint64_t seed;              /* Philox key */
  int32_t* draft_tokens;      /* out [B][K] x_k */
  float* q_token;             /* out [B][K] q_k(x_k) (1.0 for greedy positions) */
  ds_row_stats* q_stats;      /* out [B][K] statistics of q_k, read by ds_verify */
  void* workspace;            /* scratch, ds_draft_workspace_bytes(B, K, V, r) bytes
                                 (+ ds_rnn_workspace_bytes for the RNN head) */
  size_t workspace_bytes;
  int32_t* status;            /* device word, see Errors above */
  /* RNN head only (ignored for DS_HEAD_MARKOV, the value of a zeroed struct): */
  int32_t head;               /* ds_head */
  int32_t d;                  /* hidden size */
  const void* h;              /* [B][K][d]  backbone hidden states h_k */
  const void* rnn_w_ih;       /* [3r][r + d] input weights, columns [embedding ; hidden] */
  const void* rnn_w_step;     /* [4r][2r]   W_ih and W_hh packed by ds_rnn_pack_weights */
  const float* rnn_b_ih;      /* [3r] */
  const float* rnn_b_hh;      /* [3r] */
  void* states;               /* out [B][K][r] s_k of every position (bfloat16) */
  const uint64_t* seed_ptr;   /* optional device word holding the Philox key (overrides `seed`) */
  const void* P_packed;       /* optional tile-packed copy of P written by ds_pack_projection
                                 (bfloat16, 64 <= r <= 256, r % 64 == 0), or NULL; results do
                                 not depend on it, the tensor-core tiles load it faster */
} ds_draft_args;

size_t ds_draft_workspace_bytes(int32_t B, int32_t K, int32_t V, int32_t r);
ds_status ds_draft_block(const ds_draft_args* args, ds_stream_t stream);

/* Extra workspace of the RNN head (0 if the shape is outside its limits). */
size_t ds_rnn_workspace_bytes(int32_t B, int32_t K, int32_t r);

/*
 * Weight layout of the RNN head, once per model (like ds_transpose_projection):
 * packs W_ih [3r][r + d] and W_hh [3r][r] into W_step [4r][2r] so that each
 * block of 16 state units has its reset, update, new-input and new-recurrent
 * rows over [embedding ; state] next to each other. Bit-exact copy (zeros
 * where a gate does not read an input). bfloat16 only; r, d multiples of 64.
 */
ds_status ds_rnn_pack_weights(const void* W_ih, const void* W_hh, int32_t r, int32_t d, int32_t dtype,
                              void* W_step, ds_stream_t stream);

/*
 * Tile-packed copy of the Markov projection, once per model (like
 * ds_transpose_projection): for each 128-token tile, its r x 128 slice of P in
 * the 128-byte-swizzled shared-memory image the tensor cores read (64-row
 * k-blocks of two 64-token halves; in each 64 x 128-byte half, the 16-byte
 * unit u of row m stored at unit u ^ (m % 8)); tokens past V are zero. With it
 * the tile kernel brings each 32 KB stage in with one bulk copy instead of one
 * tensor copy per 128-byte row. bfloat16 only, 64 <= r <= 256, r % 64 == 0
 * (DS_ERR_UNSUPPORTED otherwise); P and P_packed device pointers, 16-byte
 * aligned, not overlapping; P_packed holds ds_packed_projection_bytes(r, V)
 * bytes (0 for unsupported shapes), packed_bytes its size (DS_ERR_WORKSPACE if
 * smaller). A bit-exact rearrangement of P.
 */
size_t ds_packed_projection_bytes(int32_t r, int32_t V);
ds_status ds_pack_projection(const void* P, int32_t r, int32_t V, int32_t dtype, void* P_packed,
                             size_t packed_bytes, ds_stream_t stream);

/*
 * Token-major copy of the Markov projection: P_t[v][k] = P[k][v] for
 * v < V, k < r (bit-exact copy, dtype as P). P is a weight of the draft head
 * ([DSpark] 방법론 › 반자기회귀 생성), so this is a once-per-model layout step,
 * run when the weights are loaded. With P_t given, the per-step draw reads the
 * r weights of the 32 tokens it refines as one contiguous block instead of r
 * rows strided by V; results are the same up to the summation order of that
 * 32-token bias (a float rounding difference). Shapes follow the limits
 * above; P and P_t are device pointers, 16-byte aligned, not overlapping.
 */
ds_status ds_transpose_projection(const void* P, int32_t r, int32_t V, int32_t dtype, void* P_t,
                                  ds_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Confidence head, survival and prefix scheduler                            */
/* ------------------------------------------------------------------------ */

/*
 * [DSpark] 방법론 › 신뢰도 기반 검증.
 *     c_k = sigmoid((w_h . h_k + w_e . E[x_{k-1}] + bias) / sts_temp[k])
 *     s_k = c_1 * ... * c_k                    (survival, monotone in k)
 * GREEDY_EARLYSTOP: candidates (b, k) sorted by s descending (ties: k then b
 * ascending); starting from N = B, A = B, J = SPS(B), each candidate is taken
 * iff J' = SPS(N+1) * (A + s) / (N+1) > J, and the walk stops at the first
 * candidate that is not taken. SPS(n) = sps[min(n, n_max) - 1].
 * FIXED_K: L_b = K. THRESHOLD: L_b = #{k : s_k >= threshold}.
 * ASYNC ([DSpark] 주요 결과 › 프로덕션 배포 결과, 한계와 주의사항): with
 * c = budget_ring[2] (the cycle counter, kept on the device), the number of
 * drafted tokens to verify this cycle is M = budget_ring[c & 1], the
 * GREEDY_EARLYSTOP count computed two cycles earlier (or the caller's initial
 * value), so the verify batch B + min(M, B*K) is fixed before this cycle's
 * confidences exist; the M candidates taken are the first M of the same sorted
 * order on the current survivals (prefix-closed). The call then stores this
 * cycle's GREEDY_EARLYSTOP count in budget_ring[c & 1] for cycle c + 2 and
 * sets budget_ring[2] = c + 1. The caller initialises the ring once as
 * {initial, initial, 0, 0}; nothing on the host changes between cycles, so the
 * cycle can be replayed from a CUDA graph.
 * The objective J is evaluated in double-float arithmetic, stored as double.
 */
typedef struct {
  int32_t B, K, d, r, V;
  int32_t dtype;              /* ds_dtype of h, E, w_h and w_e */
  const void* h;              /* [B][K][d]  backbone hidden states */
  const void* E;              /* [V][r]     Markov embedding table */
  const int32_t* anchor;      /* [B] */
  const int32_t* draft_tokens;/* [B][K] */
  const void* w_h;            /* [d] */
  const void* w_e;            /* [r] */
  float bias;                 /* b */
  const float* sts_temp;      /* [K] per-position STS temperatures (> 0) */
  const float* sps;           /* [n_max] SPS(n) for n = 1..n_max (tokens/s) */
  int32_t n_max;
  int32_t mode;               /* DS_SCHED_* */
  float threshold;            /* DS_SCHED_THRESHOLD only */
  int32_t* budget_ring;       /* DS_SCHED_ASYNC only: [4] device words {budget, budget, cycle, 0},
                                 16-byte aligned, updated by the call */
  float* conf;                /* out [B][K] c_k */
  float* conf_logit;          /* out [B][K] raw logit w_h.h_k + w_e.E[x_{k-1}] + b (before the
                                 temperature), the input of ds_sts_fit; may be NULL */
  float* survival;            /* out [B][K] s_k */
  int32_t* sched_len;         /* out [B]    L_b in [0, K] */
  double* objective;          /* out [1]    J at the chosen lengths */
  void* workspace;            /* ds_sched_workspace_bytes(B, K) bytes */
  size_t workspace_bytes;
  int32_t* status;
} ds_sched_args;

size_t ds_sched_workspace_bytes(int32_t B, int32_t K);
ds_status ds_confidence_schedule(const ds_sched_args* args, ds_stream_t stream);

/* ------------------------------------------------------------------------ */
/* STS calibration fit                                                       */
/* ------------------------------------------------------------------------ */

/*
 * [DSpark] 방법론 › 신뢰도 기반 검증 (Sequential Temperature Scaling) and
 * 주요 결과 (over-confident raw head; ECE lowered by STS). Fits the per-position
 * temperatures sts_temp used by ds_confidence_schedule, left to right, on a
 * calibration set of N samples. For k = 1..K, with T_1..T_{k-1} already fitted:
 *     pred_n(T) = prod_{j<k} sigmoid(a_nj / T_j) * sigmoid(a_nk / T)
 *     lab_n     = prod_{j<=k} y_nj
 *     ECE(T)    = sum over n_bins equal-width bins of [0, 1] (bin = floor(pred * n_bins),
 *                 clamped to the last) of |sum_{n in bin} (lab_n - pred_n)| / N
 *     T_k       = the first grid point with the smallest ECE.
 * a_nk is the raw confidence logit w_h . h_k + w_e . E[x_{k-1}] + b (before
 * the temperature; ds_confidence_schedule returns it in conf_logit) and y_nk
 * in [0, 1] the soft per-step acceptance label (the pages train on the
 * analytic rate 1 - TV(p_k, q_k)). Arithmetic: float32 with double-float
 * reductions, deterministic (no atomically accumulated sums).
 * Limits: 1 <= N <= 2^26, 1 <= K <= 64, 1 <= n_grid <= 4096, 1 <= n_bins <= 64.
 * Device-side errors: a non-finite logit -> DS_ERR_NONFINITE; a label outside
 * [0, 1] or a grid value that is not a positive finite number -> DS_ERR_INVALID_ARG.
 */
typedef struct {
  int32_t N, K;               /* calibration samples, positions */
  int32_t n_grid, n_bins;
  const float* logits;        /* [N][K] raw confidence logits a */
  const float* labels;        /* [N][K] soft per-step labels y */
  const float* grid;          /* [n_grid] candidate temperatures */
  float* sts_temp;            /* out [K] fitted T_k (a grid value) */
  int32_t* grid_index;        /* out [K] index of T_k in grid */
  float* ece;                 /* out [K] ECE at T_k */
  float* ece_curve;           /* out [K][n_grid] ECE at every grid point; may be NULL */
  void* workspace;            /* ds_sts_workspace_bytes(N, K, n_grid, n_bins) bytes */
  size_t workspace_bytes;
  int32_t* status;
} ds_sts_args;

size_t ds_sts_workspace_bytes(int32_t N, int32_t K, int32_t n_grid, int32_t n_bins);

/*
 * The STS fit's soft labels ([DSpark] 방법론 › 신뢰도 기반 검증: the calibration
 * is supervised by the analytic acceptance 1 - TV; [DSpark] 배경: the accept
 * rule min(1, p / q)). For each of `rows` rows n:
 *     alpha[n] = sum_i min(p_n(i), q_n(i)),  p_n = softmax(target[n] / T_n),
 *                                            q_n = softmax(draft[n] / T_n),
 * the probability that a token drawn from q_n passes verification against
 * p_n. T_n = 0 (greedy): 1 if both rows' argmax (lowest index on ties) agree,
 * else 0. target_logits and draft_logits are [rows][V] (dtype), temperature
 * [rows] float32, alpha out [rows] float32 in [0, 1]; all device pointers,
 * 16-byte aligned; V % 8 == 0. Float32 arithmetic (relative error ~1e-5).
 * Device errors: a NaN or +inf logit, or a row without a finite logit ->
 * DS_ERR_NONFINITE; a temperature outside {0} u [1e-3, 1e3] ->
 * DS_ERR_INVALID_ARG (that row's alpha is 0).
 */
ds_status ds_acceptance_rate(const void* target_logits, const void* draft_logits, int32_t rows, int32_t V,
                             int32_t dtype, const float* temperature, float* alpha, int32_t* status,
                             ds_stream_t stream);
ds_status ds_sts_fit(const ds_sts_args* args, ds_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Lossless verification                                                     */
/* ------------------------------------------------------------------------ */

/*
 * [DSpark] 배경: left-to-right rejection sampling that preserves the target
 * distribution. For k = 1..L_b with p_k = softmax(target_k / T_b):
 *     accept iff u * q_k(x_k) < p_k(x_k),   u = U(seed, b, k, DS_STAGE_ACCEPT)
 * At the first rejection k: y ~ normalize(max(0, p_k - q_k)) by inverse CDF
 * with u = U(seed, b, k, DS_STAGE_RESAMPLE); if all L_b pass, the bonus
 * y ~ p_{L_b+1} with u = U(seed, b, L_b+1, DS_STAGE_RESAMPLE) ([DFlash]: the
 * target scores K+1 positions per request). T_b = 0: accept iff x_k is the
 * target argmax; emit the target argmax. q_k is rebuilt from base_logits, E,
 * P and q_stats exactly as ds_draft_block defined it. Target rows are read in
 * position order across requests, and a request's rows after its first
 * rejection are skipped once that rejection is known.
 */
typedef struct {
  int32_t B, K, V, r;
  int32_t dtype;              /* ds_dtype of target_logits, base_logits, E and P */
  const void* target_logits;  /* [B][K+1][V]; only rows j <= sched_len[b] of request b are read */
  const void* base_logits;    /* [B][K][V] */
  const void* E;              /* [V][r] */
  const void* P;              /* [r][V] */
  const void* P_t;            /* [V][r] optional, as in ds_draft_args */
  const int32_t* anchor;      /* [B] */
  const int32_t* draft_tokens;/* [B][K] */
  const float* q_token;       /* [B][K] */
  const ds_row_stats* q_stats;/* [B][K] */
  const int32_t* sched_len;   /* [B] */
  const float* temperature;   /* [B] */
  uint64_t seed;
  int32_t* out_tokens;        /* out [B][K+1]: accepted prefix then y, -1 padded */
  int32_t* accept_count;      /* out [B] */
  int32_t* num_emitted;       /* out [B] = accept_count + 1 */
  void* workspace;            /* ds_verify_workspace_bytes(B, K, V, r) bytes */
  size_t workspace_bytes;
  int32_t* status;
  const void* states;         /* RNN head: [B][K][r] states from ds_draft_block (q_k is rebuilt
                                 with s_k . P); NULL for the Markov head */
  const uint64_t* seed_ptr;   /* optional device word holding the Philox key (overrides `seed`) */
  float* p_token;             /* optional out [B][K], or NULL: p_k(x_k), the target probability
                                 the accept test reads, for every position verify evaluated:
                                 always k <= a_b + 1 (up to and including the first rejection);
                                 a later scheduled position holds it too if its row was read
                                 before the rejection was known, else -1; -1 for k > L_b.
                                 Greedy requests (T = 0): 1 if x_k is the target argmax, else
                                 0 (the point mass). */
  const void* P_packed;       /* optional tile-packed copy of P, as in ds_draft_args */
} ds_verify_args;

size_t ds_verify_workspace_bytes(int32_t B, int32_t K, int32_t V, int32_t r);
ds_status ds_verify(const ds_verify_args* args, ds_stream_t stream);

/*
 * ds_verify without a caller workspace. The pages have no counterpart: this is
 * an integration entry point for callers that cannot allocate device memory
 * (hosts without a device allocator, or serving loops that must not call
 * cudaMalloc/cudaFree, which synchronise the device, between steps).
 * Arguments and results are those of ds_verify; `workspace` and
 * `workspace_bytes` are ignored. The scratch is a file-scope device array of
 * DS_VERIFY_STATIC_SCRATCH_BYTES bytes per device, allocated with the module:
 *   - calls with ds_verify_workspace_bytes(B, K, V, r) above that size return
 *     DS_ERR_WORKSPACE and launch nothing (B = 128, K = 16, V = 151936,
 *     r = 256 needs about 11 MB and fits);
 *   - the first call on a device (with that device current) looks up the
 *     array's address once; make one call per device before any stream capture;
 *     cudaDeviceReset gives the device a new context, where the array may sit
 *     elsewhere: the first call in the new context looks it up again;
 *   - calls whose executions overlap on the same device race on the array:
 *     order them on one stream or with events;
 *   - nothing in the array needs to start at zero.
 */
#define DS_VERIFY_STATIC_SCRATCH_BYTES (16u << 20)
ds_status ds_verify_static(const ds_verify_args* args, ds_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Host-resident target rows                                                 */
/* ------------------------------------------------------------------------ */

/* Copies, for every request b, rows 0..L_b of its target logits from host
 * memory to the device buffer ds_verify reads, with L_b = min(max(lens[b], 0), K)
 * (ds_verify reads no other row of request b: the accepted prefix ends at
 * L_b and the final draw uses row j <= L_b; [DSpark] 배경 on the
 * verification of a scheduled prefix, [DFlash] DFlashProposer 초기화 on the
 * K + 1 target positions per request). One cudaMemcpyAsync per request on
 * `stream`; the call returns once they are enqueued.
 *   dst, src     [B][K+1][row_bytes] (same layout on both sides); `src` is host
 *                memory (pinned for an asynchronous copy), `dst` device memory
 *   lens         host array [B]: the scheduled lengths (ds_confidence_schedule's
 *                sched_len, read back to the host)
 *   bytes_out    optional host word: the number of bytes enqueued
 * Errors: DS_ERR_INVALID_ARG for a null pointer, B < 1, K < 0 or
 * row_bytes == 0 (nothing is enqueued); DS_ERR_CUDA if an enqueue fails
 * (earlier requests' copies stay enqueued). */
ds_status ds_copy_scheduled_rows(void* dst, const void* src, int32_t B, int32_t K, size_t row_bytes,
                                 const int32_t* lens, uint64_t* bytes_out, ds_stream_t stream);

/* The same rows, fetched by a kernel that reads the host buffer over the
 * CPU-GPU link, with L_b taken from the device: `sched_len` is
 * ds_confidence_schedule's device output, so the call can follow the schedule
 * on the same stream with no host round trip (and no per-request copy set-up).
 *   dst          device [B][K+1][row_bytes]
 *   src          pinned host memory of the same layout, mapped into the
 *                device's address space (memory from cudaHostAlloc or
 *                cudaMallocHost on a system with unified addressing)
 *   sched_len    device [B]; L_b = min(max(sched_len[b], 0), K)
 *   bytes_total  optional device counter (unsigned 64-bit): the bytes fetched
 *                are added to it
 * Errors: DS_ERR_INVALID_ARG for a null pointer, B < 1, K < 0, row_bytes
 * not a positive multiple of 16, `dst` or `src` not 16-byte aligned, or `src`
 * not host memory the runtime maps for the device (cudaHostGetDevicePointer
 * fails); nothing is launched then. */
ds_status ds_fetch_scheduled_rows(void* dst, const void* src, int32_t B, int32_t K, size_t row_bytes,
                                  const int32_t* sched_len, uint64_t* bytes_total, ds_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Status and identification                                                 */
/* ------------------------------------------------------------------------ */

/* Synchronises `stream`, reads the device status word and returns it (or
 * DS_ERR_CUDA if the stream reports an error). */
ds_status ds_check_status(const int32_t* device_status, ds_stream_t stream);

/*
 * L2 residency of the Markov projection ([DSpark] 방법론 › 반자기회귀 생성: the
 * sequential loop applies the same P at every block position). Sets the
 * current device's persisting-L2 set-aside to min(bytes, the device maximum)
 * with cudaDeviceSetLimit(cudaLimitPersistingL2CacheSize) and returns the
 * set-aside now in effect (0 on failure). The tensor-core tile kernel loads P
 * with an evict-last L2 priority; with a set-aside at least P's size those
 * lines stay in L2 across the K steps of a block instead of being read from
 * HBM at every step (measured: 116 -> 42 MB of HBM reads per step at
 * B = 128, V = 151936, r = 256). The set-aside belongs to the calling
 * process's context: it lasts until changed (0 releases it) or until the
 * context is destroyed, and it reduces the L2 left to other work of the
 * process. Results do not depend on it.
 */
size_t ds_reserve_persisting_l2(size_t bytes);

/*
 * Test hook for the bounded device waits (not for production use). For every
 * later launch of the tensor-core tile kernel in this process (the draft
 * steps and the final draw of ds_verify, bfloat16 with 64 <= r <= 256):
 *   wait_polls    the number of suspended polls (each up to ~20 us) a wait makes
 *                 before it gives up; 0 restores the default (about a second);
 *   withhold_cta  the index of one CTA whose first epilogue warp withholds its
 *                 arrival at the group-record exchange of that CTA's last tile,
 *                 so that the other epilogue threads' wait runs out; -1: none.
 * At that exchange every TMA copy and MMA of the CTA has completed, so the CTA
 * records DS_ERR_TIMEOUT in the status word, releases its tensor memory and
 * returns with nothing in flight; the context stays usable, and later calls
 * (with the hook cleared) run normally. The records that CTA did not write
 * leave the call's outputs undefined. Process-wide, not synchronised with
 * launches already enqueued: set it between calls on an idle device.
 */
ds_status ds_test_set_wait_hooks(uint32_t wait_polls, int32_t withhold_cta);

/* Static description of a status code. */
const char* ds_status_string(ds_status s);

/* Library version, "major.minor.patch". */
const char* ds_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DS_DRAFT_H */
