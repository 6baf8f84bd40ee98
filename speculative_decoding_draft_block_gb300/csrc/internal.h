// Internal types shared by the kernels and the C-ABI layer (not part of the ABI).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ds_draft.h"

namespace ds {

// One partial-sum record per (row, 32-token chunk).
//   sampling rows: chunk sum (hi + lo) of 2^(t_i - ref), ref the chunk reference
//   greedy rows:   the chunk's largest logit (hi + lo) and its token in `idx`
struct ChunkRec {
  float hi, lo;
  int32_t ref;
  int32_t idx;
};

enum RowMode : int32_t {
  kSkip = 0,
  kGreedyMarkov = 1,  // draft position with T = 0: argmax of z + bias
  kSampleMarkov = 2,  // draft position with T > 0: inverse CDF of softmax((z + bias)/T)
  kResidual = 3,      // verify, first rejection: inverse CDF of max(0, p - q)
  kBonus = 4          // verify, all accepted: inverse CDF of p_{L+1}
};

// Final draw of one request in ds_verify (written by the finalize kernel).
struct FinalDesc {
  int32_t mode;     // kSkip, kResidual or kBonus
  int32_t row;      // 0-based position index j of the target (and base) row
  int32_t a_token;  // token whose E row forms the Markov bias (residual)
  int32_t out_pos;  // where the drawn token goes in out_tokens[b]
  int32_t Np, Nq;   // references of the target and draft rows
  float Rhi, Rlo;   // S_p / S_q as a double-float
};

// Per (request, target row) results of the verify row pass.
struct VRow {
  float s_hi, s_lo;  // S_p = sum 2^(t_i - ref)
  int32_t ref;
  int32_t argmax;    // T = 0 rows
  int32_t accept;    // 1 if the drafted token at this position passed
  int32_t valid;
  int32_t pad[2];
};

struct SampleParams {
  int32_t B, K, V, r, n_chunks;
  int32_t src;   // 0: draft step, 1: final draw of verify
  int32_t step;  // draft: 1-based position k
  int32_t dtype;
  const void* base_logits;    // [B][K][V]
  const void* target_logits;  // [B][K+1][V]
  const void* E;
  const void* P;
  const void* P_t;              // [V][r] token-major copy of P, or null
  const void* P_packed;         // tile-packed copy of P (ds_pack_projection), or null
  const int32_t* anchor;
  const int32_t* draft_tokens;  // [B][K] (read: previous positions; written by locate)
  const float* temperature;
  const FinalDesc* final_desc;  // [B]
  ChunkRec* chunks;             // [n_chunks][B] (chunk-major: a warp's rows store contiguously)
  // Staged A operand: the locate of step k writes E[x_k] rows here
  // (a_stage_out), the tensor-core tile kernel of step k+1 loads them with TMA
  // (a_stage_in). Null where unused (first step, last step, SIMT path).
  const void* a_stage_in;       // [B] rows of r, a_stage_stride elements apart
  void* a_stage_out;            // [B] rows of r, a_stage_stride elements apart
  int32_t a_stage_stride;       // r for the Markov head
  // RNN head: the bias rows are states, not E rows. Draft: row b of the
  // current state at a_rows + b * a_rows_stride; final draw: the state of
  // row j at a_rows + (b * K + j) * r (a_rows_stride = K * r). Null: Markov.
  const void* a_rows;
  int32_t a_rows_stride;
  // Group records: the chunks of a row are also combined per column group
  // (the contiguous token range one tile CTA covers), so that the locate scans
  // a few hundred group records and then the chunks of one group only.
  ChunkRec* supers;   // [B][sup_stride]
  int32_t sup_stride;
  int32_t sup_tiles;  // T: tiles of the launch, M-tile major
  int32_t sup_groups; // G: group g covers tiles [g*T/G, (g+1)*T/G)
  int32_t sup_nt;     // tiles per M-tile (across the vocabulary)
  int32_t sup_cpt;    // 32-token chunks per tile
  int32_t sup_rows;   // rows per M-tile
  uint64_t seed;
  const uint64_t* seed_ptr;   // when set, the key is read from the device
  int32_t* tokens_out;        // draft: draft_tokens; final: out_tokens
  float* q_token;             // draft only
  ds_row_stats* q_stats;      // draft only
  int32_t* status;
};

struct VerifyParams {
  int32_t B, K, V, r, n_chunks, dtype;
  const void* target_logits;
  const int32_t* anchor;
  const int32_t* draft_tokens;
  const float* q_token;
  const ds_row_stats* q_stats;
  const int32_t* sched_len;
  const float* temperature;
  uint64_t seed;
  const uint64_t* seed_ptr;  // when set, the key is read from the device
  VRow* vrows;  // [B][K+1]
  FinalDesc* final_desc;
  int32_t* out_tokens;
  int32_t* accept_count;
  int32_t* num_emitted;
  float* p_token;  // optional [B][K]: p_k(x_k) of the rows evaluated, -1 elsewhere
  // Per request, the lowest position whose accept test rejected (workspace,
  // set to all ones -- none yet -- before the call).
  uint32_t* first_reject;  // [B]
  int32_t* status;
};

struct SchedParams {
  int32_t B, K, d, r, V, dtype, n_max, mode;
  float bias, threshold;
  int32_t* budget_ring;  // DS_SCHED_ASYNC: [4] {budget, budget, cycle, 0}
  const void* h;
  const void* E;
  const int32_t* anchor;
  const int32_t* draft_tokens;
  const void* w_h;
  const void* w_e;
  const float* sts_temp;
  const float* sps;
  float* conf;
  float* conf_logit;  // optional
  float* survival;
  int32_t* sched_len;
  double* objective;
  int32_t* status;
};

// STS fit (sts.cu). The sample chunks per CTA are chosen at launch from the
// SM count; the workspace does not depend on them.
struct StsParams {
  int32_t N, K, G, n_bins, n_chunks, chunk;
  const float* logits;   // [N][K]
  const float* labels;   // [N][K]
  const float* grid;     // [G]
  float* sts_temp;       // [K] out
  int32_t* grid_index;   // [K] out
  float* ece;            // [K] out
  float* ece_curve;      // [K][G] out, optional
  // workspace
  unsigned* ticket;      // last-CTA counter
  float* base;           // [2][N] prefix predictions, by position parity
  float* lab;            // [2][N] prefix labels, by position parity
  long long* hist64;     // [n_bins][G] fixed-point bin totals (zero between positions)
  float* ece_all;        // [G]
  int32_t* status;
};

// RNN head (rnn.cu). One tensor-core GEMM kernel, two epilogues:
//   kGemmBias: out[m][n] = A[m] . W[n] + bias[n]   (the hidden-state part of
//              the gate inputs for every position, once per draft call);
//   kGemmGru:  the gated update of one position; W is the packed step matrix
//              (unit blocks of 32: reset, update, new-input, new-recurrent rows
//              over [e ; s]) and the epilogue writes the new state.
enum GemmEpilogue { kGemmBias = 0, kGemmGru = 1 };
struct GemmParams {
  int32_t B, K, N, Kd;          // requests, positions, output columns, reduction length
  // kGemmBias
  const float* bias;            // [N]
  float* out;                   // gh[K][N][B]
  // kGemmGru, producing the state of position p (1-based)
  const float* gh;              // gh[K][3r][B]: W_ih[:, r:] . h + b_ih
  const float* b_hh;            // [3r]
  const __nv_bfloat16* s_prev;  // row b at s_prev + b * 2r (state half of the input rows)
  __nv_bfloat16* s_next;        // row b at s_next + b * 2r
  __nv_bfloat16* states;        // [B][K][r]
  int32_t r, p;
  int32_t* status;
};
cudaError_t launch_rnn_gemm(const GemmParams& g, int mode, const void* A, const void* W,
                            int64_t w_stride, cudaStream_t s);
cudaError_t launch_rnn_init(const void* E, const int32_t* anchor, int32_t B, int32_t r, int32_t V,
                            void* gru_in, int32_t* status, cudaStream_t s);
cudaError_t launch_rnn_pack(const void* W_ih, const void* W_hh, int32_t r, int32_t d, void* W_step,
                            cudaStream_t s);

// 2-D or 3-D bfloat16 tensor map with 128-byte swizzle (draft_tc.cu).
bool encode_tmap_bf16(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims,
                      const cuuint64_t* strides, const cuuint32_t* box);

constexpr int kTileRows = 32;   // rows per sampling CTA
constexpr int kTileCols = 256;  // tokens per sampling CTA (8 chunks of 32)

inline int32_t num_chunks(int32_t V) { return (V + 31) / 32; }

// Column groups of the tile kernels. Group g covers tiles
// [floor(g*T/G), floor((g+1)*T/G)); the groups meeting M-tile mt are
// first_group(mt) .. last_group(mt), and a row's group records are stored in
// that order (slot = g - first_group(mt)), so slots follow the vocabulary.
constexpr int32_t kMaxTcGroups = 256;
inline int32_t sup_stride_for(int32_t V) {
  const int32_t simt = (V + kTileCols - 1) / kTileCols;
  return simt > kMaxTcGroups ? simt : kMaxTcGroups;
}
__host__ __device__ inline int32_t ceil_div64(int64_t a, int64_t b) { return (int32_t)((a + b - 1) / b); }
__host__ __device__ inline int32_t group_tile0(const SampleParams& p, int32_t g) {
  return (int32_t)((int64_t)g * p.sup_tiles / p.sup_groups);
}
__host__ __device__ inline int32_t first_group(const SampleParams& p, int32_t mt) {
  return ceil_div64(((int64_t)mt * p.sup_nt + 1) * p.sup_groups, p.sup_tiles) - 1;
}
__host__ __device__ inline int32_t last_group(const SampleParams& p, int32_t mt) {
  return ceil_div64((int64_t)(mt + 1) * p.sup_nt * p.sup_groups, p.sup_tiles) - 1;
}

void tc_group_layout(SampleParams& p);
void simt_group_layout(SampleParams& p);
size_t sample_tile_smem_bytes(int32_t r);
size_t locate_smem_bytes(const SampleParams& p);
bool tc_path_supported(int32_t dtype, int32_t r, int32_t V);
// Test hooks of the tensor-core tile kernel (ds_test_set_wait_hooks).
void set_tile_test_hooks(uint32_t wait_polls, int32_t withhold_cta);
cudaError_t launch_tile_tc(const SampleParams& p, cudaStream_t s);
cudaError_t launch_sample_tile(const SampleParams& p, cudaStream_t s);
cudaError_t launch_sample_locate(const SampleParams& p, cudaStream_t s);
cudaError_t launch_verify_rows(const VerifyParams& p, cudaStream_t s);
cudaError_t launch_verify_finalize(const VerifyParams& p, cudaStream_t s);
// Rows 0..L_b of each request, host (mapped, src_dev its device address) ->
// device, L_b from the device word array sched_len; bytes (optional) += count.
cudaError_t launch_fetch_rows(void* dst, const void* src_dev, int32_t B, int32_t K, size_t row_bytes,
                              const int32_t* sched_len, unsigned long long* bytes, cudaStream_t s);
cudaError_t launch_confidence(const SchedParams& p, cudaStream_t s);
cudaError_t launch_acceptance(const void* target, const void* draft, int32_t rows, int32_t V, int32_t dtype,
                              const float* temperature, float* alpha, int32_t* status, cudaStream_t s);
cudaError_t launch_schedule(const SchedParams& p, cudaStream_t s);
cudaError_t launch_sts_fit(const StsParams& p, cudaStream_t s);
size_t schedule_smem_bytes(int32_t B, int32_t K);
cudaError_t launch_transpose(const void* P, int32_t r, int32_t V, int32_t dtype, void* P_t,
                             cudaStream_t s);
size_t packed_projection_bytes(int32_t r, int32_t V);
cudaError_t launch_pack_projection(const void* P, int32_t r, int32_t V, void* P_packed, cudaStream_t s);
cudaError_t launch_philox_fill(const uint32_t* ctr, uint32_t k0, uint32_t k1, uint32_t* out,
                               int32_t n, cudaStream_t s);

}  // namespace ds
