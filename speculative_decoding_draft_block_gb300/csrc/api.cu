// C-ABI layer: argument validation, workspace layout and kernel launches.
// Declarations and the contract of every entry point are in include/ds_draft.h.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "../../include/ds_draft.h"
#include "internal.h"
#include "philox.h"

using namespace ds;

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return p != nullptr && ((uintptr_t)p & 15u) == 0; }

// The kernels are built for sm_103a only; refuse other devices up front.
ds_status device_supported() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DS_ERR_CUDA;
  static std::mutex mu;
  static int cached[64];
  static bool init = false;
  std::lock_guard<std::mutex> lock(mu);
  if (!init) {
    for (int i = 0; i < 64; ++i) cached[i] = -1;
    init = true;
  }
  if (dev < 0 || dev >= 64) return DS_ERR_UNSUPPORTED;
  if (cached[dev] < 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return DS_ERR_CUDA;
    cached[dev] = (major == 10 && minor == 3) ? 1 : 0;
  }
  return cached[dev] ? DS_OK : DS_ERR_UNSUPPORTED;
}

bool shape_ok(int32_t B, int32_t K, int32_t V, int32_t r) {
  if (B < 1 || K < 1 || K > 64 || V < 8 || (V % 8) != 0) return false;
  if (r < 16 || r > 1024 || (r % 16) != 0) return false;
  if ((int64_t)B * K > 16384) return false;
  return true;
}

ds_status from_cuda(cudaError_t e) { return e == cudaSuccess ? DS_OK : DS_ERR_CUDA; }

// Draft workspace: two sets of chunk and group records, used by alternating
// steps so that a step's records are never overwritten while the previous
// locate still reads them.
struct DraftLayout {
  size_t rec[2], sup[2], astage, total;
};

DraftLayout draft_layout(int32_t B, int32_t V, int32_t r) {
  DraftLayout l;
  const size_t rec = align_up((size_t)B * num_chunks(V) * sizeof(ChunkRec));
  const size_t sup = align_up((size_t)B * sup_stride_for(V) * sizeof(ChunkRec));
  l.rec[0] = 0;
  l.rec[1] = rec;
  l.sup[0] = 2 * rec;
  l.sup[1] = 2 * rec + sup;
  l.astage = 2 * rec + 2 * sup;
  const size_t esz = 4;  // room for f32 E rows; bf16 uses half
  l.total = l.astage + align_up((size_t)B * r * esz);
  return l;
}

size_t draft_ws(int32_t B, int32_t V, int32_t r) { return draft_layout(B, V, r).total; }

// RNN head workspace, after the draft workspace: the hidden-state part of the
// gate inputs for every position (f32 [K][3r][B]) and two input-row buffers
// [e ; s] (bf16 [2][B][2r]), alternating by position parity.
struct RnnLayout {
  size_t gh, gru_in, total;
};

// The RNN head runs the tensor-core tile kernel, whose A operand (128 rows of
// r bf16) is one 64 KB shared-memory block: 64 <= r <= 256, r % 64 == 0.
bool rnn_shape_ok(int32_t B, int32_t K, int32_t r) {
  return B >= 1 && K >= 1 && K <= 64 && (int64_t)B * K <= 16384 && r >= 64 && r <= 256 && r % 64 == 0;
}

RnnLayout rnn_layout(int32_t B, int32_t K, int32_t r) {
  RnnLayout l;
  l.gh = 0;
  l.gru_in = align_up(sizeof(float) * (size_t)B * K * 3 * r);
  l.total = l.gru_in + align_up(sizeof(__nv_bfloat16) * 2 * (size_t)B * 2 * r);
  return l;
}

struct VerifyLayout {
  size_t queue, vrows, desc, chunks, supers, total;
};

VerifyLayout verify_layout(int32_t B, int32_t K, int32_t V, int32_t r) {
  VerifyLayout l;
  l.queue = 0;  // first_reject[B]
  l.vrows = l.queue + align_up((size_t)B * sizeof(uint32_t));
  l.desc = l.vrows + align_up((size_t)B * (K + 1) * sizeof(VRow));
  l.chunks = l.desc + align_up((size_t)B * sizeof(FinalDesc));
  (void)r;
  l.supers = l.chunks + align_up((size_t)B * num_chunks(V) * sizeof(ChunkRec));
  l.total = l.supers + align_up((size_t)B * sup_stride_for(V) * sizeof(ChunkRec));
  return l;
}

// STS fit workspace: ticket, prefix buffers, fixed-point histogram, ECE curve.
struct StsLayout {
  size_t ticket, base, lab, hist64, ece_all, total;
};

bool sts_shape_ok(int32_t N, int32_t K, int32_t G, int32_t n_bins) {
  return N >= 1 && N <= (1 << 26) && K >= 1 && K <= 64 && G >= 1 && G <= 4096 && n_bins >= 1 &&
         n_bins <= 64;
}

StsLayout sts_layout(int32_t N, int32_t G, int32_t n_bins) {
  StsLayout L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += (bytes + 255) & ~size_t(255);
    return at;
  };
  L.ticket = take(sizeof(unsigned));
  L.base = take(sizeof(float) * 2 * (size_t)N);
  L.lab = take(sizeof(float) * 2 * (size_t)N);
  L.hist64 = take(sizeof(long long) * (size_t)n_bins * G);
  L.ece_all = take(sizeof(float) * (size_t)G);
  L.total = off;
  return L;
}

// The RNN head's draft loop. Per call: the hidden-state part of the gate
// inputs for all positions, the first input rows [E[anchor] ; 0] and the
// first state; per position p: tile and locate with the state s_p as A rows
// (the locate stages E[x_p] into the input rows), then the update to s_{p+1}.
ds_status draft_rnn(const ds_draft_args* a, SampleParams& p, char* rw, char* ws, const DraftLayout& l,
                    cudaStream_t s) {
  const int32_t B = a->B, K = a->K, r = a->r;
  const RnnLayout rl = rnn_layout(B, K, r);
  float* gh = reinterpret_cast<float*>(rw + rl.gh);
  __nv_bfloat16* in[2];
  in[0] = reinterpret_cast<__nv_bfloat16*>(rw + rl.gru_in);
  in[1] = in[0] + (size_t)B * 2 * r;
  const __nv_bfloat16* w_ih = reinterpret_cast<const __nv_bfloat16*>(a->rnn_w_ih);

  GemmParams g;
  memset(&g, 0, sizeof(g));
  g.B = B;
  g.K = K;
  g.N = 3 * r;
  g.Kd = a->d;
  g.bias = a->rnn_b_ih;
  g.out = gh;
  g.status = a->status;
  if (launch_rnn_gemm(g, kGemmBias, a->h, w_ih + r, (int64_t)r + a->d, s) != cudaSuccess)
    return DS_ERR_CUDA;
  if (launch_rnn_init(a->E, a->anchor, B, r, a->V, in[0], a->status, s) != cudaSuccess)
    return DS_ERR_CUDA;

  GemmParams u;
  memset(&u, 0, sizeof(u));
  u.B = B;
  u.K = K;
  u.N = 4 * r;
  u.Kd = 2 * r;
  u.gh = gh;
  u.b_hh = a->rnn_b_hh;
  u.states = reinterpret_cast<__nv_bfloat16*>(a->states);
  u.r = r;
  u.status = a->status;
  auto update = [&](int pos) {  // s_pos from the input rows of position pos - 1
    u.p = pos;
    u.s_prev = in[(pos - 1) & 1] + r;
    u.s_next = in[pos & 1] + r;
    return launch_rnn_gemm(u, kGemmGru, in[(pos - 1) & 1], a->rnn_w_step, 2 * r, s);
  };
  if (update(1) != cudaSuccess) return DS_ERR_CUDA;
  p.a_stage_stride = 2 * r;
  p.a_rows_stride = 2 * r;
  for (int k = 1; k <= K; ++k) {
    p.step = k;
    p.chunks = reinterpret_cast<ChunkRec*>(ws + l.rec[k & 1]);
    p.supers = reinterpret_cast<ChunkRec*>(ws + l.sup[k & 1]);
    p.a_stage_in = in[k & 1] + r;
    p.a_rows = in[k & 1] + r;
    p.a_stage_out = (k < K) ? in[k & 1] : nullptr;
    if (launch_tile_tc(p, s) != cudaSuccess) return DS_ERR_CUDA;
    if (launch_sample_locate(p, s) != cudaSuccess) return DS_ERR_CUDA;
    if (k < K && update(k + 1) != cudaSuccess) return DS_ERR_CUDA;
  }
  return DS_OK;
}

}  // namespace

extern "C" {

void ds_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  const Philox4 r = philox4x32_10(ctr[0], ctr[1], ctr[2], ctr[3], key[0], key[1]);
  memcpy(out, r.v, sizeof(r.v));
}

double ds_uniform(uint64_t seed, uint32_t request, uint32_t position, uint32_t stage) {
  return uniform_from_word(philox_word(seed, request, position, stage));
}

ds_status ds_philox_fill(const uint32_t* ctr, uint32_t key0, uint32_t key1, uint32_t* out,
                         int32_t n, ds_stream_t stream) {
  if (n < 0 || (n > 0 && (!aligned16(ctr) || !aligned16(out)))) return DS_ERR_INVALID_ARG;
  if (n == 0) return DS_OK;
  const ds_status st = device_supported();
  if (st != DS_OK) return st;
  return from_cuda(launch_philox_fill(ctr, key0, key1, out, n, (cudaStream_t)stream));
}

size_t ds_packed_projection_bytes(int32_t r, int32_t V) {
  if (!shape_ok(1, 1, V, r) || !tc_path_supported(DS_BF16, r, V)) return 0;
  return packed_projection_bytes(r, V);
}

ds_status ds_pack_projection(const void* P, int32_t r, int32_t V, int32_t dtype, void* P_packed,
                             size_t packed_bytes, ds_stream_t stream) {
  if (!shape_ok(1, 1, V, r)) return DS_ERR_INVALID_ARG;
  if (dtype != DS_BF16 || !tc_path_supported(dtype, r, V)) return DS_ERR_UNSUPPORTED;
  if (P == nullptr || P_packed == nullptr || !aligned16(P) || !aligned16(P_packed)) return DS_ERR_INVALID_ARG;
  const size_t need = packed_projection_bytes(r, V);
  if (packed_bytes < need) return DS_ERR_WORKSPACE;
  const char* a = static_cast<const char*>(P);
  const char* b = static_cast<const char*>(P_packed);
  if (a < b + need && b < a + (size_t)r * V * 2) return DS_ERR_INVALID_ARG;  // overlapping
  const ds_status st = device_supported();
  if (st != DS_OK) return st;
  return from_cuda(launch_pack_projection(P, r, V, P_packed, (cudaStream_t)stream));
}

ds_status ds_transpose_projection(const void* P, int32_t r, int32_t V, int32_t dtype, void* P_t,
                                  ds_stream_t stream) {
  if (!shape_ok(1, 1, V, r)) return DS_ERR_INVALID_ARG;
  if (dtype != DS_F32 && dtype != DS_BF16) return DS_ERR_INVALID_ARG;
  if (P == nullptr || P_t == nullptr || !aligned16(P) || !aligned16(P_t)) return DS_ERR_INVALID_ARG;
  const size_t bytes = (size_t)r * V * (dtype == DS_BF16 ? 2 : 4);
  const char* a = static_cast<const char*>(P);
  const char* b = static_cast<const char*>(P_t);
  if (a < b + bytes && b < a + bytes) return DS_ERR_INVALID_ARG;  // overlapping
  const ds_status st = device_supported();
  if (st != DS_OK) return st;
  return from_cuda(launch_transpose(P, r, V, dtype, P_t, (cudaStream_t)stream));
}

size_t ds_draft_workspace_bytes(int32_t B, int32_t K, int32_t V, int32_t r) {
  if (!shape_ok(B, K, V, r)) return 0;
  return draft_ws(B, V, r);
}

ds_status ds_draft_block(const ds_draft_args* a, ds_stream_t stream) {
  if (a == nullptr) return DS_ERR_INVALID_ARG;
  if (!shape_ok(a->B, a->K, a->V, a->r)) return DS_ERR_INVALID_ARG;
  if (a->dtype != DS_F32 && a->dtype != DS_BF16) return DS_ERR_INVALID_ARG;
  const void* ptrs[] = {a->base_logits, a->E, a->P, a->anchor, a->temperature,
                        a->draft_tokens, a->q_token, a->q_stats, a->status};
  for (const void* p : ptrs)
    if (!aligned16(p)) return DS_ERR_INVALID_ARG;
  if (a->P_t != nullptr && !aligned16(a->P_t)) return DS_ERR_INVALID_ARG;
  if (a->P_packed != nullptr && !aligned16(a->P_packed)) return DS_ERR_INVALID_ARG;
  if (a->seed_ptr != nullptr && ((uintptr_t)a->seed_ptr & 7u) != 0) return DS_ERR_INVALID_ARG;
  const bool rnn = a->head == DS_HEAD_RNN;
  if (a->head != DS_HEAD_MARKOV && !rnn) return DS_ERR_INVALID_ARG;
  size_t need = draft_ws(a->B, a->V, a->r);
  const size_t rnn_off = align_up(need);
  if (rnn) {
    if (a->dtype != DS_BF16 || !rnn_shape_ok(a->B, a->K, a->r)) return DS_ERR_UNSUPPORTED;
    if (a->d < 64 || a->d % 64 != 0) return DS_ERR_INVALID_ARG;
    const void* rp[] = {a->h, a->rnn_w_ih, a->rnn_w_step, a->rnn_b_ih, a->rnn_b_hh, a->states};
    for (const void* q : rp)
      if (!aligned16(q)) return DS_ERR_INVALID_ARG;
    need = rnn_off + rnn_layout(a->B, a->K, a->r).total;
  }
  if (a->workspace == nullptr || !aligned16(a->workspace) || a->workspace_bytes < need)
    return DS_ERR_WORKSPACE;
  const ds_status st = device_supported();
  if (st != DS_OK) return st;

  SampleParams p;
  memset(&p, 0, sizeof(p));
  p.B = a->B;
  p.K = a->K;
  p.V = a->V;
  p.r = a->r;
  p.n_chunks = num_chunks(a->V);
  p.src = 0;
  p.dtype = a->dtype;
  p.base_logits = a->base_logits;
  p.E = a->E;
  p.P = a->P;
  p.P_t = a->P_t;
  p.P_packed = a->P_packed;
  p.anchor = a->anchor;
  p.draft_tokens = a->draft_tokens;
  p.temperature = a->temperature;
  const DraftLayout l = draft_layout(a->B, a->V, a->r);
  char* ws = reinterpret_cast<char*>(a->workspace);
  const bool tc = tc_path_supported(a->dtype, a->r, a->V);
  p.seed = a->seed;
  p.seed_ptr = a->seed_ptr;
  p.tokens_out = a->draft_tokens;
  p.q_token = a->q_token;
  p.q_stats = a->q_stats;
  p.status = a->status;
  if (tc)
    tc_group_layout(p);
  else
    simt_group_layout(p);
  const cudaStream_t s = (cudaStream_t)stream;
  p.a_stage_stride = a->r;
  if (rnn) return draft_rnn(a, p, ws + rnn_off, ws, l, s);
  for (int k = 1; k <= a->K; ++k) {
    p.step = k;
    p.chunks = reinterpret_cast<ChunkRec*>(ws + l.rec[k & 1]);
    p.supers = reinterpret_cast<ChunkRec*>(ws + l.sup[k & 1]);
    p.a_stage_in = (tc && k > 1) ? ws + l.astage : nullptr;
    p.a_stage_out = (tc && k < a->K) ? ws + l.astage : nullptr;
    cudaError_t e = tc ? launch_tile_tc(p, s) : launch_sample_tile(p, s);
    if (e != cudaSuccess) return DS_ERR_CUDA;
    e = launch_sample_locate(p, s);
    if (e != cudaSuccess) return DS_ERR_CUDA;
  }
  return DS_OK;
}

size_t ds_rnn_workspace_bytes(int32_t B, int32_t K, int32_t r) {
  if (!rnn_shape_ok(B, K, r)) return 0;
  return rnn_layout(B, K, r).total;
}

ds_status ds_rnn_pack_weights(const void* W_ih, const void* W_hh, int32_t r, int32_t d, int32_t dtype,
                              void* W_step, ds_stream_t stream) {
  if (dtype != DS_BF16) return DS_ERR_UNSUPPORTED;
  if (r < 64 || r > 1024 || r % 64 != 0 || d < 64 || d % 64 != 0) return DS_ERR_INVALID_ARG;
  if (!aligned16(W_ih) || !aligned16(W_hh) || !aligned16(W_step)) return DS_ERR_INVALID_ARG;
  const ds_status st = device_supported();
  if (st != DS_OK) return st;
  return from_cuda(launch_rnn_pack(W_ih, W_hh, r, d, W_step, (cudaStream_t)stream));
}

size_t ds_sched_workspace_bytes(int32_t B, int32_t K) {
  (void)B;
  (void)K;
  return 0;
}

ds_status ds_confidence_schedule(const ds_sched_args* a, ds_stream_t stream) {
  if (a == nullptr) return DS_ERR_INVALID_ARG;
  if (a->B < 1 || a->K < 1 || a->K > 64 || (int64_t)a->B * a->K > 16384) return DS_ERR_INVALID_ARG;
  if (a->d < 8 || (a->d % 8) != 0 || a->r < 16 || (a->r % 16) != 0 || a->r > 1024 || a->V < 8 ||
      (a->V % 8) != 0)
    return DS_ERR_INVALID_ARG;
  if (a->dtype != DS_F32 && a->dtype != DS_BF16) return DS_ERR_INVALID_ARG;
  if (a->n_max < 1) return DS_ERR_INVALID_ARG;
  if (a->mode != DS_SCHED_GREEDY_EARLYSTOP && a->mode != DS_SCHED_FIXED_K &&
      a->mode != DS_SCHED_THRESHOLD && a->mode != DS_SCHED_ASYNC)
    return DS_ERR_INVALID_ARG;
  if (a->mode == DS_SCHED_ASYNC && !aligned16(a->budget_ring))
    return DS_ERR_INVALID_ARG;
  const void* ptrs[] = {a->h, a->E, a->anchor, a->draft_tokens, a->w_h, a->w_e, a->sts_temp,
                        a->sps, a->conf, a->survival, a->sched_len, a->objective, a->status};
  for (const void* p : ptrs)
    if (!aligned16(p)) return DS_ERR_INVALID_ARG;
  if (a->conf_logit != nullptr && !aligned16(a->conf_logit)) return DS_ERR_INVALID_ARG;
  const ds_status st = device_supported();
  if (st != DS_OK) return st;
  SchedParams p;
  memset(&p, 0, sizeof(p));
  p.B = a->B;
  p.K = a->K;
  p.d = a->d;
  p.r = a->r;
  p.V = a->V;
  p.dtype = a->dtype;
  p.n_max = a->n_max;
  p.mode = a->mode;
  p.bias = a->bias;
  p.threshold = a->threshold;
  p.budget_ring = a->budget_ring;
  p.h = a->h;
  p.E = a->E;
  p.anchor = a->anchor;
  p.draft_tokens = a->draft_tokens;
  p.w_h = a->w_h;
  p.w_e = a->w_e;
  p.sts_temp = a->sts_temp;
  p.sps = a->sps;
  p.conf = a->conf;
  p.conf_logit = a->conf_logit;
  p.survival = a->survival;
  p.sched_len = a->sched_len;
  p.objective = a->objective;
  p.status = a->status;
  const cudaStream_t s = (cudaStream_t)stream;
  if (launch_confidence(p, s) != cudaSuccess) return DS_ERR_CUDA;
  if (launch_schedule(p, s) != cudaSuccess) return DS_ERR_CUDA;
  return DS_OK;
}

size_t ds_sts_workspace_bytes(int32_t N, int32_t K, int32_t n_grid, int32_t n_bins) {
  if (!sts_shape_ok(N, K, n_grid, n_bins)) return 0;
  return sts_layout(N, n_grid, n_bins).total;
}

ds_status ds_sts_fit(const ds_sts_args* a, ds_stream_t stream) {
  if (a == nullptr) return DS_ERR_INVALID_ARG;
  if (!sts_shape_ok(a->N, a->K, a->n_grid, a->n_bins)) return DS_ERR_INVALID_ARG;
  const void* ptrs[] = {a->logits, a->labels, a->grid, a->sts_temp, a->grid_index, a->ece,
                        a->status};
  for (const void* p : ptrs)
    if (!aligned16(p)) return DS_ERR_INVALID_ARG;
  if (a->ece_curve != nullptr && !aligned16(a->ece_curve)) return DS_ERR_INVALID_ARG;
  const StsLayout L = sts_layout(a->N, a->n_grid, a->n_bins);
  if (a->workspace == nullptr || !aligned16(a->workspace) || a->workspace_bytes < L.total)
    return DS_ERR_WORKSPACE;
  const ds_status st = device_supported();
  if (st != DS_OK) return st;
  char* ws = static_cast<char*>(a->workspace);
  StsParams p;
  memset(&p, 0, sizeof(p));
  p.N = a->N;
  p.K = a->K;
  p.G = a->n_grid;
  p.n_bins = a->n_bins;
  p.logits = a->logits;
  p.labels = a->labels;
  p.grid = a->grid;
  p.sts_temp = a->sts_temp;
  p.grid_index = a->grid_index;
  p.ece = a->ece;
  p.ece_curve = a->ece_curve;
  p.ticket = reinterpret_cast<unsigned*>(ws + L.ticket);
  p.base = reinterpret_cast<float*>(ws + L.base);
  p.lab = reinterpret_cast<float*>(ws + L.lab);
  p.hist64 = reinterpret_cast<long long*>(ws + L.hist64);
  p.ece_all = reinterpret_cast<float*>(ws + L.ece_all);
  p.status = a->status;
  if (launch_sts_fit(p, (cudaStream_t)stream) != cudaSuccess) return DS_ERR_CUDA;
  return DS_OK;
}

size_t ds_verify_workspace_bytes(int32_t B, int32_t K, int32_t V, int32_t r) {
  if (!shape_ok(B, K, V, r)) return 0;
  return verify_layout(B, K, V, r).total;
}

ds_status ds_verify(const ds_verify_args* a, ds_stream_t stream) {
  if (a == nullptr) return DS_ERR_INVALID_ARG;
  if (!shape_ok(a->B, a->K, a->V, a->r)) return DS_ERR_INVALID_ARG;
  if (a->dtype != DS_F32 && a->dtype != DS_BF16) return DS_ERR_INVALID_ARG;
  const void* ptrs[] = {a->target_logits, a->base_logits, a->E, a->P, a->anchor,
                        a->draft_tokens, a->q_token, a->q_stats, a->sched_len,
                        a->temperature, a->out_tokens, a->accept_count, a->num_emitted,
                        a->status};
  for (const void* p : ptrs)
    if (!aligned16(p)) return DS_ERR_INVALID_ARG;
  if (a->P_t != nullptr && !aligned16(a->P_t)) return DS_ERR_INVALID_ARG;
  if (a->P_packed != nullptr && !aligned16(a->P_packed)) return DS_ERR_INVALID_ARG;
  const VerifyLayout l = verify_layout(a->B, a->K, a->V, a->r);
  const bool tc = tc_path_supported(a->dtype, a->r, a->V);
  if (a->workspace == nullptr || !aligned16(a->workspace) || a->workspace_bytes < l.total)
    return DS_ERR_WORKSPACE;
  if (a->states != nullptr &&
      (!aligned16(a->states) || !tc_path_supported(a->dtype, a->r, a->V) || a->dtype != DS_BF16))
    return DS_ERR_INVALID_ARG;
  if (a->seed_ptr != nullptr && ((uintptr_t)a->seed_ptr & 7u) != 0) return DS_ERR_INVALID_ARG;
  if (a->p_token != nullptr && !aligned16(a->p_token)) return DS_ERR_INVALID_ARG;
  const ds_status st = device_supported();
  if (st != DS_OK) return st;
  char* ws = reinterpret_cast<char*>(a->workspace);
  VerifyParams v;
  memset(&v, 0, sizeof(v));
  v.B = a->B;
  v.K = a->K;
  v.V = a->V;
  v.r = a->r;
  v.n_chunks = num_chunks(a->V);
  v.dtype = a->dtype;
  v.target_logits = a->target_logits;
  v.anchor = a->anchor;
  v.draft_tokens = a->draft_tokens;
  v.q_token = a->q_token;
  v.q_stats = a->q_stats;
  v.sched_len = a->sched_len;
  v.temperature = a->temperature;
  v.seed = a->seed;
  v.seed_ptr = a->seed_ptr;
  v.vrows = reinterpret_cast<VRow*>(ws + l.vrows);
  v.final_desc = reinterpret_cast<FinalDesc*>(ws + l.desc);
  v.out_tokens = a->out_tokens;
  v.accept_count = a->accept_count;
  v.num_emitted = a->num_emitted;
  v.p_token = a->p_token;
  v.first_reject = reinterpret_cast<uint32_t*>(ws + l.queue);
  v.status = a->status;
  const cudaStream_t s = (cudaStream_t)stream;
  // no rejection recorded yet: first-rejection words all ones
  if (cudaMemsetAsync(ws + l.queue, 0xff, (size_t)a->B * sizeof(uint32_t), s) != cudaSuccess)
    return DS_ERR_CUDA;
  if (launch_verify_rows(v, s) != cudaSuccess) return DS_ERR_CUDA;
  if (launch_verify_finalize(v, s) != cudaSuccess) return DS_ERR_CUDA;

  SampleParams p;
  memset(&p, 0, sizeof(p));
  p.B = a->B;
  p.K = a->K;
  p.V = a->V;
  p.r = a->r;
  p.n_chunks = v.n_chunks;
  p.src = 1;
  p.dtype = a->dtype;
  p.base_logits = a->base_logits;
  p.target_logits = a->target_logits;
  p.E = a->E;
  p.P = a->P;
  p.P_t = a->P_t;
  p.P_packed = a->P_packed;
  p.anchor = a->anchor;
  p.draft_tokens = a->draft_tokens;
  p.temperature = a->temperature;
  p.final_desc = v.final_desc;
  p.a_stage_stride = a->r;
  if (a->states != nullptr) {  // RNN head: the residual's bias row is the draft's state
    p.a_rows = a->states;
    p.a_rows_stride = a->K * a->r;
  }
  p.chunks = reinterpret_cast<ChunkRec*>(ws + l.chunks);
  p.supers = reinterpret_cast<ChunkRec*>(ws + l.supers);
  if (tc)
    tc_group_layout(p);
  else
    simt_group_layout(p);
  p.seed = a->seed;
  p.seed_ptr = a->seed_ptr;
  p.tokens_out = a->out_tokens;
  p.status = a->status;
  if ((tc ? launch_tile_tc(p, s) : launch_sample_tile(p, s)) != cudaSuccess)
    return DS_ERR_CUDA;
  if (launch_sample_locate(p, s) != cudaSuccess) return DS_ERR_CUDA;
  return DS_OK;
}

ds_status ds_copy_scheduled_rows(void* dst, const void* src, int32_t B, int32_t K, size_t row_bytes,
                                 const int32_t* lens, uint64_t* bytes_out, ds_stream_t stream) {
  if (dst == nullptr || src == nullptr || lens == nullptr || B < 1 || K < 0 || row_bytes == 0)
    return DS_ERR_INVALID_ARG;
  const size_t req_bytes = (size_t)(K + 1) * row_bytes;
  uint64_t total = 0;
  for (int32_t b = 0; b < B; ++b) {
    const int32_t L = lens[b] < 0 ? 0 : (lens[b] > K ? K : lens[b]);
    const size_t n = (size_t)(L + 1) * row_bytes;
    const size_t off = (size_t)b * req_bytes;
    if (cudaMemcpyAsync(static_cast<char*>(dst) + off, static_cast<const char*>(src) + off, n,
                        cudaMemcpyHostToDevice, (cudaStream_t)stream) != cudaSuccess) {
      if (bytes_out) *bytes_out = total;
      return DS_ERR_CUDA;
    }
    total += n;
  }
  if (bytes_out) *bytes_out = total;
  return DS_OK;
}

ds_status ds_fetch_scheduled_rows(void* dst, const void* src, int32_t B, int32_t K, size_t row_bytes,
                                  const int32_t* sched_len, uint64_t* bytes_total, ds_stream_t stream) {
  if (dst == nullptr || src == nullptr || sched_len == nullptr || B < 1 || K < 0 || row_bytes == 0 ||
      row_bytes % 16 != 0 || !aligned16(dst) || !aligned16(src) || ((uintptr_t)sched_len & 3u) != 0 ||
      ((uintptr_t)bytes_total & 7u) != 0)
    return DS_ERR_INVALID_ARG;
  const ds_status st = device_supported();
  if (st != DS_OK) return st;
  void* src_dev = nullptr;
  if (cudaHostGetDevicePointer(&src_dev, const_cast<void*>(src), 0) != cudaSuccess) {
    (void)cudaGetLastError();  // not mapped host memory: clear the error, launch nothing
    return DS_ERR_INVALID_ARG;
  }
  if (!aligned16(src_dev)) return DS_ERR_INVALID_ARG;
  return from_cuda(launch_fetch_rows(dst, src_dev, B, K, row_bytes, sched_len,
                                     reinterpret_cast<unsigned long long*>(bytes_total),
                                     (cudaStream_t)stream));
}

ds_status ds_acceptance_rate(const void* target_logits, const void* draft_logits, int32_t rows, int32_t V,
                             int32_t dtype, const float* temperature, float* alpha, int32_t* status,
                             ds_stream_t stream) {
  if (rows < 1 || V < 8 || V % 8 != 0) return DS_ERR_INVALID_ARG;
  if (dtype != DS_F32 && dtype != DS_BF16) return DS_ERR_INVALID_ARG;
  const void* ptrs[] = {target_logits, draft_logits, temperature, alpha, status};
  for (const void* q : ptrs)
    if (!aligned16(q)) return DS_ERR_INVALID_ARG;
  const ds_status st = device_supported();
  if (st != DS_OK) return st;
  return from_cuda(launch_acceptance(target_logits, draft_logits, rows, V, dtype, temperature, alpha, status,
                                     (cudaStream_t)stream));
}

size_t ds_reserve_persisting_l2(size_t bytes) {
  int dev = 0, maxp = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&maxp, cudaDevAttrMaxPersistingL2CacheSize, dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  const size_t b = bytes < (size_t)(maxp > 0 ? maxp : 0) ? bytes : (size_t)(maxp > 0 ? maxp : 0);
  if (cudaDeviceSetLimit(cudaLimitPersistingL2CacheSize, b) != cudaSuccess) (void)cudaGetLastError();
  size_t cur = 0;
  if (cudaDeviceGetLimit(&cur, cudaLimitPersistingL2CacheSize) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return cur;
}

ds_status ds_test_set_wait_hooks(uint32_t wait_polls, int32_t withhold_cta) {
  set_tile_test_hooks(wait_polls, withhold_cta);
  return DS_OK;
}

ds_status ds_check_status(const int32_t* device_status, ds_stream_t stream) {
  if (device_status == nullptr) return DS_ERR_INVALID_ARG;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return DS_ERR_CUDA;
  int32_t h = 0;
  if (cudaMemcpy(&h, device_status, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess)
    return DS_ERR_CUDA;
  return (ds_status)h;
}

const char* ds_status_string(ds_status s) {
  switch (s) {
    case DS_OK: return "ok";
    case DS_ERR_INVALID_ARG: return "invalid argument";
    case DS_ERR_UNSUPPORTED: return "unsupported device or dtype";
    case DS_ERR_WORKSPACE: return "workspace missing or too small";
    case DS_ERR_CUDA: return "CUDA runtime error";
    case DS_ERR_TIMEOUT: return "device wait timed out";
    case DS_ERR_BOUNDS: return "token id out of range";
    case DS_ERR_NONFINITE: return "non-finite logit or empty distribution";
  }
  return "unknown status";
}

const char* ds_version(void) { return "0.1.0"; }

}  // extern "C"
