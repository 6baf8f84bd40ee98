"""ctypes binding of libdsdraft.so (argument marshalling only).

Every function keeps the C name and forwards device pointers, sizes and the
current CUDA stream; all computation happens in the library's kernels. PyTorch
tensors are used only as device memory. If the shared library is missing, every
call raises: there is no fallback path.
"""

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsdraft.so")

DS_OK = 0
DS_F32, DS_BF16 = 0, 1
DS_STAGE_DRAFT, DS_STAGE_ACCEPT, DS_STAGE_RESAMPLE = 0, 1, 2
DS_SCHED_GREEDY_EARLYSTOP, DS_SCHED_FIXED_K, DS_SCHED_THRESHOLD, DS_SCHED_ASYNC = 0, 1, 2, 3
DS_HEAD_MARKOV, DS_HEAD_RNN = 0, 1
STATUS_NAMES = {0: "DS_OK", 1: "DS_ERR_INVALID_ARG", 2: "DS_ERR_UNSUPPORTED", 3: "DS_ERR_WORKSPACE",
                4: "DS_ERR_CUDA", 5: "DS_ERR_TIMEOUT", 6: "DS_ERR_BOUNDS", 7: "DS_ERR_NONFINITE"}

# Every symbol include/ds_draft.h declares.
EXPORTS = ("ds_philox4x32_10", "ds_uniform", "ds_philox_fill", "ds_draft_workspace_bytes",
           "ds_draft_block", "ds_sched_workspace_bytes", "ds_confidence_schedule",
           "ds_verify_workspace_bytes", "ds_verify", "ds_check_status", "ds_status_string",
           "ds_version", "ds_transpose_projection", "ds_verify_static", "ds_sts_workspace_bytes",
           "ds_sts_fit", "ds_rnn_workspace_bytes", "ds_rnn_pack_weights", "ds_copy_scheduled_rows",
           "ds_fetch_scheduled_rows", "ds_test_set_wait_hooks", "ds_reserve_persisting_l2",
           "ds_acceptance_rate", "ds_packed_projection_bytes", "ds_pack_projection")

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32


class DraftArgs(ctypes.Structure):
    _fields_ = [("B", _i32), ("K", _i32), ("V", _i32), ("r", _i32), ("dtype", _i32),
                ("base_logits", _vp), ("E", _vp), ("P", _vp), ("P_t", _vp), ("anchor", _vp),
                ("temperature", _vp), ("seed", ctypes.c_uint64), ("draft_tokens", _vp),
                ("q_token", _vp), ("q_stats", _vp), ("workspace", _vp),
                ("workspace_bytes", ctypes.c_size_t), ("status", _vp),
                ("head", _i32), ("d", _i32), ("h", _vp), ("rnn_w_ih", _vp), ("rnn_w_step", _vp),
                ("rnn_b_ih", _vp), ("rnn_b_hh", _vp), ("states", _vp), ("seed_ptr", _vp),
                ("P_packed", _vp)]


class SchedArgs(ctypes.Structure):
    _fields_ = [("B", _i32), ("K", _i32), ("d", _i32), ("r", _i32), ("V", _i32), ("dtype", _i32),
                ("h", _vp), ("E", _vp), ("anchor", _vp), ("draft_tokens", _vp), ("w_h", _vp),
                ("w_e", _vp), ("bias", ctypes.c_float), ("sts_temp", _vp), ("sps", _vp),
                ("n_max", _i32), ("mode", _i32), ("threshold", ctypes.c_float),
                ("budget_ring", _vp),
                ("conf", _vp), ("conf_logit", _vp), ("survival", _vp), ("sched_len", _vp),
                ("objective", _vp),
                ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t), ("status", _vp)]


class StsArgs(ctypes.Structure):
    _fields_ = [("N", _i32), ("K", _i32), ("n_grid", _i32), ("n_bins", _i32),
                ("logits", _vp), ("labels", _vp), ("grid", _vp), ("sts_temp", _vp),
                ("grid_index", _vp), ("ece", _vp), ("ece_curve", _vp),
                ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t), ("status", _vp)]


class VerifyArgs(ctypes.Structure):
    _fields_ = [("B", _i32), ("K", _i32), ("V", _i32), ("r", _i32), ("dtype", _i32),
                ("target_logits", _vp), ("base_logits", _vp), ("E", _vp), ("P", _vp), ("P_t", _vp),
                ("anchor", _vp), ("draft_tokens", _vp), ("q_token", _vp), ("q_stats", _vp),
                ("sched_len", _vp), ("temperature", _vp), ("seed", ctypes.c_uint64),
                ("out_tokens", _vp), ("accept_count", _vp), ("num_emitted", _vp),
                ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t), ("status", _vp),
                ("states", _vp), ("seed_ptr", _vp), ("p_token", _vp), ("P_packed", _vp)]


_lib = None


def load():
    """Load libdsdraft.so (once). Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libdsdraft.so is not built (run `python -m "
                           "speculative_decoding_draft_block_gb300.build`); no fallback exists")
    lib = ctypes.CDLL(LIB_PATH)
    lib.ds_philox4x32_10.argtypes = [ctypes.POINTER(ctypes.c_uint32)] * 3
    lib.ds_philox4x32_10.restype = None
    lib.ds_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32]
    lib.ds_uniform.restype = ctypes.c_double
    lib.ds_philox_fill.argtypes = [_vp, ctypes.c_uint32, ctypes.c_uint32, _vp, _i32, _vp]
    lib.ds_philox_fill.restype = ctypes.c_int
    for f in ("ds_draft_workspace_bytes", "ds_verify_workspace_bytes"):
        getattr(lib, f).argtypes = [_i32] * 4
        getattr(lib, f).restype = ctypes.c_size_t
    lib.ds_sched_workspace_bytes.argtypes = [_i32] * 2
    lib.ds_sched_workspace_bytes.restype = ctypes.c_size_t
    lib.ds_draft_block.argtypes = [ctypes.POINTER(DraftArgs), _vp]
    lib.ds_confidence_schedule.argtypes = [ctypes.POINTER(SchedArgs), _vp]
    lib.ds_verify.argtypes = [ctypes.POINTER(VerifyArgs), _vp]
    lib.ds_verify_static.argtypes = [ctypes.POINTER(VerifyArgs), _vp]
    lib.ds_verify_static.restype = ctypes.c_int
    for f in ("ds_draft_block", "ds_confidence_schedule", "ds_verify"):
        getattr(lib, f).restype = ctypes.c_int
    lib.ds_rnn_workspace_bytes.argtypes = [_i32] * 3
    lib.ds_rnn_workspace_bytes.restype = ctypes.c_size_t
    lib.ds_rnn_pack_weights.argtypes = [_vp, _vp, _i32, _i32, _i32, _vp, _vp]
    lib.ds_rnn_pack_weights.restype = ctypes.c_int
    lib.ds_sts_workspace_bytes.argtypes = [_i32] * 4
    lib.ds_sts_workspace_bytes.restype = ctypes.c_size_t
    lib.ds_sts_fit.argtypes = [ctypes.POINTER(StsArgs), _vp]
    lib.ds_sts_fit.restype = ctypes.c_int
    lib.ds_transpose_projection.argtypes = [_vp, _i32, _i32, _i32, _vp, _vp]
    lib.ds_transpose_projection.restype = ctypes.c_int
    lib.ds_copy_scheduled_rows.argtypes = [_vp, _vp, _i32, _i32, ctypes.c_size_t, _vp,
                                           ctypes.POINTER(ctypes.c_uint64), _vp]
    lib.ds_copy_scheduled_rows.restype = ctypes.c_int
    lib.ds_fetch_scheduled_rows.argtypes = [_vp, _vp, _i32, _i32, ctypes.c_size_t, _vp, _vp, _vp]
    lib.ds_fetch_scheduled_rows.restype = ctypes.c_int
    lib.ds_packed_projection_bytes.argtypes = [_i32, _i32]
    lib.ds_packed_projection_bytes.restype = ctypes.c_size_t
    lib.ds_pack_projection.argtypes = [_vp, _i32, _i32, _i32, _vp, ctypes.c_size_t, _vp]
    lib.ds_pack_projection.restype = ctypes.c_int
    lib.ds_acceptance_rate.argtypes = [_vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp]
    lib.ds_acceptance_rate.restype = ctypes.c_int
    lib.ds_reserve_persisting_l2.argtypes = [ctypes.c_size_t]
    lib.ds_reserve_persisting_l2.restype = ctypes.c_size_t
    lib.ds_test_set_wait_hooks.argtypes = [ctypes.c_uint32, _i32]
    lib.ds_test_set_wait_hooks.restype = ctypes.c_int
    lib.ds_check_status.argtypes = [_vp, _vp]
    lib.ds_check_status.restype = ctypes.c_int
    lib.ds_status_string.argtypes = [ctypes.c_int]
    lib.ds_status_string.restype = ctypes.c_char_p
    lib.ds_version.argtypes = []
    lib.ds_version.restype = ctypes.c_char_p
    _lib = lib
    return lib


class DsError(RuntimeError):
    def __init__(self, code, what=""):
        super().__init__("%s%s" % (STATUS_NAMES.get(code, str(code)), (": " + what) if what else ""))
        self.code = code


def check(code, what=""):
    if code != DS_OK:
        raise DsError(code, what)
    return code


def _ptr(t, name):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return DS_BF16
    if t.dtype == torch.float32:
        return DS_F32
    raise ValueError("logits/weights must be bfloat16 or float32")


# ---- randomness --------------------------------------------------------------

def ds_philox4x32_10(ctr, key):
    lib = load()
    c = (ctypes.c_uint32 * 4)(*[int(v) & 0xFFFFFFFF for v in ctr])
    k = (ctypes.c_uint32 * 2)(*[int(v) & 0xFFFFFFFF for v in key])
    o = (ctypes.c_uint32 * 4)()
    lib.ds_philox4x32_10(c, k, o)
    return tuple(o)


def ds_uniform(seed, request, position, stage):
    return load().ds_uniform(int(seed), int(request), int(position), int(stage))


def ds_philox_fill(ctr, key0, key1, out, stream=None):
    """ctr, out: int32 CUDA tensors [n, 4] (bit patterns of uint32)."""
    return load().ds_philox_fill(_ptr(ctr, "ctr"), int(key0) & 0xFFFFFFFF, int(key1) & 0xFFFFFFFF,
                                 _ptr(out, "out"), int(ctr.shape[0]), _stream(stream))


# ---- workspace sizes --------------------------------------------------------------

def ds_draft_workspace_bytes(B, K, V, r):
    return load().ds_draft_workspace_bytes(B, K, V, r)


def ds_sched_workspace_bytes(B, K):
    return load().ds_sched_workspace_bytes(B, K)


def ds_verify_workspace_bytes(B, K, V, r):
    return load().ds_verify_workspace_bytes(B, K, V, r)


# ---- the three calls ----------------------------------------------------------

def ds_draft_block(base_logits, E, P, anchor, temperature, seed, draft_tokens, q_token, q_stats,
                   workspace, status, stream=None, P_t=None, rnn=None, seed_ptr=None, P_packed=None):
    """Draft one block. ``rnn`` selects the RNN head: a dict with h [B, K, d],
    w_ih [3r, r + d], w_step (from ds_rnn_pack_weights), b_ih, b_hh (float32
    [3r]) and states (output [B, K, r]); the workspace must then also hold
    ds_rnn_workspace_bytes(B, K, r)."""
    B, K, V = base_logits.shape
    extra = {}
    if rnn is not None:
        extra = dict(head=DS_HEAD_RNN, d=int(rnn["h"].shape[2]), h=_ptr(rnn["h"], "h"),
                     rnn_w_ih=_ptr(rnn["w_ih"], "w_ih"), rnn_w_step=_ptr(rnn["w_step"], "w_step"),
                     rnn_b_ih=_ptr(rnn["b_ih"], "b_ih"), rnn_b_hh=_ptr(rnn["b_hh"], "b_hh"),
                     states=_ptr(rnn["states"], "states"))
    a = DraftArgs(B=B, K=K, V=V, r=E.shape[1], dtype=_dtype_code(base_logits),
                  base_logits=_ptr(base_logits, "base_logits"), E=_ptr(E, "E"), P=_ptr(P, "P"),
                  P_t=None if P_t is None else _ptr(P_t, "P_t"),
                  anchor=_ptr(anchor, "anchor"), temperature=_ptr(temperature, "temperature"),
                  seed=int(seed), draft_tokens=_ptr(draft_tokens, "draft_tokens"),
                  q_token=_ptr(q_token, "q_token"), q_stats=_ptr(q_stats, "q_stats"),
                  workspace=_ptr(workspace, "workspace"),
                  workspace_bytes=workspace.numel() * workspace.element_size(),
                  status=_ptr(status, "status"),
                  seed_ptr=None if seed_ptr is None else _ptr(seed_ptr, "seed_ptr"),
                  P_packed=None if P_packed is None else _ptr(P_packed, "P_packed"), **extra)
    return load().ds_draft_block(ctypes.byref(a), _stream(stream))


def ds_rnn_workspace_bytes(B, K, r):
    return load().ds_rnn_workspace_bytes(B, K, r)


def ds_rnn_pack_weights(w_ih, w_hh, w_step, stream=None):
    """W_step [4r, 2r] from W_ih [3r, r + d] and W_hh [3r, r] (once per model)."""
    r3, rd = w_ih.shape
    r = r3 // 3
    return load().ds_rnn_pack_weights(_ptr(w_ih, "w_ih"), _ptr(w_hh, "w_hh"), r, rd - r,
                                      _dtype_code(w_ih), _ptr(w_step, "w_step"), _stream(stream))


def ds_confidence_schedule(h, E, anchor, draft_tokens, w_h, w_e, bias, sts_temp, sps, mode,
                           conf, survival, sched_len, objective, status, threshold=0.0,
                           workspace=None, stream=None, budget_ring=None, conf_logit=None):
    B, K, d = h.shape
    a = SchedArgs(B=B, K=K, d=d, r=E.shape[1], V=E.shape[0], dtype=_dtype_code(h),
                  h=_ptr(h, "h"), E=_ptr(E, "E"), anchor=_ptr(anchor, "anchor"),
                  draft_tokens=_ptr(draft_tokens, "draft_tokens"), w_h=_ptr(w_h, "w_h"),
                  w_e=_ptr(w_e, "w_e"), bias=float(bias), sts_temp=_ptr(sts_temp, "sts_temp"),
                  sps=_ptr(sps, "sps"), n_max=int(sps.shape[0]), mode=int(mode),
                  threshold=float(threshold),
                  budget_ring=None if budget_ring is None else _ptr(budget_ring, "budget_ring"),
                  conf=_ptr(conf, "conf"),
                  conf_logit=None if conf_logit is None else _ptr(conf_logit, "conf_logit"),
                  survival=_ptr(survival, "survival"), sched_len=_ptr(sched_len, "sched_len"),
                  objective=_ptr(objective, "objective"),
                  workspace=_ptr(workspace, "workspace") if workspace is not None else None,
                  workspace_bytes=0 if workspace is None else workspace.numel() * workspace.element_size(),
                  status=_ptr(status, "status"))
    return load().ds_confidence_schedule(ctypes.byref(a), _stream(stream))


def ds_verify(target_logits, base_logits, E, P, anchor, draft_tokens, q_token, q_stats, sched_len,
              temperature, seed, out_tokens, accept_count, num_emitted, workspace, status,
              stream=None, P_t=None, states=None, seed_ptr=None, p_token=None, P_packed=None):
    B, K1, V = target_logits.shape
    a = VerifyArgs(B=B, K=K1 - 1, V=V, r=E.shape[1], dtype=_dtype_code(target_logits),
                   target_logits=_ptr(target_logits, "target_logits"),
                   base_logits=_ptr(base_logits, "base_logits"), E=_ptr(E, "E"), P=_ptr(P, "P"),
                   P_t=None if P_t is None else _ptr(P_t, "P_t"),
                   anchor=_ptr(anchor, "anchor"), draft_tokens=_ptr(draft_tokens, "draft_tokens"),
                   q_token=_ptr(q_token, "q_token"), q_stats=_ptr(q_stats, "q_stats"),
                   sched_len=_ptr(sched_len, "sched_len"), temperature=_ptr(temperature, "temperature"),
                   seed=int(seed), out_tokens=_ptr(out_tokens, "out_tokens"),
                   accept_count=_ptr(accept_count, "accept_count"),
                   num_emitted=_ptr(num_emitted, "num_emitted"),
                   workspace=_ptr(workspace, "workspace"),
                   workspace_bytes=workspace.numel() * workspace.element_size(),
                   status=_ptr(status, "status"),
                   states=None if states is None else _ptr(states, "states"),
                   seed_ptr=None if seed_ptr is None else _ptr(seed_ptr, "seed_ptr"),
                   p_token=None if p_token is None else _ptr(p_token, "p_token"),
                   P_packed=None if P_packed is None else _ptr(P_packed, "P_packed"))
    return load().ds_verify(ctypes.byref(a), _stream(stream))


def ds_packed_projection_bytes(r, V):
    return int(load().ds_packed_projection_bytes(r, V))


def ds_pack_projection(P, P_packed, stream=None):
    """Tile-packed copy of the bfloat16 projection P [r, V] (once per model; see ds_draft.h)."""
    r, V = P.shape
    return load().ds_pack_projection(_ptr(P, "P"), r, V, _dtype_code(P), _ptr(P_packed, "P_packed"),
                                     P_packed.numel() * P_packed.element_size(), _stream(stream))


def ds_transpose_projection(P, P_t, stream=None):
    """P_t[v, k] = P[k, v] on the device (once per model; see ds_draft.h)."""
    r, V = P.shape
    return load().ds_transpose_projection(_ptr(P, "P"), r, V, _dtype_code(P), _ptr(P_t, "P_t"),
                                          _stream(stream))


def ds_acceptance_rate(target_logits, draft_logits, temperature, alpha, status, stream=None):
    """alpha[n] = sum_i min(p_n(i), q_n(i)) of [rows, V] target and draft logits."""
    rows, V = target_logits.shape
    return load().ds_acceptance_rate(_ptr(target_logits, "target_logits"), _ptr(draft_logits, "draft_logits"),
                                     rows, V, _dtype_code(target_logits), _ptr(temperature, "temperature"),
                                     _ptr(alpha, "alpha"), _ptr(status, "status"), _stream(stream))


def ds_reserve_persisting_l2(nbytes):
    """Persisting-L2 set-aside of the current device (see ds_draft.h); returns the
    bytes now set aside."""
    return int(load().ds_reserve_persisting_l2(int(nbytes)))


def ds_test_set_wait_hooks(wait_polls, withhold_cta):
    """Test hook of the bounded device waits (see ds_draft.h); (0, -1) clears it."""
    return load().ds_test_set_wait_hooks(int(wait_polls), int(withhold_cta))


def ds_verify_static(target_logits, base_logits, E, P, anchor, draft_tokens, q_token, q_stats,
                     sched_len, temperature, seed, out_tokens, accept_count, num_emitted, status,
                     stream=None, P_t=None, states=None, seed_ptr=None, p_token=None, P_packed=None):
    """ds_verify with the library's static scratch (no workspace argument)."""
    B, K1, V = target_logits.shape
    a = VerifyArgs(B=B, K=K1 - 1, V=V, r=E.shape[1], dtype=_dtype_code(target_logits),
                   target_logits=_ptr(target_logits, "target_logits"),
                   base_logits=_ptr(base_logits, "base_logits"), E=_ptr(E, "E"), P=_ptr(P, "P"),
                   P_t=None if P_t is None else _ptr(P_t, "P_t"),
                   anchor=_ptr(anchor, "anchor"), draft_tokens=_ptr(draft_tokens, "draft_tokens"),
                   q_token=_ptr(q_token, "q_token"), q_stats=_ptr(q_stats, "q_stats"),
                   sched_len=_ptr(sched_len, "sched_len"), temperature=_ptr(temperature, "temperature"),
                   seed=int(seed), out_tokens=_ptr(out_tokens, "out_tokens"),
                   accept_count=_ptr(accept_count, "accept_count"),
                   num_emitted=_ptr(num_emitted, "num_emitted"),
                   workspace=None, workspace_bytes=0, status=_ptr(status, "status"),
                   states=None if states is None else _ptr(states, "states"),
                   seed_ptr=None if seed_ptr is None else _ptr(seed_ptr, "seed_ptr"),
                   p_token=None if p_token is None else _ptr(p_token, "p_token"),
                   P_packed=None if P_packed is None else _ptr(P_packed, "P_packed"))
    return load().ds_verify_static(ctypes.byref(a), _stream(stream))


def ds_sts_workspace_bytes(N, K, n_grid, n_bins):
    return load().ds_sts_workspace_bytes(N, K, n_grid, n_bins)


def ds_sts_fit(logits, labels, grid, n_bins, sts_temp, grid_index, ece, workspace, status,
               ece_curve=None, stream=None):
    """Left-to-right STS temperature fit (float32 logits and labels [N, K], grid [G])."""
    for t, name in ((logits, "logits"), (labels, "labels"), (grid, "grid")):
        if t.dtype != torch.float32:
            raise TypeError("%s must be float32" % name)
    N, K = logits.shape
    a = StsArgs(N=N, K=K, n_grid=int(grid.shape[0]), n_bins=int(n_bins),
                logits=_ptr(logits, "logits"), labels=_ptr(labels, "labels"),
                grid=_ptr(grid, "grid"), sts_temp=_ptr(sts_temp, "sts_temp"),
                grid_index=_ptr(grid_index, "grid_index"), ece=_ptr(ece, "ece"),
                ece_curve=None if ece_curve is None else _ptr(ece_curve, "ece_curve"),
                workspace=_ptr(workspace, "workspace"),
                workspace_bytes=workspace.numel() * workspace.element_size(),
                status=_ptr(status, "status"))
    return load().ds_sts_fit(ctypes.byref(a), _stream(stream))


def ds_copy_scheduled_rows(dst, src, lens, stream=None):
    """Rows 0..L_b of each request's target logits, host ``src`` -> device
    ``dst`` (both [B, K+1, V]); ``lens``: host int32 tensor [B]. Returns
    (status, bytes enqueued)."""
    if dst.dim() != 3 or tuple(src.shape) != tuple(dst.shape) or src.dtype != dst.dtype:
        raise ValueError("dst and src must be [B, K+1, V] tensors of one dtype")
    if src.is_cuda or not src.is_contiguous():
        raise ValueError("src must be a contiguous host tensor")
    if lens.is_cuda or lens.dtype != torch.int32 or lens.numel() != dst.shape[0] or not lens.is_contiguous():
        raise ValueError("lens must be a contiguous host int32 tensor [B]")
    n = ctypes.c_uint64(0)
    code = load().ds_copy_scheduled_rows(_ptr(dst, "dst"), ctypes.c_void_p(src.data_ptr()),
                                         int(dst.shape[0]), int(dst.shape[1]) - 1,
                                         int(dst.shape[2]) * dst.element_size(),
                                         ctypes.c_void_p(lens.data_ptr()), ctypes.byref(n),
                                         _stream(stream))
    return code, int(n.value)


def ds_fetch_scheduled_rows(dst, src, sched_len, bytes_total=None, stream=None):
    """Rows 0..L_b of each request's target logits, fetched by a kernel from
    the pinned host tensor ``src`` into device ``dst`` (both [B, K+1, V]);
    ``sched_len``: device int32 [B]; ``bytes_total``: optional device int64
    counter the fetched bytes are added to."""
    if dst.dim() != 3 or tuple(src.shape) != tuple(dst.shape) or src.dtype != dst.dtype:
        raise ValueError("dst and src must be [B, K+1, V] tensors of one dtype")
    if src.is_cuda or not src.is_contiguous() or not src.is_pinned():
        raise ValueError("src must be a contiguous pinned host tensor")
    if sched_len.dtype != torch.int32 or sched_len.numel() != dst.shape[0]:
        raise ValueError("sched_len must be a device int32 tensor [B]")
    if bytes_total is not None and (bytes_total.dtype != torch.int64 or bytes_total.numel() < 1):
        raise ValueError("bytes_total must be a device int64 tensor")
    return load().ds_fetch_scheduled_rows(_ptr(dst, "dst"), ctypes.c_void_p(src.data_ptr()),
                                          int(dst.shape[0]), int(dst.shape[1]) - 1,
                                          int(dst.shape[2]) * dst.element_size(),
                                          _ptr(sched_len, "sched_len"),
                                          None if bytes_total is None else _ptr(bytes_total, "bytes_total"),
                                          _stream(stream))


def ds_check_status(status, stream=None):
    return load().ds_check_status(_ptr(status, "status"), _stream(stream))


def ds_status_string(code):
    return load().ds_status_string(int(code)).decode()


def ds_version():
    return load().ds_version().decode()
