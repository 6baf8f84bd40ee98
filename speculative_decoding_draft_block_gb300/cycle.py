"""One speculative cycle on the GPU through the C ABI: draft -> schedule -> verify.

`DeviceCycle` owns the device buffers of one workload (PyTorch allocations used
as plain device memory) and issues the three library calls on a stream. It does
no arithmetic of its own.
"""

import numpy as np
import torch

from . import _lib
from ._lib import check


def _to_device(a, device):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def to_host_pinned(a):
    """Pinned host copy of an input array (bf16 kept as bf16)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(a)
    return t.pin_memory()


INPUT_KEYS = ("base_logits", "target_logits", "E", "P", "anchor", "temperature", "h", "w_h",
              "w_e", "sts_temp", "sps")


GUARD_BYTES = 256                 # per side of a guarded buffer (a multiple of 16)
GUARD_BYTE = 0xA5                 # the sentinel byte of the guard regions


class DeviceCycle:
    def __init__(self, inp, device="cuda", mode=_lib.DS_SCHED_GREEDY_EARLYSTOP, threshold=0.0,
                 token_major_projection=True, initial_budget=None, rnn_weights=None,
                 device_seed=False, guards=False, packed_projection=True):
        """``rnn_weights`` (dict w_ih, w_hh as bfloat16 bits, b_ih, b_hh float32)
        selects the RNN head; its step matrix is packed once here.
        ``device_seed``: the Philox key is read from a device word (``seed_dev``,
        set with ``set_seed``) instead of the ``seed`` argument, so that a
        captured cycle can be replayed with a fresh key each time.
        ``packed_projection``: the tile-packed copy of P (ds_pack_projection) is
        made once here and passed to draft and verify when the shape allows.
        ``guards``: every buffer the library writes (outputs and workspaces) sits
        between two GUARD_BYTES regions of sentinel bytes; ``guard_damage()``
        lists the buffers whose guards changed (a write out of bounds)."""
        self.inp = inp
        self.device = torch.device(device)
        self.mode = mode
        self.threshold = threshold
        B, K, V, r = inp["B"], inp["K"], inp["V"], inp["r"]
        self.B, self.K, self.V, self.r, self.d = B, K, V, r, inp["d"]
        dev = self.device
        self._guarded = [] if guards else None
        self.t = {k: _to_device(inp[k], dev) for k in INPUT_KEYS}
        self.t["anchor"] = self.t["anchor"].to(torch.int32)
        self.conf_bias = float(inp["conf_bias"])
        i32, f32 = torch.int32, torch.float32
        self.draft_tokens = self._out("draft_tokens", (B, K), i32)
        self.q_token = self._out("q_token", (B, K), f32)
        self.q_stats = self._out("q_stats", (B, K, 4), i32)
        self.conf = self._out("conf", (B, K), f32)
        self.conf_logit = self._out("conf_logit", (B, K), f32)   # raw logit: the STS fit's input
        self.survival = self._out("survival", (B, K), f32)
        self.sched_len = self._out("sched_len", (B,), i32)
        self.objective = self._out("objective", (2,), torch.float64)
        self.out_tokens = self._out("out_tokens", (B, K + 1), i32)
        self.accept_count = self._out("accept_count", (B,), i32)
        self.num_emitted = self._out("num_emitted", (B,), i32)
        self.p_token = self._out("p_token", (B, K), f32)   # target probability of each verified token
        self.status = self._out("status", (4,), i32)
        # asynchronous scheduler: budgets of the next two cycles and the cycle
        # counter, all on the device; the first two cycles use initial_budget
        if initial_budget is None:
            initial_budget = B * K // 2
        self.initial_budget = int(initial_budget)
        self.budget_ring = self._out("budget_ring", (4,), i32)
        self.budget_ring.copy_(torch.tensor([self.initial_budget, self.initial_budget, 0, 0], dtype=i32))
        self.seed_dev = torch.zeros((2,), dtype=torch.int64, device=dev) if device_seed else None
        wd = _lib.ds_draft_workspace_bytes(B, K, V, r)
        wv = _lib.ds_verify_workspace_bytes(B, K, V, r)
        if wd == 0 or wv == 0:
            raise ValueError("shape not supported by the library")
        self.rnn = None
        if rnn_weights is not None:
            wr = _lib.ds_rnn_workspace_bytes(B, K, r)
            if wr == 0:
                raise ValueError("shape not supported by the RNN head")
            wd = (wd + 255) // 256 * 256 + wr
            rw = {k: _to_device(rnn_weights[k], dev) for k in ("w_ih", "w_hh", "b_ih", "b_hh")}
            rw["h"] = self.t["h"]
            rw["w_step"] = self._out("w_step", (4 * r, 2 * r), rw["w_ih"].dtype)
            check(_lib.ds_rnn_pack_weights(rw["w_ih"], rw["w_hh"], rw["w_step"]), "ds_rnn_pack_weights")
            rw["states"] = self._out("states", (B, K, r), rw["w_ih"].dtype)
            self.rnn = rw
        self.ws_draft = self._out("ws_draft", (wd,), torch.uint8)
        self.ws_verify = self._out("ws_verify", (wv,), torch.uint8)
        # weight layout step, once per model: the token-major copy of P
        self.P_t = None
        if token_major_projection:
            P = self.t["P"]
            self.P_t = self._out("P_t", (P.shape[1], P.shape[0]), P.dtype)
            check(_lib.ds_transpose_projection(P, self.P_t), "ds_transpose_projection")
        # weight layout step, once per model: the tile-packed copy of P
        self.P_packed = None
        nbytes = _lib.ds_packed_projection_bytes(r, V) if inp["bf16"] else 0
        if packed_projection and nbytes > 0:
            self.P_packed = self._out("P_packed", (nbytes,), torch.uint8)
            check(_lib.ds_pack_projection(self.t["P"], self.P_packed), "ds_pack_projection")

    def _out(self, name, shape, dtype):
        """A zeroed device buffer; with guards, the middle of a larger buffer
        whose GUARD_BYTES on each side hold the sentinel byte."""
        n = 1
        for x in shape:
            n *= x
        if self._guarded is None:
            return torch.zeros(shape, dtype=dtype, device=self.device)
        esz = torch.empty((), dtype=dtype).element_size()
        nbytes = n * esz
        body = (nbytes + 15) // 16 * 16
        raw = torch.full((GUARD_BYTES + body + GUARD_BYTES,), GUARD_BYTE, dtype=torch.uint8,
                         device=self.device)
        raw[GUARD_BYTES:GUARD_BYTES + nbytes].zero_()
        self._guarded.append((name, raw, nbytes))
        return raw[GUARD_BYTES:GUARD_BYTES + nbytes].view(dtype).view(shape)

    def guard_damage(self):
        """Names of the guarded buffers whose guard bytes (before the buffer, or
        after its last element up to the guard's end) are no longer the
        sentinel. Empty without guards."""
        bad = []
        for name, raw, nbytes in self._guarded or []:
            host = raw.cpu().numpy()
            if (host[:GUARD_BYTES] != GUARD_BYTE).any() or (host[GUARD_BYTES + nbytes:] != GUARD_BYTE).any():
                bad.append(name)
        return bad

    def set_seed(self, seed):
        """Write the Philox key to the device word (a device-side fill: capturable)."""
        seed = int(seed) & 0xFFFFFFFFFFFFFFFF
        self.seed_dev[0].fill_(seed - (1 << 64) if seed >= (1 << 63) else seed)  # same 64 bits

    def reset_ring(self):
        self.budget_ring.copy_(torch.tensor([self.initial_budget, self.initial_budget, 0, 0],
                                            dtype=torch.int32))

    # -- the three calls ---------------------------------------------------------
    def draft(self, seed, stream=None):
        t = self.t
        check(_lib.ds_draft_block(t["base_logits"], t["E"], t["P"], t["anchor"], t["temperature"],
                                  seed, self.draft_tokens, self.q_token, self.q_stats,
                                  self.ws_draft, self.status, stream, P_t=self.P_t, rnn=self.rnn,
                                  seed_ptr=self.seed_dev, P_packed=self.P_packed),
              "ds_draft_block")

    def schedule(self, stream=None):
        t = self.t
        check(_lib.ds_confidence_schedule(t["h"], t["E"], t["anchor"], self.draft_tokens, t["w_h"],
                                          t["w_e"], self.conf_bias, t["sts_temp"], t["sps"],
                                          self.mode, self.conf, self.survival, self.sched_len,
                                          self.objective, self.status, threshold=self.threshold,
                                          stream=stream, budget_ring=self.budget_ring,
                                          conf_logit=self.conf_logit),
              "ds_confidence_schedule")

    def verify(self, seed, stream=None):
        t = self.t
        check(_lib.ds_verify(t["target_logits"], t["base_logits"], t["E"], t["P"], t["anchor"],
                             self.draft_tokens, self.q_token, self.q_stats, self.sched_len,
                             t["temperature"], seed, self.out_tokens, self.accept_count,
                             self.num_emitted, self.ws_verify, self.status, stream, P_t=self.P_t,
                             states=None if self.rnn is None else self.rnn["states"],
                             seed_ptr=self.seed_dev, p_token=self.p_token, P_packed=self.P_packed),
              "ds_verify")

    def run(self, seed, stream=None):
        """Enqueue one cycle (three library calls); no host synchronisation."""
        self.draft(seed, stream)
        self.schedule(stream)
        self.verify(seed, stream)

    def check_status(self, stream=None):
        code = _lib.ds_check_status(self.status, stream)
        check(code, "device status")

    def reset_status(self):
        self.status.zero_()

    def results(self):
        st = self.q_stats.cpu().numpy()
        return {
            "tokens": self.draft_tokens.cpu().numpy().astype(np.int64),
            "q_token": self.q_token.cpu().numpy().astype(np.float64),
            "q_sum": st[..., 0].view(np.float32).astype(np.float64) + st[..., 1].view(np.float32),
            "q_ref": st[..., 2].copy(),
            "conf": self.conf.cpu().numpy().astype(np.float64),
            "conf_logit": self.conf_logit.cpu().numpy().astype(np.float64),
            "survival": self.survival.cpu().numpy().astype(np.float64),
            "L": self.sched_len.cpu().numpy().astype(np.int64),
            "objective": float(self.objective[0].item()),
            "out_tokens": self.out_tokens.cpu().numpy().astype(np.int64),
            "accept_count": self.accept_count.cpu().numpy().astype(np.int64),
            "num_emitted": self.num_emitted.cpu().numpy().astype(np.int64),
            "p_token": self.p_token.cpu().numpy().astype(np.float64),
            "states": None if self.rnn is None else
            self.rnn["states"].cpu().view(torch.int16).numpy().view(np.uint16),
        }


DRAFT_INPUT_KEYS = ("base_logits", "anchor", "temperature", "h")


class HostPipeline:
    """Cycles whose per-step inputs arrive in pinned host memory.

    A step copies its draft inputs (base logits, anchor, temperatures, h) into
    one of two device slots on a copy stream, runs the draft and the schedule,
    then ``ds_fetch_scheduled_rows`` pulls the target rows that verify reads
    (rows 0..L_b of request b) straight from the pinned host tensor, with L_b
    read on the device: nothing waits on the host inside a step. Verify runs
    and the scheduled lengths and emitted tokens are copied back. Given
    ``next_host``, a step also starts the copy of the next step's draft inputs
    into the other slot at once, so that it overlaps this step; that needs the
    next step's inputs to be known already (for instance two request groups
    served in turn). Events order every reuse: a slot is refilled only after
    the verify that last read it, and a draft waits for its slot's copy.
    Weights and tables stay resident in the ``DeviceCycle``.
    """

    def __init__(self, cyc, stream=None):
        self.cyc = cyc
        dev = cyc.device
        self.stream = stream if stream is not None else torch.cuda.current_stream(dev)
        self.copy_stream = torch.cuda.Stream(dev)
        self.slots = [{k: cyc.t[k] for k in DRAFT_INPUT_KEYS},
                      {k: torch.empty_like(cyc.t[k]) for k in DRAFT_INPUT_KEYS}]
        self.ready = [torch.cuda.Event(), torch.cuda.Event()]
        self.free = [torch.cuda.Event(), torch.cuda.Event()]
        self.done = [torch.cuda.Event(), torch.cuda.Event()]
        B, K = cyc.B, cyc.K
        self.lens = [torch.empty((B,), dtype=torch.int32).pin_memory() for _ in range(2)]
        self.out_tokens = [torch.empty((B, K + 1), dtype=torch.int32).pin_memory() for _ in range(2)]
        self.num_emitted = [torch.empty((B,), dtype=torch.int32).pin_memory() for _ in range(2)]
        self.rows_bytes = torch.zeros((1,), dtype=torch.int64, device=dev)  # fetched target-row bytes
        self.input_bytes = 0    # staged draft-input bytes
        self._next = 0          # slot of the next unstaged step
        self._staged = None     # (slot, host inputs) of a copy already enqueued
        self.d2h_bytes = (B + B * (K + 1) + B) * 4  # per step: lengths, tokens, counts

    def reset_counts(self):
        self.input_bytes = 0
        self.rows_bytes.zero_()

    def h2d_bytes(self):
        """Bytes copied to the device since the last reset (reads the device
        counter: call once the steps are done)."""
        return self.input_bytes + int(self.rows_bytes.item())

    def _stage(self, slot, host):
        cs = self.copy_stream
        cs.wait_event(self.free[slot])
        with torch.cuda.stream(cs):
            for k in DRAFT_INPUT_KEYS:
                dst, src = self.slots[slot][k], host[k]
                if src.dtype != dst.dtype:
                    if src.element_size() != dst.element_size():
                        raise ValueError("host input %s has dtype %s, the device buffer %s" %
                                         (k, src.dtype, dst.dtype))
                    src = src.view(dst.dtype)
                dst.copy_(src, non_blocking=True)
                self.input_bytes += src.numel() * src.element_size()
        self.ready[slot].record(cs)

    def step(self, host, seed, next_host=None):
        """One cycle on ``host`` (pinned tensors: the draft inputs and
        ``target_logits`` [B, K+1, V]). Returns the pinned host tensors
        (lengths, out_tokens, num_emitted) and the event after which they hold
        this step's results; they are reused two steps later."""
        cyc, s = self.cyc, self.stream
        if self._staged is not None and self._staged[1] is host:
            slot = self._staged[0]
        else:
            slot = self._next
            self._stage(slot, host)
        self._staged = None
        self._next = slot ^ 1
        if next_host is not None:
            self._stage(slot ^ 1, next_host)
            self._staged = (slot ^ 1, next_host)
        s.wait_event(self.ready[slot])
        resident = {k: cyc.t[k] for k in DRAFT_INPUT_KEYS}
        cyc.t.update(self.slots[slot])
        try:
            cyc.draft(seed, s)
            cyc.schedule(s)
            check(_lib.ds_fetch_scheduled_rows(cyc.t["target_logits"], host["target_logits"], cyc.sched_len,
                                               self.rows_bytes, s), "ds_fetch_scheduled_rows")
            cyc.verify(seed, s)
            self.free[slot].record(s)
            with torch.cuda.stream(s):
                self.lens[slot].copy_(cyc.sched_len, non_blocking=True)
                self.out_tokens[slot].copy_(cyc.out_tokens, non_blocking=True)
                self.num_emitted[slot].copy_(cyc.num_emitted, non_blocking=True)
            self.done[slot].record(s)
        finally:
            cyc.t.update(resident)
        return self.lens[slot], self.out_tokens[slot], self.num_emitted[slot], self.done[slot]
