"""Benchmark: draft + schedule + verify cycles on synthetic inputs, one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one full cycle (ds_draft_block, ds_confidence_schedule, ds_verify) over
one batch of the workload with inputs resident in HBM. The metric is drafted
block tokens per second, B*K / t_cycle, summed over replicas. Multi-GPU runs are
independent replicas (one process per GPU, no collective on the data path).
`--impl reference` times the float64 CPU oracle on a bounded sample instead.
"""
import argparse
import ctypes
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "draft+verify tokens/s at B=128,K=16,V=151936; % of HBM/tensor roofline"
DEFAULT_WORKLOAD = "B128_K16_V151936"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
NOMINAL_HBM_GBS = 8000.0   # nominal HBM3e figure, for the second fraction the line reports


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(PEAKS_FALLBACK), "fallback"


# ---- clocks (read-only NVML queries during the timed region) -------------------

class ClockSampler:
    """Samples SM clock and throttle reasons every few ms through NVML (ctypes)."""
    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}

    def __init__(self, index, period_s=0.005):
        self.index, self.period = index, period_s
        self.samples, self.reasons = [], 0
        self.max_mhz = None
        self.ok = False
        try:
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nv.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            if self.nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h)) != 0:
                return
            mx = ctypes.c_uint()
            if self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = int(mx.value)
            self.ok = True
        except OSError:
            self.ok = False

    def _run(self):
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        get_r = getattr(self.nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(self.nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
        while not self.stop.is_set():
            if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk)) == 0:
                self.samples.append(int(clk.value))
            if get_r(self.h, ctypes.byref(rs)) == 0:
                self.reasons |= int(rs.value)
            time.sleep(self.period)

    def __enter__(self):
        if self.ok:
            self.stop = threading.Event()
            self.th = threading.Thread(target=self._run, daemon=True)
            self.th.start()
        return self

    def __exit__(self, *a):
        if self.ok:
            self.stop.set()
            self.th.join()

    def summary(self):
        if not self.ok or not self.samples:
            return None
        names = sorted(n for bit, n in self.REASONS.items() if self.reasons & bit and bit != 0x1)
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": names, "samples": len(self.samples)}


# ---- workload accounting ---------------------------------------------------------

def draft_algorithmic(inp, rnn=False):
    """Algorithmic HBM bytes and tensor FLOPs of one ds_draft_block call (K
    block positions), counted as the measurement section of the survey defines
    them: every input byte once per cycle. The base logits z (B*K*V), the
    projection P once (r*V: its K-1 re-reads within the call are L2 traffic,
    reported separately), the conditioning rows and hidden states
    (B*K*(r + d): h feeds the confidence head of the same cycle) and the
    outputs (token, q, stats: 24 B per position). FLOPs: the bias product
    2*B*K*r*V.
    RNN head in addition: the packed step matrix (4r x 2r) and W_ih's hidden
    columns (3r x d) once, and per position the input rows [e ; s] (B x 2r),
    the gate inputs (B x 3r float32, written once and read once) and the state
    (B x r, written, read back as the next input); FLOPs of the gated update
    (2*B*4r*2r per position) and of the hidden-state GEMM (2*B*K*3r*d)."""
    B, K, V, r, d = inp["B"], inp["K"], inp["V"], inp["r"], inp["d"]
    eb = 2 if inp["bf16"] else 4
    by = B * K * V * eb + r * V * eb + B * K * (r + d) * eb + B * K * (4 + 4 + 16)
    fl = 2.0 * B * K * r * V
    if rnn:
        by += 4 * r * 2 * r * eb + 3 * r * d * eb
        by += K * (B * 2 * r * eb + 2 * B * 3 * r * 4 + 2 * B * r * eb)
        fl += K * 2.0 * B * 4 * r * 2 * r + 2.0 * B * K * 3 * r * d
    return by, fl


def verify_algorithmic(inp, L, accept, temperature):
    """Algorithmic bytes and FLOPs of one ds_verify call: the target rows up to
    the first rejection (or the bonus row), sum_b min(a_b + 1, L_b + 1) rows;
    for each sampling request that rejects (a_b < L_b, T_b > 0) its base row
    at the rejection (q is rebuilt there), and P once if any request rejects;
    FLOPs: one bias row per rejecting request (2*r*V each). Greedy requests
    rebuild nothing. a_b and L_b are the run's (equal to the oracle's by the
    parity tests)."""
    import numpy as np
    V, r = inp["V"], inp["r"]
    eb = 2 if inp["bf16"] else 4
    L = np.asarray(L, dtype=np.int64)
    a = np.asarray(accept, dtype=np.int64)
    rows = int(np.minimum(a + 1, L + 1).sum())
    n_rej = int(np.sum((a < L) & (np.asarray(temperature) > 0)))
    by = rows * V * eb + n_rej * V * eb + (r * V * eb if n_rej else 0)
    return by, 2.0 * n_rej * r * V, rows, n_rej


def gpu_launches_per_cycle(w, rnn=False):
    """Kernels one cycle launches: draft (tile and locate per position; the RNN
    head adds the hidden-state GEMM, the first input rows and one update per
    position), schedule (confidence, scheduler), verify (rows, finalize, tile,
    locate)."""
    draft = 3 * w.K + 2 if rnn else 2 * w.K
    return draft + 2 + 4


# Per-step inputs (copied host -> device every step in the end-to-end run).
# The weights (E, P and its token-major copy, w_h, w_e) and the tables (STS
# temperatures, SPS) stay resident, as in a serving engine.
STEP_KEYS = ("base_logits", "target_logits", "anchor", "temperature", "h")


# Sources of the draft-step kernels (tile + locate) and everything they include.
STEP_SOURCES = ("draft_tc.cu", "sample.cu", "locate.cuh", "common.cuh", "fastpath.cuh",
                "sampling.cuh", "sm100.cuh", "internal.h", "philox.h")


def sources_digest():
    """sha256 over the draft-step kernels' sources: ties recorded ncu traffic to
    the kernels it measured."""
    import hashlib
    d = os.path.join(ROOT, "speculative_decoding_draft_block_gb300", "csrc")
    h = hashlib.sha256()
    for f in STEP_SOURCES:
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()


def recorded_traffic(workload):
    """DRAM bytes per draft step from the committed ncu summary, if it still
    matches the sources; None otherwise."""
    path = os.path.join(ROOT, "profiles", "draft_step_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    ent = rec.get(workload)
    if not ent or ent.get("sources_sha256") != sources_digest():
        return None
    return float(ent["dram_bytes_per_step"])


# ---- CPU oracle timing ------------------------------------------------------------

def oracle_sample(inp, seed, n_req, rnn_w=None):
    """Time the oracle's cycle on the first n_req requests (schedule on all)."""
    import numpy as np
    import oracle
    rows = np.arange(n_req)
    t0 = time.perf_counter()
    states = None
    if rnn_w is not None:
        d = oracle.rnn_draft_block(inp["base_logits"][rows], inp["E"], inp["P"], inp["anchor"][rows],
                                   inp["temperature"][rows], seed, inp["h"][rows], rnn_w["w_ih"],
                                   rnn_w["w_hh"], rnn_w["b_ih"], rnn_w["b_hh"], inp["bf16"])
        states = d["states"]
    else:
        d = oracle.draft_block(inp["base_logits"][rows], inp["E"], inp["P"], inp["anchor"][rows],
                               inp["temperature"][rows], seed)
    c = oracle.confidence(inp["h"][rows], inp["E"], inp["anchor"][rows], d["tokens"], inp["w_h"],
                          inp["w_e"], inp["conf_bias"], inp["sts_temp"])
    sch = oracle.schedule(oracle.survival(c), inp["sps"])
    oracle.verify(inp["target_logits"][rows], inp["base_logits"][rows], inp["E"], inp["P"],
                  inp["anchor"][rows], d["tokens"], sch["L"], inp["temperature"][rows], seed,
                  states=states)
    dt = time.perf_counter() - t0
    return dt, n_req * inp["K"]


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except ImportError:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    return os.cpu_count() or 1


def cpu_baseline(inp, seed, budget_s=12.0, rnn_w=None):
    n_req = 1
    dt, toks = oracle_sample(inp, seed, n_req, rnn_w)
    if dt < budget_s / 4:
        n_req = max(1, min(inp["B"], int(budget_s / max(dt, 1e-3))))
        dt, toks = oracle_sample(inp, seed, n_req, rnn_w)
    return {"value": toks / dt, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
            "sample": "%d of %d requests x K=%d positions: float64 draft (bias matmul + exp/cumsum "
                      "per position), confidence + schedule, verify; %.1f s" %
                      (n_req, inp["B"], inp["K"], dt)}


# ---- main -------------------------------------------------------------------------

def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 1, 0
    import torch.distributed as dist
    rank = int(os.environ["RANK"])
    local = int(os.environ.get("LOCAL_RANK", rank))
    import torch
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    if backend == "nccl":
        torch.cuda.set_device(local)
    dist.init_process_group(backend=backend)
    return rank, ws, local


def reduce_max(x, ws):
    if ws <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def run_reference(args, rank, ws):
    if rank != 0:
        return
    from speculative_decoding_draft_block_gb300.workloads import WORKLOADS, make_inputs
    w = WORKLOADS[args.workload]
    inp = make_inputs(w)
    n_req = max(1, int(os.environ.get("DS_REF_REQUESTS", "2")))
    for i in range(args.warmup):
        oracle_sample(inp, 0x5EED0000 + i, n_req)
    tot, toks = 0.0, 0
    for i in range(args.steps):
        dt, t = oracle_sample(inp, 0x5EED1000 + i, n_req)
        tot += dt
        toks += t
    value = toks / tot
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "K": w.K, "V": w.V, "r": w.r, "d": w.d,
                       "sample_requests": n_req},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": blas_threads(),
                             "kind": "oracle",
                             "sample": "%d of %d requests per step, all K=%d positions" %
                                       (n_req, w.B, w.K)},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


STS_METRIC = "STS fit: calibration sample-positions/s (N=65536, K=16, 256-point grid, 15 bins)"
STS_N, STS_K, STS_G, STS_BINS = 65536, 16, 256, 15
MUFU_PER_CLK_SM = 16       # exp2 / reciprocal issue rate per SM per clock
MUFU_PER_EVAL = 2          # one exp2 and one reciprocal per sigmoid


def run_sts(args, rank, ws, local):
    """Time ds_sts_fit (all K positions) on the synthetic calibration set."""
    import numpy as np
    import torch
    from speculative_decoding_draft_block_gb300 import _lib
    from speculative_decoding_draft_block_gb300.workloads import make_sts_inputs, sts_grid

    if not os.path.exists(_lib.LIB_PATH):
        from speculative_decoding_draft_block_gb300 import build
        build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    d = make_sts_inputs(STS_N, STS_K, seed=7 + rank)
    grid_h = sts_grid(0.05, 5.0, STS_G)
    a = torch.from_numpy(d["logits"]).to(dev)
    y = torch.from_numpy(d["labels"]).to(dev)
    grid = torch.from_numpy(grid_h).to(dev)
    T = torch.empty((STS_K,), dtype=torch.float32, device=dev)
    idx = torch.empty((STS_K,), dtype=torch.int32, device=dev)
    ece = torch.empty((STS_K,), dtype=torch.float32, device=dev)
    wsb = torch.empty((_lib.ds_sts_workspace_bytes(STS_N, STS_K, STS_G, STS_BINS),), dtype=torch.uint8,
                      device=dev)
    status = torch.zeros((4,), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def fit():
        _lib.check(_lib.ds_sts_fit(a, y, grid, STS_BINS, T, idx, ece, wsb, status), "ds_sts_fit")

    for _ in range(args.warmup):
        fit()
    torch.cuda.synchronize(dev)
    barrier(ws)
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    sampler = ClockSampler(local)
    with sampler:
        for i in range(K):
            flush.zero_()
            ev[i][0].record(stream)
            fit()
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
    barrier(ws)
    _lib.check(_lib.ds_check_status(status), "device status")
    ms = np.array([e0.elapsed_time(e1) for e0, e1 in ev])
    total_s = reduce_max(float(ms.sum()) / 1e3, ws)
    units = STS_N * STS_K
    value = ws * units * K / total_s
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    fmax = (sampler.max_mhz or 2070) * 1e6
    peak = sms * MUFU_PER_CLK_SM * fmax / MUFU_PER_EVAL / 1e12          # T evaluations / s
    evals = STS_N * STS_K * STS_G
    achieved = evals / (float(ms.mean()) * 1e-3) / 1e12
    line = {
        "metric": STS_METRIC, "value": value, "unit": "sample-positions/s", "n_gpus": ws,
        "steps": K, "warmup": args.warmup, "ms_per_step": float(ms.mean()),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded logistic calibration set, over-confident raw head)",
        "config": {"workload": "sts_N%d_K%d_G%d_bins%d" % (STS_N, STS_K, STS_G, STS_BINS),
                   "parallelism": "replicas" if ws > 1 else "single",
                   "l2": "flushed between steps (256 MiB write, outside the timed events)"},
        "roofline": {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "T sigmoid evals/s",
                     "frac": achieved / peak, "traffic": None,
                     "kernel": "whole ds_sts_fit call (sts_fit_kernel, one launch per position)",
                     "peak_source": "derived: SMs x %d MUFU/clk / %d MUFU per evaluation x max SM clock"
                                    % (MUFU_PER_CLK_SM, MUFU_PER_EVAL)},
        "gpu_launches": K * STS_K,
        "fitted_temps": [float(x) for x in T.cpu().numpy()],
        "ece": [float(x) for x in ece.cpu().numpy()],
        "clocks": sampler.summary(),
    }
    # end to end: logits and labels copied from pinned host memory, temperatures copied back
    ha = torch.from_numpy(d["logits"]).pin_memory()
    hy = torch.from_numpy(d["labels"]).pin_memory()
    hT = torch.empty((STS_K,), dtype=torch.float32).pin_memory()
    E = max(1, args.e2e_steps)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(E):
        a.copy_(ha, non_blocking=True)
        y.copy_(hy, non_blocking=True)
        fit()
        hT.copy_(T, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_s = reduce_max(e0.elapsed_time(e1) / 1e3, ws)
    line["e2e"] = {"value": ws * units * E / e2e_s, "unit": "sample-positions/s",
                   "h2d_bytes_per_step": int(ha.numel() * 4 + hy.numel() * 4),
                   "d2h_bytes_per_step": int(hT.numel() * 4), "steps": E}
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        import oracle
        n = 8192
        t0 = time.perf_counter()
        oracle.sts_fit(d["logits"][:n], d["labels"][:n], grid_h.astype(np.float64), STS_BINS)
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": n * STS_K / dt, "unit": "sample-positions/s",
                                "cores": 1, "kind": "oracle",
                                "sample": "first %d of %d samples, all %d positions and %d grid points"
                                          % (n, STS_N, STS_K, STS_G)}
    if rank == 0:
        print(json.dumps(line), flush=True)


def time_graph_replays(args, inp, dev, rnn_w, seed0, flush, stream, ws, per):
    """The cycle captured once (Philox key and scheduler ring on the device, the
    key advanced inside the graph) and timed as K replays with CUDA events; the
    per-call split and the draft-step roofline come from the launched calls."""
    import numpy as np
    import torch
    from speculative_decoding_draft_block_gb300.cycle import DeviceCycle
    K = args.steps
    gc = DeviceCycle(inp, device=dev, mode=args.mode, threshold=args.threshold, rnn_weights=rnn_w,
                     device_seed=True)
    gc.set_seed(seed0)
    gc.run(0)
    torch.cuda.synchronize(dev)
    gc.reset_status()
    graph = torch.cuda.CUDAGraph()
    failed = None
    try:
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                gc.run(0)
                gc.seed_dev[0].add_(1)
        torch.cuda.synchronize(dev)
    except Exception as ex:  # noqa: BLE001 - reported in the line, timing falls back
        failed = "%s: %s" % (type(ex).__name__, str(ex)[:200])
    # every rank takes the same path through the barriers below
    if reduce_max(1.0 if failed else 0.0, ws) > 0:
        raise RuntimeError(failed or "CUDA graph capture failed on another rank")
    gc.set_seed(seed0 + 1000)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize(dev)
    barrier(ws)
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    for i in range(K):
        flush.zero_()
        gev[i][0].record(stream)
        graph.replay()
        gev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    barrier(ws)
    gc.check_status()
    return np.array([a.elapsed_time(b) for a, b in gev]), float(np.median(per.sum(axis=1)))


DRAFT_KEYS = ("base_logits", "anchor", "temperature", "h")
MODE_NAMES = {0: "greedy_earlystop", 1: "fixed_k", 2: "threshold", 3: "async"}


def time_e2e(args, cyc, inp, stream, dev, seed0, ws):
    """End to end through the public API (``HostPipeline``), as a caller holding
    each step's inputs in pinned host memory runs it: the draft's inputs are
    copied in, draft and schedule run, only the target rows that verify reads
    (rows 0..L_b of request b) are fetched from the pinned host tensor by a
    kernel that reads L_b on the device, verify runs, and the scheduled lengths
    and emitted tokens come back. Each step also starts the copy of the next step's draft inputs
    (independent request groups served in turn), which overlaps the current
    step. Every copy is inside the timed region: the copy stream waits for the
    start event, and the last step stages nothing ahead. The bytes are counted
    from the copies (the fetched rows on a device counter)."""
    import numpy as np
    import torch
    from speculative_decoding_draft_block_gb300.cycle import HostPipeline, to_host_pinned
    B, K = inp["B"], inp["K"]
    host = {k: to_host_pinned(inp[k]) for k in STEP_KEYS}
    pipe = HostPipeline(cyc, stream)
    for i in range(2):
        pipe.step(host, seed0 + i)
    torch.cuda.synchronize(dev)
    barrier(ws)
    E = max(1, args.e2e_steps)
    # the timed region is run three times and the median reported (the host
    # link is shared with the rest of the machine); every sample is listed
    values, h2d = [], 0
    for rep in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        pipe.reset_counts()
        e0.record(stream)
        pipe.copy_stream.wait_event(e0)
        for i in range(E):
            pipe.step(host, seed0 + 5000 + 100 * rep + i, next_host=host if i + 1 < E else None)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_s = reduce_max(e0.elapsed_time(e1) / 1e3, ws)
        values.append(ws * B * K * E / e2e_s)
        h2d = pipe.h2d_bytes()
    return {"value": float(np.median(values)), "unit": "tokens/s", "samples": [float(v) for v in values],
            "h2d_bytes_per_step": int(h2d / E), "d2h_bytes_per_step": int(pipe.d2h_bytes),
            "steps": E,
            "copied": list(DRAFT_KEYS) + ["target_logits rows 0..L_b", "sched_len", "out_tokens",
                                           "num_emitted"],
            "overlap": "next step's draft inputs copied during the current step (copy stream); "
                       "target rows 0..L_b fetched by a kernel from pinned host memory, L_b read "
                       "on the device"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--mode", type=int, default=0, choices=(0, 1, 2, 3),
                    help="scheduler: 0 greedy + early stop, 1 fixed K, 2 survival threshold, "
                         "3 asynchronous (budget from two cycles back)")
    ap.add_argument("--threshold", type=float, default=0.5, help="survival threshold of mode 2")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", dest="graph", action="store_false",
                    help="time the launched calls instead of replays of one captured cycle")
    ap.add_argument("--head", choices=("markov", "rnn"), default="markov",
                    help="sequential head of the draft block (default: Markov)")
    ap.add_argument("--l2-persist", type=float, default=None,
                    help="MB of L2 to set aside for persisting lines (keeps P resident across "
                         "the draft steps); default: P's size; 0 disables")
    ap.add_argument("--part", choices=("cycle", "sts"), default="cycle",
                    help="cycle: draft+schedule+verify (default); sts: the STS calibration fit")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    rank, ws, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank, ws)
        return
    if args.part == "sts":
        run_sts(args, rank, ws, local)
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    import numpy as np
    import torch
    from speculative_decoding_draft_block_gb300 import _lib
    from speculative_decoding_draft_block_gb300.cycle import DeviceCycle, to_host_pinned
    from speculative_decoding_draft_block_gb300.workloads import WORKLOADS, make_inputs

    if not os.path.exists(_lib.LIB_PATH):
        from speculative_decoding_draft_block_gb300 import build
        build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = WORKLOADS[args.workload]
    inp = make_inputs(w)
    rnn = args.head == "rnn"
    rnn_w = None
    if rnn:
        from speculative_decoding_draft_block_gb300.workloads import make_rnn_weights
        rnn_w = make_rnn_weights(w.r, w.d)
    cyc = DeviceCycle(inp, device=dev, mode=args.mode, threshold=args.threshold, rnn_weights=rnn_w)
    p_bytes = w.r * w.V * (2 if w.bf16 else 4)
    want = p_bytes if args.l2_persist is None else int(args.l2_persist * 1e6)
    l2_persist = _lib.ds_reserve_persisting_l2(want)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)   # > 129 MB L2
    seed0 = 0x5EED0000 + 7919 * rank

    for i in range(args.warmup):
        cyc.run(seed0 + i)
    torch.cuda.synchronize(dev)
    cyc.reset_status()
    barrier(ws)
    torch.cuda.synchronize(dev)

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    sampler = ClockSampler(local)
    t_wall = time.perf_counter()
    with sampler:
        for i in range(K):
            flush.zero_()                       # untimed L2 flush between cycles
            e = ev[i]
            e[0].record(stream)
            cyc.draft(seed0 + 1000 + i)
            e[1].record(stream)
            cyc.schedule()
            e[2].record(stream)
            cyc.verify(seed0 + 1000 + i)
            e[3].record(stream)
        torch.cuda.synchronize(dev)
    barrier(ws)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - t_wall
    cyc.check_status()
    per = np.array([[e[0].elapsed_time(e[1]), e[1].elapsed_time(e[2]), e[2].elapsed_time(e[3])]
                    for e in ev])
    cycle_ms = per.sum(axis=1)
    graph_launch_ms = None
    graph_error = None
    try:
        if args.graph:
            cycle_ms, graph_launch_ms = time_graph_replays(args, inp, dev, rnn_w, seed0, flush, stream,
                                                           ws, per)
    except Exception as ex:  # the capture is refused: keep the launched timing and say why
        graph_error = "%s: %s" % (type(ex).__name__, str(ex)[:200])
    # the median timed cycle (the survey's protocol), the slowest rank's
    med_ms = reduce_max(float(np.median(cycle_ms)), ws)
    B, Kb, V = w.B, w.K, w.V
    value = ws * B * Kb / (med_ms * 1e-3)
    res = cyc.results()

    peaks, peak_src = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    tc = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
    d_by, d_fl = draft_algorithmic(inp, rnn)     # per ds_draft_block call (K steps)
    s_by, s_fl = d_by / Kb, d_fl / Kb            # per draft step
    d_ms = float(np.median(per[:, 0])) / Kb      # median draft step (tile + locate kernels)
    t_hbm = s_by / (hbm * 1e9)
    t_tc = s_fl / (tc * 1e12)
    traffic = None if rnn else recorded_traffic(w.name)
    if t_hbm >= t_tc:
        achieved = s_by / (d_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "traffic": traffic}
    else:
        achieved = s_fl / (d_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": tc, "unit": "TFLOP/s",
                "frac": achieved / tc, "traffic": traffic}
    if roof["unit"] == "GB/s":
        roof["frac_nominal"] = roof["achieved"] / NOMINAL_HBM_GBS
    eb = 2 if w.bf16 else 4
    p_rereads = (Kb - 1) * w.r * V * eb / Kb     # per step: P read again by steps 2..K
    roof.update({"kernel": "draft step = tile_tc_kernel + sample_locate_kernel (K per ds_draft_block)"
                 + (" + rnn_gemm_kernel<update> (+ 1/K of the hidden-state GEMM)" if rnn else ""),
                 "peak_source": peak_src, "peak_kind": "burst copy (hbm_gbs); sustained bf16 GEMM",
                 "algorithmic_bytes_per_step": s_by, "algorithmic_flops_per_step": s_fl,
                 "bytes_rule": "per cycle B*K*V + r*V (P once) + B*K*(r+d) elements + outputs, / K",
                 "t_roof_us": 1e6 * max(t_hbm, t_tc), "t_meas_us": 1e3 * d_ms,
                 "traffic_over_algorithmic": None if traffic is None else traffic / s_by,
                 # the same step if P had to come from DRAM at every step (the L2 misses
                 # this accounting leaves to the kernel)
                 "p_every_step": {"bytes_per_step": s_by + p_rereads,
                                  "achieved_gbs": (s_by + p_rereads) / (d_ms * 1e-3) / 1e9,
                                  "frac": (s_by + p_rereads) / (d_ms * 1e-3) / 1e9 / hbm}})
    v_by, v_fl, v_rows, n_rej = verify_algorithmic(inp, res["L"], res["accept_count"], inp["temperature"])
    t_draft_roof = max(d_by / (hbm * 1e9), d_fl / (tc * 1e12))
    t_verify_roof = max(v_by / (hbm * 1e9), v_fl / (tc * 1e12))
    cycle_roof_us = 1e6 * (t_draft_roof + t_verify_roof)
    comp_med = {"draft": float(np.median(per[:, 0])), "schedule": float(np.median(per[:, 1])),
                "verify": float(np.median(per[:, 2]))}

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": med_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.bf16 else "f32",
        "data": "synthetic (seeded, shapes and distributions of the workload)",
        "config": {"workload": w.name, "B": B, "K": Kb, "V": V, "r": w.r, "d": w.d,
                   "parallelism": "replicas" if ws > 1 else "single",
                   "l2": "flushed between steps (256 MiB write, outside the timed events); "
                         "inputs also exceed L2",
                   "mode": MODE_NAMES[args.mode],
                   "threshold": args.threshold if args.mode == 2 else None,
                   "head": args.head, "cuda_graph": graph_launch_ms is not None,
                   "timing": "median of the timed cycles (CUDA events; max over ranks)",
                   "l2_persisting_bytes": l2_persist,
                   "cuda_graph_error": graph_error},
        "ms_per_step_mean": float(cycle_ms.mean()),
        "components_ms": comp_med,
        "components_roofline_us": {"draft": 1e6 * t_draft_roof, "verify": 1e6 * t_verify_roof,
                                   "verify_target_rows": v_rows, "verify_rejecting_requests": n_rej},
        "components_roofline_frac": {"draft": 1e3 * t_draft_roof / comp_med["draft"],
                                     "verify": 1e3 * t_verify_roof / comp_med["verify"]},
        "launched_cycle_ms": graph_launch_ms,
        "emitted_tokens_per_s": ws * float(res["num_emitted"].sum()) / (med_ms * 1e-3),
        "verified_tokens_per_s": ws * float((res["L"] + 1).sum()) / (med_ms * 1e-3),
        "mean_sched_len": float(res["L"].mean()), "mean_accepted": float(res["accept_count"].mean()),
        "cycle_roofline_us": cycle_roof_us, "cycle_roofline_frac": cycle_roof_us / (1e3 * med_ms),
        "roofline": roof,
        "gpu_launches": K * (gpu_launches_per_cycle(w, rnn)),
        "wall_s": wall,
        "clocks": sampler.summary(),
    }

    if not args.no_e2e:
        line["e2e"] = time_e2e(args, cyc, inp, stream, dev, seed0, ws)
        cyc.check_status()

    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp, 0x5EED0000, rnn_w=rnn_w)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
