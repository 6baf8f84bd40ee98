"""Seeded synthetic inputs for the draft/schedule/verify cycle.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic, so the CUDA path and the test oracle can both consume its
arrays. Everything is generated on the host with NumPy (PCG64 streams derived
from one SeedSequence), in float32, and rounded once to bfloat16 (round to
nearest even) where a workload is bf16, so both sides read identical bits.

Recipe (every workload):
  z[b, k, :]      ~ N(0, sigma_z^2)           k = 1 .. K+1
  true token      t[b, k] ~ U[0, V)  gets  + bump_k
  target[b, k, :] = z[b, k, :] + N(0, sigma_b^2)   sigma_b per request where mixed
  base_logits     = z[:, 1..K, :]   (row K+1 only feeds the bonus target row)
  anchor          ~ U[0, V)
  E, P            ~ N(0, 1/r);  h ~ N(0, 1);  w_h, w_e ~ N(0, 1/d)
  STS temps T_k, sampling temperature, SPS table, confidence bias b: per config.
"""

from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
import os

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    K: int
    V: int
    r: int
    d: int
    bf16: bool
    sigma_z: float
    bump0: float
    bump_decay: float          # bump_k = max(0, bump0 - bump_decay * (k - 1))
    sigma_b: tuple             # (lo, hi) uniform per request; lo == hi for a constant
    sts: tuple                 # (lo, hi) uniform per position; (1, 1) for none
    temps: tuple               # sampling temperatures drawn uniformly per request
    sps_kind: str              # "tiny", "hyperbolic" or "piecewise"
    sps_nmax: int
    conf_bias: float
    seed: int = 0
    extra: dict = field(default_factory=dict)


def _sps_table(kind, n_max):
    n = np.arange(1, n_max + 1, dtype=np.float64)
    if kind == "tiny":
        return (n / (1.0 + n / 64.0)).astype(np.float32)
    if kind == "hyperbolic":
        return (n * 9e4 / (1.0 + n / 96.0)).astype(np.float32)
    if kind == "piecewise":
        knots = np.array([1.0, 64.0, 256.0, 1024.0, 2048.0])
        vals = knots * 9e4 / (1.0 + knots / 96.0)
        return np.interp(n, knots, vals).astype(np.float32)   # flat beyond 2048
    raise ValueError(kind)


def _cfg(name, **kw):
    return Workload(name=name, **kw)


# The five workloads the method is measured on: batch B, block K, vocabulary
# V, rank r, hidden size d, logit spread sigma_z, the true token's bump (bump0,
# falling by bump_decay per position), per-request target noise sigma_b, STS
# temperatures, sampling temperatures, the SPS table and the confidence bias.
# Where a workload leaves a value open it takes the B=32 workload's (bf16
# N(0, 1.5^2) logits, +5 bump, STS temperatures U[0.8, 1.5]).
TINY = _cfg("tiny_B4_K4_V1024", B=4, K=4, V=1024, r=32, d=256, bf16=False, sigma_z=2.0,
            bump0=4.0, bump_decay=0.0, sigma_b=(0.5, 0.5), sts=(1.0, 1.0), temps=(1.0,),
            sps_kind="tiny", sps_nmax=4 * 5, conf_bias=0.0, seed=1000)
B32 = _cfg("B32_K8_V151936", B=32, K=8, V=151936, r=256, d=2560, bf16=True, sigma_z=1.5,
           bump0=5.0, bump_decay=0.0, sigma_b=(0.7, 0.7), sts=(0.8, 1.5), temps=(1.0,),
           sps_kind="hyperbolic", sps_nmax=32 * 9, conf_bias=3.0, seed=1001)
B128 = _cfg("B128_K16_V151936", B=128, K=16, V=151936, r=256, d=4096, bf16=True, sigma_z=1.5,
            bump0=5.0, bump_decay=0.25, sigma_b=(0.3, 1.2), sts=(0.8, 1.5), temps=(1.0,),
            sps_kind="hyperbolic", sps_nmax=128 * 17, conf_bias=3.0, seed=1002)
B512 = _cfg("B512_K16_V129280", B=512, K=16, V=129280, r=256, d=7168, bf16=True, sigma_z=1.5,
            bump0=5.0, bump_decay=0.0, sigma_b=(0.3, 1.5), sts=(0.8, 1.5), temps=(1.0,),
            sps_kind="piecewise", sps_nmax=8192, conf_bias=3.0, seed=1003)
B256 = _cfg("B256_K32_V151936", B=256, K=32, V=151936, r=256, d=4096, bf16=True, sigma_z=1.5,
            bump0=6.0, bump_decay=0.2, sigma_b=(0.2, 1.0), sts=(0.8, 1.5), temps=(0.0, 0.6, 1.0),
            sps_kind="hyperbolic", sps_nmax=256 * 33, conf_bias=3.0, seed=1004)

# Same per-step shape as the B=128 workload with fewer block positions: for
# profiler captures, which replay each kernel many times and must stay small.
B128_K4 = _cfg("B128_K4_V151936", B=128, K=4, V=151936, r=256, d=4096, bf16=True, sigma_z=1.5,
               bump0=5.0, bump_decay=0.25, sigma_b=(0.3, 1.2), sts=(0.8, 1.5), temps=(1.0,),
               sps_kind="hyperbolic", sps_nmax=128 * 5, conf_bias=3.0, seed=1005)

WORKLOADS = {w.name: w for w in (TINY, B32, B128, B512, B256, B128_K4)}


def scaled(w, **changes):
    """A copy of a workload with some fields replaced (smaller parity cases)."""
    kw = {k: getattr(w, k) for k in w.__dataclass_fields__}
    kw.update(changes)
    if "sps_nmax" not in changes:
        kw["sps_nmax"] = kw["B"] * (kw["K"] + 1) if w.sps_kind != "piecewise" else w.sps_nmax
    return Workload(**kw)


def to_bf16_bits(x):
    """Round float32 to bfloat16 (nearest even) and return the uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


def _normal(seedseq, shape, scale):
    rng = np.random.Generator(np.random.PCG64(seedseq))
    return rng.standard_normal(size=shape, dtype=np.float32) * np.float32(scale)


def make_inputs(w, seed=None, threads=None):
    """Generate one workload's inputs as host NumPy arrays (deterministic in the seed).

    Logit-like arrays are uint16 bfloat16 bit patterns when ``w.bf16`` else
    float32. Returns a dict; see the module docstring for the recipe.
    """
    seed = w.seed if seed is None else seed
    ss = np.random.SeedSequence(seed)
    (s_small, s_E, s_P, s_h, s_rows) = ss.spawn(5)
    rng = np.random.Generator(np.random.PCG64(s_small))
    B, K, V, r, d = w.B, w.K, w.V, w.r, w.d
    K1 = K + 1

    true_tok = rng.integers(0, V, size=(B, K1), dtype=np.int64)
    anchor = rng.integers(0, V, size=B, dtype=np.int64).astype(np.int32)
    lo, hi = w.sigma_b
    sigma_b = rng.uniform(lo, hi, size=B).astype(np.float32) if hi > lo else np.full(B, lo, np.float32)
    lo, hi = w.sts
    sts = rng.uniform(lo, hi, size=K).astype(np.float32) if hi > lo else np.full(K, lo, np.float32)
    temps = np.asarray(w.temps, dtype=np.float32)
    temperature = temps[rng.integers(0, len(temps), size=B)] if len(temps) > 1 else np.full(B, temps[0], np.float32)
    w_h = rng.standard_normal(d).astype(np.float32) / np.float32(np.sqrt(d))
    w_e = rng.standard_normal(r).astype(np.float32) / np.float32(np.sqrt(d))
    bump = np.maximum(0.0, w.bump0 - w.bump_decay * np.arange(K1)).astype(np.float32)

    conv = to_bf16_bits if w.bf16 else (lambda a: np.ascontiguousarray(a, dtype=np.float32))
    ldt = np.uint16 if w.bf16 else np.float32
    base = np.empty((B, K, V), dtype=ldt)
    target = np.empty((B, K1, V), dtype=ldt)
    row_seeds = s_rows.spawn(B)

    def fill(b):
        sz, sn = row_seeds[b].spawn(2)
        z = _normal(sz, (K1, V), w.sigma_z)
        z[np.arange(K1), true_tok[b]] += bump
        t = z + _normal(sn, (K1, V), sigma_b[b])
        base[b] = conv(z[:K])
        target[b] = conv(t)

    nthreads = threads or min(16, os.cpu_count() or 1)
    with ThreadPoolExecutor(nthreads) as ex:
        list(ex.map(fill, range(B)))

    def big(seedseq, shape, scale, parts):
        out = np.empty(shape, dtype=ldt)
        flat = out.reshape(-1)
        n = flat.size
        step = -(-n // parts)
        seeds = seedseq.spawn(parts)

        def part(i):
            a, e = i * step, min(n, (i + 1) * step)
            if a < e:
                flat[a:e] = conv(_normal(seeds[i], (e - a,), scale))
        with ThreadPoolExecutor(nthreads) as ex:
            list(ex.map(part, range(parts)))
        return out

    E = big(s_E, (V, r), 1.0 / np.sqrt(r), 16)
    P = big(s_P, (r, V), 1.0 / np.sqrt(r), 16)
    h = big(s_h, (B, K, d), 1.0, 16)
    if w.bf16:
        w_h = to_bf16_bits(w_h)
        w_e = to_bf16_bits(w_e)
    return {
        "workload": w.name, "B": B, "K": K, "V": V, "r": r, "d": d, "bf16": w.bf16,
        "base_logits": base, "target_logits": target, "E": E, "P": P,
        "anchor": anchor, "temperature": temperature, "h": h, "w_h": w_h, "w_e": w_e,
        "conf_bias": float(w.conf_bias), "sts_temp": sts,
        "sps": _sps_table(w.sps_kind, w.sps_nmax), "true_tokens": true_tok, "sigma_b": sigma_b,
    }


def make_sts_inputs(N, K, seed=7, t_true=(1.2, 2.5), noise=0.25):
    """Synthetic calibration set for the STS fit (float32, deterministic in the seed).

    Raw confidence logits a[n, k] ~ N(2 - 0.1 k, 1.5^2). The soft per-step
    acceptance labels follow a logistic law in a / T_true[k] with N(0, noise^2)
    jitter, T_true[k] ~ U[t_true]: with T_true > 1 the raw confidences are
    over-confident, the situation the calibration exists to correct.
    """
    ss = np.random.SeedSequence(seed)
    rng = np.random.Generator(np.random.PCG64(ss))
    k = np.arange(K, dtype=np.float32)
    a = (2.0 - 0.1 * k)[None, :] + rng.standard_normal((N, K), dtype=np.float32) * np.float32(1.5)
    lo, hi = t_true
    T = rng.uniform(lo, hi, size=K).astype(np.float32)
    jitter = rng.standard_normal((N, K), dtype=np.float32) * np.float32(noise)
    x = (a / T[None, :] + jitter).astype(np.float64)
    y = np.where(x >= 0, 1.0 / (1.0 + np.exp(-np.abs(x))), np.exp(-np.abs(x)) / (1.0 + np.exp(-np.abs(x))))
    return {"logits": np.ascontiguousarray(a, dtype=np.float32),
            "labels": np.ascontiguousarray(y, dtype=np.float32), "t_true": T}


def sts_grid(lo=0.05, hi=5.0, n=256):
    """Candidate STS temperatures: n log-spaced float32 values in [lo, hi]."""
    return np.geomspace(lo, hi, n).astype(np.float32)


def make_rnn_weights(r, d, seed=11, bf16=True):
    """Random weights of the RNN head's gated update (deterministic in the seed).

    W_ih [3r, r + d]: embedding columns ~ N(0, 1), hidden columns ~ N(0, 1/d);
    W_hh [3r, r] ~ N(0, 4/r); biases ~ N(0, 0.1^2) (float32). The scales put
    the gate pre-activations at O(1) for the embeddings and hidden states of
    the workloads above. Weights are bfloat16 bit patterns when ``bf16``.
    """
    ss = np.random.SeedSequence(seed)
    rng = np.random.Generator(np.random.PCG64(ss))
    w_ih = np.empty((3 * r, r + d), dtype=np.float32)
    w_ih[:, :r] = rng.standard_normal((3 * r, r), dtype=np.float32)
    w_ih[:, r:] = rng.standard_normal((3 * r, d), dtype=np.float32) / np.float32(np.sqrt(d))
    w_hh = rng.standard_normal((3 * r, r), dtype=np.float32) * np.float32(2.0 / np.sqrt(r))
    b_ih = (rng.standard_normal(3 * r, dtype=np.float32) * np.float32(0.1)).astype(np.float32)
    b_hh = (rng.standard_normal(3 * r, dtype=np.float32) * np.float32(0.1)).astype(np.float32)
    conv = to_bf16_bits if bf16 else (lambda a: a)
    return {"w_ih": conv(w_ih), "w_hh": conv(w_hh), "b_ih": b_ih, "b_hh": b_hh}
