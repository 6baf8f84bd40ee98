"""Reference oracle for draft-block sampling, confidence scheduling and verification.

TEST INFRASTRUCTURE ONLY. This package is a plain, slow, CPU implementation in
float64 (NumPy) plus a pure-Python Philox4x32-10. It exists so that the CUDA path
can be checked against something written directly from the method's statement.
Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import it. The product library
never imports, links or calls anything here, and nothing here imports the
product package: the two share no code.

Sources (cited by page title and section):
  * DSpark summary page -- "DSpark: 반자기회귀 생성과 신뢰도 기반 검증으로
    speculative decoding 가속하기": sections 배경 (background: the
    draft/verify cycle and the lossless rejection rule), 방법론 › 반자기회귀 생성
    (semi-autoregressive generation, the Markov head), 방법론 › 신뢰도 기반 검증
    (confidence head, STS, survival, hardware-aware prefix scheduler).
  * vLLM MTP/DFlash page -- "[vLLM] MTP & DFlash": section DFlashProposer 초기화
    (one bonus token plus K drafted tokens per request and cycle).
  * Philox4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
    as 1, 2, 3", SC'11.

Parity status per function (see the pins in tests/test_oracle_*.py):
  philox4x32_10, uniform ........ pinned (an independent library implementation:
                                  Triton's Philox run by its CPU interpreter)
  inverse_cdf, argmax_first ..... pinned (hand-built CDFs, brute force)
  markov_logits, draft_block .... pinned (full-rank transition matrix, the
                                  "of course / no problem" toy, exact law by
                                  enumeration)
  confidence, survival .......... pinned (closed-form sigmoid, cumprod,
                                  monotonicity, order preservation under STS)
  schedule ...................... pinned (brute force over prefix-closed
                                  selections, linear-SPS closed form,
                                  non-anticipation metamorphic test)
  verify ........................ pinned (acceptance = 1 - TV(p, q) by exact
                                  integration over u; V=8, K=3 losslessness by
                                  exhaustive enumeration)
  sts_fit, ece .................. pinned (hand-binned ECE values, one-bin closed
                                  form, exact recovery of the true temperatures
                                  with zero ECE, prefix and causality
                                  metamorphic tests, first-index ties)
  acceptance_rate ............... pinned (equals the verify rule's accept
                                  probability integrated exactly over u;
                                  p = q gives 1, disjoint supports 0; T = 0
                                  argmax agreement)
  gru_cell, rnn_draft_block ..... pinned (torch.nn.GRUCell in float64, closed
                                  forms with saturated gates, a frozen zero
                                  state drawing from the base logits alone,
                                  memory beyond the previous token, bfloat16
                                  rounding against the generator's rounding)
  cycle ......................... composition of the above
"""

from .philox import philox4x32_10, uniform, STAGE_DRAFT, STAGE_ACCEPT, STAGE_RESAMPLE
from .sampling import inverse_cdf, argmax_first, softmax_weights
from .draft import markov_logits, draft_block, draft_step
from .confidence import confidence, survival
from .schedule import (schedule, sps_at, async_budgets, SCHED_GREEDY_EARLYSTOP, SCHED_FIXED_K,
                       SCHED_THRESHOLD, SCHED_ASYNC)
from .verify import verify, verify_request
from .cycle import cycle
from .bf16 import bf16_bits_to_f64
from .sts import sts_fit, sts_curves, ece
from .rnn import gru_cell, rnn_draft_block
from .acceptance import acceptance_rate

__all__ = [
    "philox4x32_10", "uniform", "STAGE_DRAFT", "STAGE_ACCEPT", "STAGE_RESAMPLE",
    "inverse_cdf", "argmax_first", "softmax_weights",
    "markov_logits", "draft_block", "draft_step",
    "confidence", "survival",
    "schedule", "sps_at", "async_budgets", "SCHED_GREEDY_EARLYSTOP", "SCHED_FIXED_K",
    "SCHED_THRESHOLD", "SCHED_ASYNC",
    "verify", "verify_request", "cycle", "bf16_bits_to_f64",
    "sts_fit", "sts_curves", "ece", "gru_cell", "rnn_draft_block", "acceptance_rate",
]
