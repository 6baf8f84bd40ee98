"""One speculative cycle: draft, confidence + schedule, verify (test infrastructure only).

Composition of the oracle's stages in the order the DSpark summary page gives
(방법론: semi-autoregressive drafting, then confidence-scheduled verification).
"""

from .draft import draft_block
from .confidence import confidence, survival
from .schedule import schedule, SCHED_GREEDY_EARLYSTOP
from .verify import verify


def cycle(inp, seed, mode=SCHED_GREEDY_EARLYSTOP, threshold=0.0):
    """Run the whole cycle on one input dict (see the workload generator's keys).

    Keys used: base_logits [B,K,V], target_logits [B,K+1,V], E, P, anchor,
    temperature, h, w_h, w_e, conf_bias, sts_temp, sps.
    """
    d = draft_block(inp["base_logits"], inp["E"], inp["P"], inp["anchor"],
                    inp["temperature"], seed)
    c = confidence(inp["h"], inp["E"], inp["anchor"], d["tokens"], inp["w_h"],
                   inp["w_e"], inp["conf_bias"], inp["sts_temp"])
    s = survival(c)
    sch = schedule(s, inp["sps"], mode=mode, threshold=threshold)
    v = verify(inp["target_logits"], inp["base_logits"], inp["E"], inp["P"], inp["anchor"],
               d["tokens"], sch["L"], inp["temperature"], seed)
    return {"draft": d, "conf": c, "survival": s, "schedule": sch, "verify": v}
