"""Write tests/golden/tiny_cycle.json from the oracle alone.

Run: python tests/golden/make_golden.py
It calls only the oracle and the seeded workload generator; no value in the
output comes from the CUDA path.
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from speculative_decoding_draft_block_gb300.workloads import TINY, make_inputs  # noqa: E402

SEED = 0x5EED0000


def main():
    inp = make_inputs(TINY)
    res = oracle.cycle(inp, SEED)
    out = {
        "workload": TINY.name, "input_seed": TINY.seed, "philox_seed": SEED,
        "draft_tokens": res["draft"]["tokens"].tolist(),
        "q_token": [[float(v) for v in row] for row in res["draft"]["q_token"]],
        "conf": [[float(v) for v in row] for row in res["conf"]],
        "sched_len": res["schedule"]["L"].tolist(),
        "accept_count": res["verify"]["accept_count"].tolist(),
        "out_tokens": res["verify"]["out_tokens"].tolist(),
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_cycle.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print("wrote", path)


if __name__ == "__main__":
    main()
