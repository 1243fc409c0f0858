"""Writes tests/golden/tiny_gqa_d64.json: oracle values for the tiny GQA workload.

Calls only `oracle/` and the seeded input module. The pages print no worked numeric example
for attention, so the stored values here are the oracle's own, kept as a regression record:
`tests/test_golden.py` checks that the oracle still reproduces them, and the GPU parity
tests may compare against them as well.

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import fa_inputs  # noqa: E402
import oracle  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_gqa_d64.json")
ROWS = [0, 1, 2, 31, 63, 64, 100, 127]  # flat (h*ql + i) rows of O, L, dQ
KV_ROWS = [0, 1, 17, 62, 63]


def main():
    w = fa_inputs.BY_NAME["tiny_gqa_d64"]
    inp = fa_inputs.make_inputs(w)
    q, k, v, do = inp.widened()
    o, lse = oracle.fwd(q, k, v, None, scale=w.scale, causal=w.causal, nthreads=1)
    dq, dk, dv = oracle.bwd(q, k, v, None, do, scale=w.scale, causal=w.causal, nthreads=1)
    d = w.head_dim
    rec = {
        "workload": w.name,
        "note": "oracle f64 values on the seeded inputs of fa_inputs.make_inputs; rows are flat "
                "indices into [B*H*ql] (O, L, dQ) and kv rows of kv head 0 (dK, dV)",
        "rows": ROWS,
        "kv_rows": KV_ROWS,
        "L": [float(x) for x in lse.reshape(-1)],
        "O": [[float(x) for x in o.reshape(-1, d)[r]] for r in ROWS],
        "dQ": [[float(x) for x in dq.reshape(-1, d)[r]] for r in ROWS],
        "dK": [[float(x) for x in dk[0, 0, j]] for j in KV_ROWS],
        "dV": [[float(x) for x in dv[0, 0, j]] for j in KV_ROWS],
        "sum_abs": {n: float(np.abs(a).sum()) for n, a in
                    (("O", o), ("dQ", dq), ("dK", dk), ("dV", dv))},
    }
    with open(OUT, "w") as f:
        json.dump(rec, f, indent=0)
    print("wrote", OUT)


if __name__ == "__main__":
    main()
