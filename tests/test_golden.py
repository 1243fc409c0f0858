"""The oracle still reproduces the values stored in tests/golden (regression record).

The stored values were written by tests/golden/make_golden.py, which calls only the oracle."""
import json
import os

import numpy as np

import fa_inputs
import oracle

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_tiny_golden_reproduced(oracle_lib):
    rec = json.load(open(os.path.join(HERE, "tiny_gqa_d64.json")))
    w = fa_inputs.BY_NAME[rec["workload"]]
    q, k, v, do = fa_inputs.make_inputs(w).widened()
    o, lse = oracle.fwd(q, k, v, None, scale=w.scale, causal=w.causal)
    dq, dk, dv = oracle.bwd(q, k, v, None, do, scale=w.scale, causal=w.causal)
    d = w.head_dim
    np.testing.assert_allclose(lse.reshape(-1), rec["L"], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(o.reshape(-1, d)[rec["rows"]], rec["O"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dq.reshape(-1, d)[rec["rows"]], rec["dQ"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dk[0, 0, rec["kv_rows"]], rec["dK"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dv[0, 0, rec["kv_rows"]], rec["dV"], rtol=1e-12, atol=1e-13)
