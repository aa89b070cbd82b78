"""The oracle still produces the values recorded in tests/golden/oracle_regression.json
(written by tests/golden/make_golden.py from the oracle alone)."""
import json
import os

import numpy as np

import oracle
from programming_flashattention_fwd_gb300.inputs import WORKLOADS, make_qkv, sample_rows

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "oracle_regression.json")


def test_oracle_regression_fixtures(orc):
    with open(GOLDEN) as f:
        cases = json.load(f)
    assert cases
    for name, c in cases.items():
        w = WORKLOADS[c["workload"]].with_(**c["overrides"])
        q, k, v = make_qkv(w)
        rows = sample_rows(w, n=c["n_sample"])
        np.testing.assert_array_equal(rows, np.asarray(c["rows"], dtype=np.int64))
        o, lse = orc.rows(q, k, v, w.is_fp16, w.causal, w.softmax_scale, rows)
        np.testing.assert_allclose(o[:, :4], np.asarray(c["o_first4"]), rtol=0, atol=1e-12, err_msg=name)
        np.testing.assert_allclose(o.sum(axis=1), np.asarray(c["o_rowsum"]), rtol=0, atol=1e-11, err_msg=name)
        np.testing.assert_allclose(lse, np.asarray(c["lse"]), rtol=0, atol=1e-12, err_msg=name)
