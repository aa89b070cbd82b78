"""Write the oracle regression fixtures in this folder.

The pages print no worked numeric example, so every stored value here comes from the
float64 oracle (``oracle/``) on seeded inputs from the package's input generator; the
oracle itself is pinned by tests/test_oracle_pins.py.  These fixtures only guard against
later, unintended changes to the oracle's arithmetic.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from programming_flashattention_fwd_gb300.inputs import WORKLOADS, make_qkv, sample_rows  # noqa: E402

CASES = [
    # name, workload, overrides, number of sampled rows
    ("mha_s128_d64_bf16", "mha_b1_h2_s128_d64", {}, 12),
    ("mha_s128_d64_bf16_causal", "mha_b1_h2_s128_d64", {"causal": True}, 12),
    ("gqa_s200_d128_fp16_causal", "mha_b1_h2_s128_d64",
     {"Hq": 4, "Hkv": 2, "Sq": 200, "Sk": 200, "D": 128, "dtype": "fp16", "causal": True,
      "q_std": 2.0, "k_std": 2.0}, 12),
]


def main():
    out = {}
    for name, wname, over, n in CASES:
        w = WORKLOADS[wname].with_(**over)
        q, k, v = make_qkv(w)
        rows = sample_rows(w, n=n)
        o, lse = oracle.rows(q, k, v, w.is_fp16, w.causal, w.softmax_scale, rows)
        out[name] = {
            "workload": wname, "overrides": over, "n_sample": n,
            "rows": rows.tolist(),
            "o_first4": [[float(x) for x in r[:4]] for r in o],
            "o_rowsum": [float(x) for x in o.sum(axis=1)],
            "lse": [float(x) for x in lse],
        }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_regression.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
