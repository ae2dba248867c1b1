"""Write tests/golden/oracle_tiny_rows.json from the oracle (and nothing else).

Run from the repository root: ``python tests/golden/make_golden.py``.
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import oracle  # noqa: E402
from hybrid_sliding_window_02_b300 import inputs as gen  # noqa: E402

ROWS = [[0, h, i] for h in range(4) for i in (0, 1, 126, 127, 128, 300, 511)]


def main():
    x = gen.prefill_inputs(1, 512, 4, 1, 64, seed=0, dtype=torch.float32)
    o, l = oracle.swa_sink_fwd_rows(x.q, x.k, x.v, x.sink, 128, ROWS)
    doc = {
        "workload": "tiny fp32: B=1 T=512 Hq=4 Hkv=1 D=64 W=128, inputs from "
                    "hybrid_sliding_window_02_b300.inputs.prefill_inputs(seed=0, float32)",
        "written_by": "tests/golden/make_golden.py (oracle only)",
        "rows": ROWS,
        "out_first8": [[float(v) for v in r[:8]] for r in o],
        "out_sum": [float(r.sum()) for r in o],
        "lse": [float(v) for v in l],
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_tiny_rows.json")
    with open(path, "w") as f:
        json.dump(doc, f, indent=1)
    print("wrote", path)


if __name__ == "__main__":
    main()
