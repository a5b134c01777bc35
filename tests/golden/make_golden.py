"""Write tests/golden/oracle_regression.json from the CPU oracle alone.

Each entry names a small seeded workload (inputs come from
swiglu_rmsnorm_add_gb300.synthetic) and stores the SHA-256 of the oracle's
output bytes, so any later change to the oracle's arithmetic shows up as a
failing regression test. Run from the repository root:

    python tests/golden/make_golden.py
"""
import hashlib
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import oracle  # noqa: E402
from swiglu_rmsnorm_add_gb300 import synthetic  # noqa: E402

DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def digest(*ts):
    h = hashlib.sha256()
    for t in ts:
        h.update(t.contiguous().view(torch.uint8).numpy().tobytes())
    return h.hexdigest()


def cases():
    out = []
    for dt in DT:
        x, w = synthetic.rms_inputs(4, 1536, DT[dt], 1000)
        o = torch.empty_like(x)
        oracle.rmsnorm(x, w, o, synthetic.EPS)
        out.append({"op": "rmsnorm", "rows": 4, "D": 1536, "dtype": dt, "seed": 1000,
                    "sha256": digest(o)})
        x, r, w = synthetic.add_rms_inputs(16, 1536, DT[dt], 1001)
        o = torch.empty_like(x)
        oracle.add_rmsnorm(x, r, w, o, synthetic.EPS)
        out.append({"op": "add_rmsnorm", "rows": 16, "D": 1536, "dtype": dt, "seed": 1001,
                    "sha256": digest(x, o)})
        gu = synthetic.glu_inputs(2, 1024, DT[dt], 1003)
        for act in ("silu", "relu"):
            o = torch.empty(2, 1024, dtype=DT[dt])
            oracle.glu(gu, o, act)
            out.append({"op": act, "T": 2, "I": 1024, "dtype": dt, "seed": 1003, "sha256": digest(o)})
    inp = synthetic.rope_inputs(64, 1002, num_blocks=64)
    n = oracle.rope_kv_store(inp["q"], inp["k"], inp["v"], inp["cos"], inp["sin"], inp["pos"],
                             inp["slot_mapping"], inp["kv_cache"])
    out.append({"op": "rope_kv_store", "T": 64, "num_blocks": 64, "dtype": "bf16", "seed": 1002,
                "errors": n, "sha256": digest(inp["q"], inp["kv_cache"])})
    return out


if __name__ == "__main__":
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_regression.json")
    with open(path, "w") as f:
        json.dump({"_about": "SHA-256 of oracle outputs on seeded inputs; written by make_golden.py",
                   "cases": cases()}, f, indent=1)
    print("wrote", path)
