"""Writes tests/golden/tiny_call.json from the oracle alone.

The workload is the tiny single call: M=1, H=256, C=4 (wide 1024),
hc_lowrank=32, seed 0, inputs from the seeded generators; the formulas are
those of families/qwen4/mod.rs ("## Hyper-connections", the decoder-layer
inject-add) as the oracle implements them. The fixture is a regression record
of the oracle (floats stored as hex), not a value printed on the pages: the
pages print no worked example.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from hyper_connection_residual_call_gb300 import inputs  # noqa: E402


def compute():
    s = inputs.TINY
    seed = inputs.SEEDS["tiny"]
    wts = inputs.make_hc_weights(s.H, s.C, s.L, seed)
    raw = inputs.make_residual(s.M, s.H, s.C, seed)
    out = inputs.make_sublayer_out(s.M, s.H, seed)
    orc = oracle.get()
    r = orc.hc_call(raw, wts.g, wts.down, wts.up, wts.inject, H=s.H, C=s.C, L=s.L, threads=1)
    raw2 = orc.inject_add(raw, out, r["gate"], H=s.H, C=s.C)
    return {"mixed": r["mixed"], "gate": r["gate"], "inv_rms": r["inv_rms"], "a": r["a"],
            "raw_after_inject": raw2}


def main():
    res = compute()
    doc = {"workload": "tiny single call: M=1, H=256, C=4, hc_lowrank=32, seed 0",
           "source": "oracle/hc_oracle.c via tests/golden/make_golden.py",
           "values": {k: [float(x).hex() for x in v.reshape(-1)] for k, v in res.items()}}
    with open(os.path.join(HERE, "tiny_call.json"), "w") as f:
        json.dump(doc, f, indent=0)


if __name__ == "__main__":
    main()
