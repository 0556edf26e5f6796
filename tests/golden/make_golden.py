"""Writes tests/golden/config1_oracle.json from the oracle alone (synth inputs, config 1).

Run from the repo root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))
import oracle  # noqa: E402
import synth  # noqa: E402

cfg = synth.config(1)
inp = synth.prefill_inputs(cfg)
rows = []
for t in [0, 5, 63, 64, 65, 128, 200, 255]:
    r = oracle.prefill_row(inp, t, cfg.k, cfg.scale)
    rows.append(dict(t=t, idx_sorted=sorted(int(i) for i in r["idx"]),
                     o_rowsum=[float(x) for x in r["o"].sum(axis=1)], lse=[float(x) for x in r["lse"]]))
out = dict(source="oracle on synth config 1 (tiny prefill L=256, seed 0); regenerate with make_golden.py",
           rows=rows)
with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "config1_oracle.json"), "w") as f:
    json.dump(out, f, indent=1)
