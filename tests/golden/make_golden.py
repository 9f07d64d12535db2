"""Write the stored oracle fixtures of tests/golden/.

Calls only oracle/ (and synth/ for the seeded inputs).  The pages print no worked example,
so these fixtures pin the oracle against unintended change, not against the pages:
routing and three output rows of the tiny fp32 layer (T=128, d=64, f=256, E=4, top-1,
capacity factor 1.0, seed 0).

Run:  python tests/golden/make_golden.py
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import synth  # noqa: E402


def main():
    cfg = synth.CONFIGS["tiny_fp32"]
    inp = synth.host_inputs(cfg, 128, seed=0)
    out, r = oracle.layer_forward(inp["tokens"], inp["Wg"], inp["W1"], inp["W2"], cfg.k, cfg.cf)
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_fp32_T128_seed0.txt")
    with open(path, "w") as fh:
        fh.write("# oracle fixture: tiny fp32 MoE layer T=128 d=64 f=256 E=4 top-1 cf=1.0, seed 0\n")
        fh.write("# written by tests/golden/make_golden.py (oracle/ + synth/ only)\n")
        fh.write("topk_idx: " + " ".join(map(str, r.topk_idx.reshape(-1).tolist())) + "\n")
        fh.write("slot_of: " + " ".join(map(str, r.disp.slot_of.reshape(-1).tolist())) + "\n")
        fh.write("counts_raw: " + " ".join(map(str, r.disp.counts_raw.tolist())) + "\n")
        fh.write("logits_row0: " + " ".join(float(v).hex() for v in r.logits[0]) + "\n")
        fh.write("out_rows_0_1_127: " + " ".join(repr(float(v)) for v in out[[0, 1, 127]].reshape(-1)) + "\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
