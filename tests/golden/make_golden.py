"""Writes tests/golden/tiny_oracle.json: sampled outputs of the fp64 oracle on
the seeded tiny workload (T=256, d=512, E=16, inter=128, top-6, 12 x 256
latent routing).  Calls only oracle/ and the seeded input generator (which
holds none of the layer's arithmetic); no value here comes from the CUDA
path.  Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import pathlib
import sys

import numpy as np

ROOT = pathlib.Path(__file__).resolve().parents[2]
sys.path.insert(0, str(ROOT))

import moe_inputs as mi  # noqa: E402
from oracle import moe_oracle as O  # noqa: E402

TOKENS = [0, 1, 2, 3, 17, 100, 200, 255]   # sampled token rows
COLS = 64                                   # leading output columns stored per sampled token


def main():
    inp = mi.make_inputs("tiny")
    cfg = inp["cfg"]
    r = O.forward_bits(inp)
    s = np.sort(r["logits"], axis=1)[:, ::-1]
    gap = s[:, cfg.top_k - 1] - s[:, cfg.top_k]           # k-th minus (k+1)-th logit
    doc = {
        "about": "fp64 oracle outputs of the seeded tiny workload, written by tests/golden/make_golden.py "
                 "(oracle/ and the seeded input generator only)",
        "workload": cfg.note,
        "dims": dict(T=cfg.T, d=cfg.d, E=cfg.E, inter=cfg.inter, top_k=cfg.top_k, n_heads=cfg.n_heads,
                     head_dim=cfg.head_dim),
        "offsets": [int(v) for v in r["offsets"]],
        "tokens": TOKENS,
        "topk_idx": [[int(v) for v in r["topk_idx"][t]] for t in TOKENS],
        "topk_gap": [float(gap[t]) for t in TOKENS],
        "gates": [[float(v) for v in r["gates"][t]] for t in TOKENS],
        "out_cols": COLS,
        "out": [[float(v) for v in r["out"][t, :COLS]] for t in TOKENS],
    }
    path = ROOT / "tests" / "golden" / "tiny_oracle.json"
    path.write_text(json.dumps(doc, indent=1) + "\n")
    print(path)


if __name__ == "__main__":
    main()
