"""Writes tests/golden/tiny_oracle.json from the CPU oracle alone.

The stored values come only from ``oracle`` applied to the seeded ``tiny``
workload (1 query, L=4096, indexer 4x32, k=256, 8 heads of width 64).  The
input hash lets a reader on another machine check that the generator produced
the same bytes before trusting the stored outputs.

    python tests/golden/make_golden.py
"""
import hashlib
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import dsa_inputs as gen  # noqa: E402
import oracle  # noqa: E402


def input_digest(x):
    h = hashlib.sha256()
    for a in (x.q_idx, x.w_idx, x.k_idx, x.q, x.kv, x.offsets, x.row_offsets, x.row_len):
        h.update(np.ascontiguousarray(a).tobytes())
    return h.hexdigest()


def main():
    x = gen.tiny()
    scores, idx, out = oracle.decode_step(x)
    s = scores[0]
    doc = {
        "workload": "tiny: 1 query, L=4096, H_i=4, D_i=32, k=256, H_q=8, D_k=D_v=64, scale 1",
        "written_by": "tests/golden/make_golden.py (CPU oracle only)",
        "input_sha256": input_digest(x),
        "scores_int32_sha256": hashlib.sha256(s.astype(np.int32).tobytes()).hexdigest(),
        "scores_zero_count": int((s == 0).sum()),
        "idx": idx[0].tolist(),
        "out": [float(v) for v in out[0].reshape(-1)],
    }
    with open(os.path.join(ROOT, "tests", "golden", "tiny_oracle.json"), "w") as f:
        json.dump(doc, f, indent=0)


if __name__ == "__main__":
    main()
