"""Writes tests/golden/tiny_layer_m4_seed0.json: the oracle's results for the
tiny decode layer (H=512, 16 routed experts, top-4, I = I_s = 256, M = 4
tie-free tokens, seed 0).

The pages print no worked example with numbers, so this fixture holds no
value from them: it is a record of the oracle itself, written by this script
(which calls only the oracle and the seeded input generators).  The test that
reads it (tests/test_golden.py) makes any change to the oracle's arithmetic
show up as a failing comparison; the oracle's correctness is pinned
elsewhere (tests/test_oracle.py), against the format definitions, brute
force, closed forms and library routines.

Usage, from the repository root:  python -m tests.golden.make_golden
"""

from __future__ import annotations

import json
import os

import numpy as np

from moe_decode_layer_bf16_gb300 import synth
from moe_decode_layer_bf16_gb300.dims import TINY
from oracle import moe_oracle as orc
from tests.fixtures_moe import oracle_layer, tie_free_tokens, to_np

HERE = os.path.dirname(os.path.abspath(__file__))
PATH = os.path.join(HERE, "tiny_layer_m4_seed0.json")
M, SEED = 4, 0
COLS = list(range(0, TINY.hidden, 37))  # sampled output columns


def compute() -> dict:
    lw = synth.make_layer(TINY, seed=SEED)
    x, res, redrawn = tie_free_tokens(TINY, lw, M, seed=SEED)
    r = orc.moe_decode_layer(oracle_layer(TINY, lw), to_np(x), to_np(res))
    out, ro = np.asarray(r["out"]), np.asarray(r["residual_out"])
    return {
        "what": "oracle results, tiny decode layer (H=512, E=16, top-4, I=Is=256), M=4 tie-free tokens, seed 0",
        "redrawn_tokens": int(redrawn),
        "topk_ids": np.asarray(r["ids"]).astype(int).tolist(),
        "topk_weights": [[float(v) for v in row] for row in np.asarray(r["weights"])],
        "sorted_routes": np.asarray(r["sorted_routes"]).astype(int).tolist(),
        "expert_offsets": np.asarray(r["offsets"]).astype(int).tolist(),
        "columns": COLS,
        "out": [[float(out[t, c]) for c in COLS] for t in range(M)],
        "residual_out": [[float(ro[t, c]) for c in COLS] for t in range(M)],
        "out_row_sum": [float(v) for v in out.sum(axis=1)],
        "out_row_sumsq": [float(v) for v in (out * out).sum(axis=1)],
        "residual_out_row_sum": [float(v) for v in ro.sum(axis=1)],
    }


if __name__ == "__main__":
    with open(PATH, "w") as f:
        json.dump(compute(), f, indent=1)
        f.write("\n")
    print(PATH)
