"""Writes the stored expected values under tests/golden/.  Calls only the oracle.

single_band_worked_example.json: a hand-checkable case with one RoPE band
(head dim 2, so omega_0 = 1 for any theta), query center 1, concentration R = 1
(no norm term), pre-RoPE keys equal to 1 at positions 0..3, current position 4,
future offsets {1, 2}, budget 2.  The test re-derives every score from the closed
form s_p = (cos(5 - p) + cos(6 - p)) / 2.
"""
import json
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))
from oracle import tri_oracle as O  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))


def single_band():
    pos = np.arange(4.0)
    k_post = np.stack([np.cos(pos), np.sin(pos)], axis=1)
    t, offs, theta, B = 4, [1, 2], 1e4, 2
    res = O.compress_unit(np.array([[1.0 + 0j]]), np.array([[1.0]]), np.array([[1.0]]),
                          k_post, np.eye(4), pos, t, offs, theta, B)
    return {
        "about": "one band (d=2), c=1, R=1, keys e^{ip} at p=0..3, t=4, offsets {1,2}, B=2; "
                 "closed form s_p = (cos(5-p)+cos(6-p))/2",
        "positions": pos.tolist(), "t": t, "offsets": offs, "theta": theta, "B": B,
        "s": res["s"][0].tolist(), "a": res["a"].tolist(), "idx": res["idx"].tolist(),
    }


if __name__ == "__main__":
    with open(os.path.join(HERE, "single_band_worked_example.json"), "w") as f:
        json.dump(single_band(), f, indent=1)
        f.write("\n")
