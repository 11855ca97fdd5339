"""Writes tests/golden/tiny_oracle_digests.txt from the oracle alone.

The digests pin the oracle's encoding of the tiny Wgrad workload (dY [256,128]
N(0,1e-3^2), X [256,256] N(0,1) with 2 outlier channels x20, seed 0) across
machines and across later edits: any change to them must come with a commit
message naming the passage (or reading of it) that justifies the change.
Run: python tests/golden/make_golden.py
"""
import hashlib
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from workloads import config_inputs  # noqa: E402

MODES = [  # (label, rot, rot_block, rnd, seed)
    ("none_rne", oracle.ROT_NONE, 32, oracle.ROUND_RNE, 0),
    ("det16_rne", oracle.ROT_HADAMARD_DET, 16, oracle.ROUND_RNE, 0),
    ("det32_rne", oracle.ROT_HADAMARD_DET, 32, oracle.ROUND_RNE, 0),
    ("det256_rne", oracle.ROT_HADAMARD_DET, 256, oracle.ROUND_RNE, 0),
    ("rand32_rne", oracle.ROT_HADAMARD_RAND, 32, oracle.ROUND_RNE, 1),
    ("none_sr", oracle.ROT_NONE, 32, oracle.ROUND_SR, 1),
]


def digests():
    d = config_inputs("tiny", seed=0)
    out = []
    out.append(("input_dY", hashlib.sha256(d["dY"].tobytes()).hexdigest()))
    out.append(("input_X", hashlib.sha256(d["X"].tobytes()).hexdigest()))
    for label, rot, nb, rnd, seed in MODES:
        for name, tag in (("dY", 1), ("X", 2)):
            c, s = oracle.quantize(d[name], oracle.CONTRACT_ROWS, rot, nb, rnd, seed, tag)
            h = hashlib.sha256(c.tobytes() + s.tobytes()).hexdigest()
            out.append((f"{label}_{name}", h))
    return out


if __name__ == "__main__":
    path = os.path.join(HERE, "tiny_oracle_digests.txt")
    with open(path, "w") as f:
        f.write("# sha256 of oracle codes||scales, tiny Wgrad workload; "
                "written by tests/golden/make_golden.py\n")
        for k, v in digests():
            f.write(f"{k} {v}\n")
    print("wrote", path)
