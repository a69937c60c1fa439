"""Write tests/golden/generator_sha256.json: digests of the LCG-based workloads.

These freeze the seeded input streams (not any GEMM result); the normal
workload is left out because its values pass through the host's libm.
Run from the repository root:  python tests/golden/make_generator_hashes.py
"""
import hashlib
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

from seeded_inputs import WORKLOADS, make_workload  # noqa: E402


def main():
    out = {}
    for w in WORKLOADS:
        if w.dist == "normal":
            continue
        A, B = make_workload(w)
        out[w.name] = {
            "A": hashlib.sha256(np.ascontiguousarray(A).tobytes()).hexdigest(),
            "B": hashlib.sha256(np.ascontiguousarray(B).tobytes()).hexdigest(),
        }
    with open(os.path.join(HERE, "generator_sha256.json"), "w") as f:
        json.dump(out, f, indent=1, sort_keys=True)
        f.write("\n")


if __name__ == "__main__":
    main()
