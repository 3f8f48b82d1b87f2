"""Writes the stored oracle fixtures in this folder.

Calls only the CPU oracle and the seeded input generators.  Rerun it (and
say in the commit message which passage justifies the change) only when the
oracle's arithmetic changes on purpose.

    python tests/golden/make_golden.py
"""
import hashlib
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle      # noqa: E402
import workloads   # noqa: E402


def tiny_fixture():
    wl = workloads.make("tiny", seed=0)
    res = oracle.run_workload(wl)
    return {
        "workload": "tiny S=128 H=256 E=8 K=2 bf16, uniform routing, identity experts, seed 0",
        "cnt": res["cnt"].tolist(),
        "off": res["off"].tolist(),
        "n_invalid": res["n_invalid"],
        "tok_map": res["tok_map"].reshape(-1).tolist(),
        "packed_src": res["packed_src"].tolist(),
        "sha256_packed_x": hashlib.sha256(res["packed_x"].tobytes()).hexdigest(),
        "sha256_out": hashlib.sha256(res["out"].tobytes()).hexdigest(),
    }


if __name__ == "__main__":
    with open(os.path.join(HERE, "tiny_seed0.json"), "w") as f:
        json.dump(tiny_fixture(), f, indent=None, separators=(",", ":"))
        f.write("\n")
