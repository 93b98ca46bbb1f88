"""Write oracle_tiny_b1_l32.txt: the FP64 oracle's output for the seed-0
tiny workload (B=1, Hq 32, Hkv 8, D 128, block 16, context 32).

Calls only the oracle and the seeded input generator. Run from the
repository root:  python tests/golden/make_golden.py
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import hashlib  # noqa: E402

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from paged_gqa_decode_attention_gb300 import workloads  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_tiny_b1_l32.txt")


def input_digest(arrays) -> str:
    """sha256 over the raw bytes of (q, k, v, block_table, context_lens)."""
    h = hashlib.sha256()
    for a in arrays:
        h.update(np.ascontiguousarray(a).tobytes())
    return h.hexdigest()


def main():
    wl = workloads.tiny(seed=0)
    arrays = workloads.host_arrays(wl)
    out = oracle.paged_decode(*arrays, oracle.BF16, wl.scale, threads=1)
    with open(OUT, "w") as f:
        f.write("# FP64 oracle output out[0, hq, d] for workloads.tiny(seed=0); "
                "one row per query head, 128 values, repr of float64\n")
        f.write(f"# inputs-sha256 {input_digest(arrays)}\n")
        for hq in range(out.shape[1]):
            f.write(" ".join(repr(float(x)) for x in out[0, hq]) + "\n")


if __name__ == "__main__":
    main()
