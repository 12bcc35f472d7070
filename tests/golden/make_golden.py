"""Writes oracle_small.txt: the fp64 oracle's outputs on a few tiny seeded
cases (forward fp16 / bf16, causal or not; backward; 8-bit forward).

The pages print no attention outputs and no worked example, so nothing here
comes from them: this is a frozen record of the oracle itself, so that any
later change to its arithmetic makes tests/test_golden.py fail and has to be
justified. It calls only the oracle and the seeded input generator.

    python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

from attention_forward_flashattention_gb300 import inputs as I  # noqa: E402

# name, B, H, N, d, dtype, causal, seed index
CASES = [
    ("fwd_fp16", 1, 1, 5, 64, "fp16", False, 7001),
    ("fwd_bf16_causal", 1, 2, 3, 64, "bf16", True, 7002),
    ("bwd_fp16_causal", 1, 1, 4, 64, "fp16", True, 7003),
    ("fwd_e4m3", 1, 1, 2, 128, "e4m3", False, 7004),
]


def case_arrays(oracle, name, B, H, N, d, dtype, causal, seed):
    """The named output arrays of one case, flattened, in a fixed order."""
    w = I.custom(name, B, H, N, d, dtype, causal, seed)
    if dtype == "e4m3":
        f = I.fp8_inputs(w)
        o, lse, _ = oracle.attn_fp8(f.q, f.k, f.vt, f.q_scale, f.k_scales, f.v_scale, causal,
                                    w.scale, nthreads=1)
        return [("O", o.ravel()), ("LSE", lse.ravel())]
    q, k, v = I.qkv_bits(w)
    if name.startswith("bwd"):
        g = oracle.attn_bwd(q, k, v, I.dout_bits(w), dtype, causal, w.scale, nthreads=1)
        return [(t.upper(), g[t].ravel()) for t in ("dq", "dk", "dv")]
    o, lse = oracle.attn_fwd(q, k, v, dtype, causal, w.scale, nthreads=1)
    return [("O", o.ravel()), ("LSE", lse.ravel())]


def main():
    import oracle
    oracle.build()
    lines = ["# fp64 oracle outputs on tiny seeded cases (tests/golden/make_golden.py);",
             "# one line per array: case name, array name, count, values (17 significant digits)"]
    for c in CASES:
        for arr, vals in case_arrays(oracle, *c):
            lines.append(" ".join([c[0], arr, str(vals.size)] + [f"{x:.17g}" for x in vals]))
    with open(os.path.join(HERE, "oracle_small.txt"), "w") as fh:
        fh.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
