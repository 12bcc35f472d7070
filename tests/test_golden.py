"""The oracle against its frozen record (tests/golden/oracle_small.txt).

The pages print no attention outputs and no worked example, so the record
pins nothing to them: it pins the oracle to itself, so that a change to its
arithmetic (a reordered sum, a changed decode or mask) shows up here and has
to be justified. The tolerance (1e-12 relative) absorbs last-place
differences between C libraries' exp / log on different hosts.
"""
import os
import sys

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))

import make_golden  # noqa: E402


def _record():
    out = {}
    with open(os.path.join(HERE, "golden", "oracle_small.txt")) as fh:
        for line in fh:
            if line.startswith("#") or not line.strip():
                continue
            parts = line.split()
            case, arr, n = parts[0], parts[1], int(parts[2])
            vals = np.array([float(x) for x in parts[3:]], dtype=np.float64)
            assert vals.size == n, (case, arr)
            out[(case, arr)] = vals
    return out


def test_record_covers_every_case():
    rec = _record()
    assert {c[0] for c in make_golden.CASES} == {k[0] for k in rec}


@pytest.mark.parametrize("case", make_golden.CASES, ids=[c[0] for c in make_golden.CASES])
def test_oracle_reproduces_its_record(oracle_mod, case):
    rec = _record()
    for arr, vals in make_golden.case_arrays(oracle_mod, *case):
        want = rec[(case[0], arr)]
        assert vals.shape == want.shape, (case[0], arr)
        assert np.all(np.abs(vals - want) <= 1e-12 * np.abs(want) + 1e-15), (case[0], arr)


def test_record_closed_form_row_zero():
    """Causal row 0 sees only key 0: its output is v_0 and, in the backward,
    dS_00 = P_00 (dO_0.v_0 - dO_0.O_0) = 0, so dQ_0 is exactly zero."""
    rec = _record()
    assert np.all(rec[("bwd_fp16_causal", "DQ")][:64] == 0.0)
