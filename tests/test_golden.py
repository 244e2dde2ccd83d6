"""Stored oracle values (tests/golden/, written by tests/golden/make_golden.py
from the oracle alone) against a fresh oracle run: any change to the oracle's
forward or backward arithmetic, or to the seeded inputs, fails here.  The
tolerance covers only the rounding differences between compilers and machines
(fp64, a few hundred operations per value).  CPU only."""
import os

import numpy as np
import pytest

from tests.golden import make_golden

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.mark.parametrize("stem,w,dseed", list(make_golden.cases()),
                         ids=[c[0] for c in make_golden.cases()])
def test_oracle_matches_stored_values(stem, w, dseed):
    stored = make_golden.read(os.path.join(GOLDEN, f"{stem}.txt"))
    fresh = make_golden.compute(w, dseed)
    assert set(stored) == set(fresh)
    for k, v in fresh.items():
        assert stored[k].shape == v.shape, k
        scale = max(float(np.abs(v).max()), 1e-300)
        err = float(np.abs(stored[k] - v).max()) / scale
        assert err <= 1e-12, f"{stem} {k}: {err:.3e}"
