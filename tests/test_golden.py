"""Hand-worked fixtures under tests/golden/ (each file states its derivation and citation)."""
import glob
import json
import os

import numpy as np
import pytest

GOLDEN = sorted(glob.glob(os.path.join(os.path.dirname(__file__), "golden", "*.json")))


@pytest.mark.parametrize("path", GOLDEN, ids=[os.path.basename(p) for p in GOLDEN])
def test_golden_delta_rule(path, oracle_mod):
    fx = json.load(open(path))
    L = len(fx["g"])
    q = np.array(fx["q"], float)[:, None, :]
    k = np.array(fx["k"], float)[:, None, :]
    v = np.array(fx["v"], float)[:, None, :]
    g = np.array(fx["g"], float)[:, None]
    beta = np.array(fx["beta"], float)[:, None]
    S0 = np.array(fx["S0"], float)[None]
    o, S, snap = oracle_mod.delta_rule(q, k, v, g, beta, S0, snapshots=True)
    tol = fx["tolerance"]
    np.testing.assert_allclose(o[:, 0], np.array(fx["o"]), rtol=0, atol=tol)
    np.testing.assert_allclose(snap[:, 0], np.array(fx["S_after"]), rtol=0, atol=tol)
    assert L == len(fx["S_after"])
