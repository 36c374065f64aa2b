import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")

# Margin demanded between consecutive router choices among the K+1 best of every token, so that
# fp32 summation-order differences cannot change the selected set or its order.
GAP = 1e-5


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line


def gap_filter(K, gap=GAP):
    """Row filter for synth.make_block: accept a token when its K+1 largest router choices
    (computed by the oracle) are separated by more than `gap`."""
    import oracle

    def ok(x, Wr, bias):
        _, ch = oracle.router(x, Wr, bias)
        top = -np.sort(-ch, axis=1)[:, :K + 1].astype(np.float64)
        if top.shape[1] < 2:
            return np.ones(x.shape[0], bool)
        return (np.diff(-top, axis=1) > gap).all(axis=1)

    return ok


def top_p_filter(K, ksel, top_p, gap=GAP):
    """Row filter for top-p cases: besides the choice margin, the selected experts' sigmoid
    scores must be pairwise separated, and no running sum of the sorted scores may sit within
    `gap` of top_p * total — so fp32 summation order cannot change the kept prefix."""
    import oracle
    choice_ok = gap_filter(K, gap)

    def ok(x, Wr, bias):
        good = choice_ok(x, Wr, bias)
        sig, ch = oracle.router(x, Wr, bias)
        idx, _, _ = oracle.select(sig, ch, K, 0, 1.0, ksel, 0.0)
        for t in range(x.shape[0]):
            sel = idx[t][idx[t] >= 0]
            s = np.sort(sig[t, sel].astype(np.float64))[::-1]
            if len(s) > 1 and np.min(-np.diff(s)) <= gap:
                good[t] = False
            cum = np.cumsum(s)
            if np.min(np.abs(cum - top_p * cum[-1])) <= gap:
                good[t] = False
        return good

    return ok
