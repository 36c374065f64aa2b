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
