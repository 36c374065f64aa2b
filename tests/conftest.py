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


def oracle_rows(blk, rows, ksel=0, top_p=0.0):
    """The oracle's block output for each token in `rows`, one unchanged oracle.moe_forward
    call per token, spread over the host cores with threads (the oracle is C behind ctypes,
    which releases the GIL, and it keeps no state between calls). Returns {t: (out, idx, w)}."""
    import concurrent.futures as cf
    import oracle

    def one(t):
        ro, ri, rw, _ = oracle.moe_forward(blk, x=blk["x"][t:t + 1], ksel=ksel, top_p=top_p)
        return t, (ro[0], ri[0], rw[0])

    rows = list(rows)
    if len(rows) <= 2:
        return dict(one(t) for t in rows)
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(rows), os.cpu_count() or 1))) as ex:
        return dict(ex.map(one, rows))


def heavy_tail_x(rng, T, H, n_out=3, lo=100.0, hi=1000.0):
    """x ~ N(0, 1) with n_out entries per row replaced by +-U(lo, hi): activations whose
    largest entries are 100-1000 times their rms."""
    x = rng.standard_normal((T, H)).astype(np.float32)
    for t in range(T):
        pos = rng.choice(H, size=n_out, replace=False)
        x[t, pos] = (rng.uniform(lo, hi, n_out) * rng.choice([-1.0, 1.0], n_out)).astype(np.float32)
    return x


def with_heavy_tails(blk, seed, K, max_redraws=1000):
    """A copy of blk whose x is heavy-tailed (heavy_tail_x); rows are redrawn until every
    token passes gap_filter(K)."""
    rng = np.random.default_rng(seed)
    T, H = blk["x"].shape
    x = heavy_tail_x(rng, T, H)
    ok = gap_filter(K)
    for _ in range(max_redraws):
        good = ok(x, blk["Wr"], blk["bias"])
        if good.all():
            return dict(blk, x=x)
        bad = np.nonzero(~good)[0]
        x[bad] = heavy_tail_x(rng, len(bad), H)
    raise RuntimeError("with_heavy_tails: no rows pass the gap filter")


def plant_tie(blk, K, places, seed, b_off=None, gap=GAP, tries=200):
    """A copy of blk with an exact router tie between experts a < b: b's router row and bias
    are copies of a's, so the two choices are bitwise equal on any summation order that treats
    both rows alike. Token t's x is then moved along W_r[a] until exactly places[t] other
    experts beat a (a is pick places[t], b would be the next pick), with every other
    consecutive gap among the K + 2 best choices above `gap`. b = a + b_off (default E // 4).
    Returns (blk, a, b)."""
    import oracle
    cfg = blk["cfg"]
    E, H = cfg["E"], cfg["H"]
    a = E // 3
    b = min(E - 1, a + (max(1, E // 4) if b_off is None else b_off))
    assert b > a
    Wr = blk["Wr"].copy()
    bias = blk["bias"].copy()
    Wr[b] = Wr[a]
    bias[b] = bias[a]
    rng = np.random.default_rng(seed)
    T = blk["x"].shape[0]
    x = blk["x"].copy()
    others = np.array([e for e in range(E) if e not in (a, b)])
    alphas = np.linspace(-12.0, 12.0, 2401)
    W64, b64 = Wr.astype(np.float64), bias.astype(np.float64)
    d = W64 @ W64[a]
    for t in range(T):
        want = int(places[t])
        for _ in range(tries):
            L = (W64 @ x[t].astype(np.float64))[None, :] + alphas[:, None] * d[None, :]
            c = 1.0 / (1.0 + np.exp(-L)) + b64[None, :]
            above = (c[:, others] > c[:, [a]]).sum(axis=1)
            cand = np.nonzero(above == want)[0]
            if len(cand):
                # the alpha whose nearest competitor of a is farthest away
                marg = np.min(np.abs(c[cand][:, others] - c[cand][:, [a]]), axis=1)
                xt = (x[t] + alphas[cand[np.argmax(marg)]] * Wr[a]).astype(np.float32)
                _, ch = oracle.router(xt[None, :], Wr, bias)
                ch = ch[0]
                order = sorted(range(E), key=lambda e: (-float(ch[e]), e))[:K + 2]
                top = ch[order].astype(np.float64)
                pair = order.index(a)
                gaps = -np.diff(top)
                if (order[pair] == a and pair + 1 < len(order) and order[pair + 1] == b and pair == want
                        and gaps[pair] == 0.0 and np.all(np.delete(gaps, pair) > gap)):
                    x[t] = xt
                    break
            x[t] = rng.standard_normal(H).astype(np.float32)
        else:
            raise RuntimeError(f"plant_tie: token {t} found no place {want}")
    return dict(blk, x=x, Wr=Wr, bias=bias), a, b


def tail_inputs(blk, seed, K, scale=3.0, max_redraws=1000):
    """Inputs of the layer tail for blk's shapes: a residual row per token (N(0, scale^2)) and a
    norm weight ~ U(0.5, 1.5); rows are redrawn until the normalised rows pass gap_filter(K).
    Returns (resid, norm_w, eps)."""
    import oracle
    rng = np.random.default_rng(seed)
    T, H = blk["x"].shape
    eps = 1e-5
    w = rng.uniform(0.5, 1.5, H).astype(np.float32)
    resid = (rng.standard_normal((T, H)) * scale).astype(np.float32)
    ok = gap_filter(K)
    for _ in range(max_redraws):
        good = ok(oracle.rmsnorm(resid, w, eps), blk["Wr"], blk["bias"])
        if good.all():
            return resid, w, eps
        bad = np.nonzero(~good)[0]
        resid[bad] = (rng.standard_normal((len(bad), H)) * scale).astype(np.float32)
    raise RuntimeError("tail_inputs: no rows pass the gap filter")
