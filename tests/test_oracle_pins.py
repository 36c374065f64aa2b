"""Pins of the CPU oracle against facts fixed by the pages and by mathematics.

Each test checks the oracle against something other than itself: hand-worked examples from the
pages' definitions (tests/golden/), closed forms, brute force on tiny inputs, textbook special
cases computed by a library routine, and invariants. A plausible slip in the oracle — nibble
order, the -8 offset, scale before/after the sum, gate/up swapped, SiLU on the wrong operand,
tie-break direction, weights taken from the biased choice, renorm epsilon, combine weights,
shared-expert weight, bucket stability — fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from conftest import golden_lines, gap_filter

F8, F4, F2, F32, F4G = oracle.FMT_INT8, oracle.FMT_INT4, oracle.FMT_INT2, oracle.FMT_F32, oracle.FMT_INT4G


# ---------------------------------------------------------------- independent decoder (numpy)
def np_deq(fmt, W, n):
    """Dequantise a packed [O, row_bytes] matrix to float64 [O, n] with numpy bit operations —
    written separately from the oracle's per-element decoder."""
    W = np.asarray(W, dtype=np.uint8)
    if fmt == F8:
        return W[:, :n].view(np.int8).astype(np.float64)
    if fmt == F4:
        lo = (W & 0x0F).astype(np.int64) - 8
        hi = (W >> 4).astype(np.int64) - 8
        return np.stack([lo, hi], axis=2).reshape(W.shape[0], -1)[:, :n].astype(np.float64)
    if fmt == F2:
        f = [((W >> (2 * j)) & 3).astype(np.int64) - 2 for j in range(4)]
        return np.stack(f, axis=2).reshape(W.shape[0], -1)[:, :n].astype(np.float64)
    raise ValueError(fmt)


def rand_packed(rng, fmt, O, n):
    rb = oracle.row_bytes(fmt, n)
    if fmt == F8:
        return rng.integers(-128, 128, size=(O, rb), dtype=np.int8).view(np.uint8)
    return rng.integers(0, 256, size=(O, rb), dtype=np.uint8)


def ulp_close(a, b, ulps=1):
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    sp = np.spacing(np.maximum(np.abs(a), np.abs(b)).astype(np.float32))
    return np.all(np.abs(a.astype(np.float64) - b.astype(np.float64)) <= ulps * sp)


# ---------------------------------------------------------------- unpack
def test_unpack_golden():
    n_cases = 0
    for line in golden_lines("unpack.txt"):
        lhs, rhs = line.split(":")
        fmt, n, hx = lhs.split()
        fmt, n = int(fmt), int(n)
        row = np.frombuffer(bytes.fromhex(hx), dtype=np.uint8)
        expect = np.array([float(v) for v in rhs.split()], np.float32)
        got = oracle.deq_row(fmt, row, n)
        assert np.array_equal(got, expect), (line, got)
        assert np.array_equal(np_deq(fmt, row[None, :], n)[0], expect), line
        n_cases += 1
    assert n_cases >= 10


def test_row_bytes():
    # QT row strides: In, ceil(In/2), ceil(In/4) bytes, 4*In for f32
    assert [oracle.row_bytes(F8, n) for n in (1, 7, 8)] == [1, 7, 8]
    assert [oracle.row_bytes(F4, n) for n in (1, 2, 3, 6144)] == [1, 1, 2, 3072]
    assert [oracle.row_bytes(F2, n) for n in (1, 4, 5, 2048)] == [1, 1, 2, 512]
    assert oracle.row_bytes(F32, 5) == 20
    assert [oracle.row_bytes(F4G, n) for n in (1, 2, 3, 6144)] == [1, 1, 2, 3072]


# ---------------------------------------------------------------- quantised GEMV
@pytest.mark.parametrize("fmt", [F8, F4, F2])
@pytest.mark.parametrize("O,n", [(5, 13), (3, 16), (7, 1)])
def test_qgemv_unit_vectors_give_scaled_columns(fmt, O, n):
    rng = np.random.default_rng(100 + fmt * 10 + n)
    W = rand_packed(rng, fmt, O, n)
    s = rng.uniform(0.5, 2.0, O).astype(np.float32)
    D = np_deq(fmt, W, n)
    for i in range(n):
        e = np.zeros(n, np.float32)
        e[i] = 1.0
        y = oracle.qgemv(fmt, W, s, e, O, n)
        assert np.array_equal(y, (D[:, i].astype(np.float32) * s)), i


@pytest.mark.parametrize("fmt", [F8, F4, F2])
def test_qgemv_scale_multiplies_rounded_sum(fmt):
    rng = np.random.default_rng(7 + fmt)
    O, n = 9, 301
    W = rand_packed(rng, fmt, O, n)
    s = rng.uniform(1e-3, 1e-2, O).astype(np.float32)
    v = rng.standard_normal(n).astype(np.float32)
    y = oracle.qgemv(fmt, W, s, v, O, n)
    exact = np.array([math.fsum(np_deq(fmt, W, n)[o] * v.astype(np.float64)) for o in range(O)])
    expect = exact.astype(np.float32) * s  # round the sum to float once, then scale
    assert ulp_close(y, expect, 1)


@pytest.mark.parametrize("fmt", [F8, F4, F2])
def test_scale_one_int_path_equals_float_path(fmt):
    # With all scales 1 the quantised path equals the f32 path on the dequantised weights.
    rng = np.random.default_rng(11 + fmt)
    O, n = 17, 257
    W = rand_packed(rng, fmt, O, n)
    Wf = np_deq(fmt, W, n).astype(np.float32)
    v = rng.standard_normal(n).astype(np.float32)
    y_int = oracle.qgemv(fmt, W, np.ones(O, np.float32), v, O, n)
    y_f32 = oracle.qgemv(F32, Wf.view(np.uint8), None, v, O, n)
    assert np.array_equal(y_int, y_f32)


# ---------------------------------------------------------------- int4-grouped GEMV (format 4)
def np_group_scales(s, O, n, gs):
    """[O, n] float64 matrix of the scale that applies to each weight: s[o, i // gs]."""
    ng = (n + gs - 1) // gs
    return np.repeat(np.asarray(s, np.float64).reshape(O, ng), gs, axis=1)[:, :n]


@pytest.mark.parametrize("O,n,gs", [(4, 96, 32), (3, 100, 32), (5, 64, 128)])
def test_grouped_unit_vectors_pick_the_group_scale(O, n, gs):
    # e_i selects column i: y[o] = deq(W[o,i]) * s[o, i // gs] — the scale of row o's group of i
    # (a transposed [ng][O] scale layout or a wrong group index fails here)
    rng = np.random.default_rng(500 + n + gs)
    W = rand_packed(rng, F4G, O, n)
    ng = (n + gs - 1) // gs
    s = rng.uniform(0.5, 2.0, O * ng).astype(np.float32)
    D = np_deq(F4, W, n)
    S = np_group_scales(s, O, n, gs)
    for i in range(n):
        e = np.zeros(n, np.float32)
        e[i] = 1.0
        y = oracle.qgemv_grouped(W, s, gs, e, O, n)
        assert np.array_equal(y, (D[:, i] * S[:, i]).astype(np.float32)), i


@pytest.mark.parametrize("O,n,gs", [(7, 300, 32), (5, 256, 64), (3, 96, 128), (4, 37, 1)])
def test_grouped_matches_dense_brute_force(O, n, gs):
    # the exact sum of deq * group scale * v (math.fsum over the dense float64 matrix), rounded
    # once to float: the oracle's double accumulation may differ by at most one float ulp
    rng = np.random.default_rng(600 + n + gs)
    W = rand_packed(rng, F4G, O, n)
    ng = (n + gs - 1) // gs
    s = rng.uniform(1e-3, 1e-2, O * ng).astype(np.float32)
    v = rng.standard_normal(n).astype(np.float32)
    y = oracle.qgemv_grouped(W, s, gs, v, O, n)
    dense = np_deq(F4, W, n) * np_group_scales(s, O, n, gs)
    expect = np.array([math.fsum(dense[o] * v.astype(np.float64)) for o in range(O)]).astype(np.float32)
    assert ulp_close(y, expect, 1)


def test_grouped_single_group_equals_per_row_int4():
    # gs >= In: one scale per row, i.e. the per-row int4 format (rounded once here, twice there)
    rng = np.random.default_rng(701)
    O, n = 11, 192
    W = rand_packed(rng, F4, O, n)
    s = rng.uniform(0.5, 2.0, O).astype(np.float32)
    v = rng.standard_normal(n).astype(np.float32)
    for gs in (n, 4 * n):
        assert ulp_close(oracle.qgemv_grouped(W, s, gs, v, O, n), oracle.qgemv(F4, W, s, v, O, n), 1)


# ---------------------------------------------------------------- IDOT (int8 activations)
def test_qrow_i8_hand_worked_half_even():
    # amax = 127 gives s = 1 and 1/s = 1 exactly, so q is lrintf(x): ties go to the even integer
    x = np.array([127.0, 2.5, 3.5, -2.5, -0.5, 0.5, 1.5, -126.6, 0.49], np.float32)
    q, s = oracle.qrow_i8(x)
    assert s == 1.0
    assert q.tolist() == [127, 2, 4, -2, 0, 0, 2, -127, 0]


def test_qrow_i8_extremes_and_floor():
    rng = np.random.default_rng(801)
    x = rng.standard_normal(301).astype(np.float32)
    q, s = oracle.qrow_i8(x)
    i = int(np.argmax(np.abs(x)))
    assert abs(int(q[i])) == 127 and np.sign(q[i]) == np.sign(x[i])
    assert np.all(np.abs(q.astype(np.int64)) <= 127)
    # every element within half a step (plus float rounding of x / s)
    assert np.all(np.abs(x.astype(np.float64) - q * np.float64(s)) <= 0.5 * s * (1 + 1e-6))
    # all-zero row: the scale floor 1e-12, q = 0
    q0, s0 = oracle.qrow_i8(np.zeros(7, np.float32))
    assert s0 == np.float32(1e-12) and not q0.any()
    # power-of-two scaling of x scales s exactly and leaves q unchanged
    q2, s2 = oracle.qrow_i8(x * np.float32(8.0))
    assert np.array_equal(q2, q) and s2 == np.float32(8.0) * np.float32(s)


@pytest.mark.parametrize("fmt", [F8, F4])
def test_idot_gemv_is_exact_integer_dot_then_two_products(fmt):
    # brute force with numpy's integer matmul on the independently decoded weights
    rng = np.random.default_rng(810 + fmt)
    O, n = 13, 352
    W = rand_packed(rng, fmt, O, n)
    s = rng.uniform(1e-3, 1e-2, O).astype(np.float32)
    q = rng.integers(-127, 128, n).astype(np.int8)
    sx = np.float32(0.0137)
    y = oracle.qgemv_idot(fmt, W, s, q, sx, O, n)
    dot = np_deq(fmt, W, n).astype(np.int64) @ q.astype(np.int64)
    expect = (dot.astype(np.float32) * s) * sx
    assert np.array_equal(y, expect)


@pytest.mark.parametrize("fmt", [F8, F4])
def test_idot_on_integer_activations_equals_exact_path(fmt):
    # x already on the int8 grid with max |x| = 127: s = 1, q = x, and the IDOT product equals
    # the exact path bit for bit (both round the exact integer sum once, then scale)
    rng = np.random.default_rng(820 + fmt)
    O, n = 9, 256
    W = rand_packed(rng, fmt, O, n)
    s = rng.uniform(0.5, 2.0, O).astype(np.float32)
    x = rng.integers(-126, 127, n).astype(np.float32)
    x[17] = -127.0
    q, sx = oracle.qrow_i8(x)
    assert sx == 1.0 and np.array_equal(q.astype(np.float32), x)
    assert np.array_equal(oracle.qgemv_idot(fmt, W, s, q, sx, O, n), oracle.qgemv(fmt, W, s, x, O, n))


@pytest.mark.parametrize("fmt", [F8, F4])
def test_idot_error_is_a_fraction_of_a_percent(fmt):
    # the pages state ~0.3 % RMS added error per matmul for int8 activations
    rng = np.random.default_rng(830 + fmt)
    O, n = 256, 2048
    W = rand_packed(rng, fmt, O, n)
    s = rng.uniform(0.5, 1.5, O).astype(np.float32)
    x = rng.standard_normal(n).astype(np.float32)
    q, sx = oracle.qrow_i8(x)
    y_i = oracle.qgemv_idot(fmt, W, s, q, sx, O, n).astype(np.float64)
    y_e = oracle.qgemv(fmt, W, s, x, O, n).astype(np.float64)
    rel = np.sqrt(np.mean((y_i - y_e) ** 2) / np.mean(y_e ** 2))
    assert 1e-4 < rel < 1e-2, rel


@pytest.mark.parametrize("fmt,bits", [(F8, 8), (F4, 4), (F2, 2)])
def test_pages_quantizer_roundtrip(fmt, bits):
    """Quantise float rows the way the pages' quantize_rows / pack_int4 / pack_int2 do
    (symmetric per row, s = amax/qmax, v = round-half-even(w/s) clamped, stored as v+8 in a
    nibble (low nibble first) or v+2 in a 2-bit field), then dequantise with the oracle:
    |deq*s - w| <= s/2 wherever w/s was in range."""
    rng = np.random.default_rng(5 + bits)
    O, n = 6, 37
    w = rng.standard_normal((O, n)).astype(np.float32)
    qmax = (1 << (bits - 1)) - 1
    rb = oracle.row_bytes(fmt, n)
    packed = np.zeros((O, rb), np.uint8)
    scales = np.zeros(O, np.float32)
    for o in range(O):
        s = max(np.float32(np.abs(w[o]).max()) / np.float32(qmax), np.float32(1e-8))
        scales[o] = s
        v = np.clip(np.rint(w[o] / s), -qmax - 1, qmax).astype(np.int64)
        if fmt == F8:
            packed[o, :n] = v.astype(np.int8).view(np.uint8)
        elif fmt == F4:
            for i in range(n):
                packed[o, i // 2] |= np.uint8((v[i] + 8) << (4 * (i % 2)))
        else:
            for i in range(n):
                packed[o, i // 4] |= np.uint8((v[i] + 2) << (2 * (i % 4)))
    for o in range(O):
        d = oracle.deq_row(fmt, packed[o], n) * scales[o]
        assert np.all(np.abs(d - w[o]) <= scales[o] * 0.5 * (1 + 1e-6) + 1e-12), o


# ---------------------------------------------------------------- router
def test_router_closed_form():
    rng = np.random.default_rng(3)
    T, H, E = 3, 8, 5
    x = rng.standard_normal((T, H)).astype(np.float32)
    Wr = np.zeros((E, H), np.float32)
    cols = [4, 0, 7, 2, 2]
    for e, c in enumerate(cols):
        Wr[e, c] = 2.0 ** -e  # logit = x[c] * 2^-e exactly
    bias = rng.uniform(-0.1, 0.1, E).astype(np.float32)
    sig, ch = oracle.router(x, Wr, bias)
    for t in range(T):
        for e, c in enumerate(cols):
            lg = float(x[t, c]) * 2.0 ** -e
            s = 1.0 / (1.0 + math.exp(-lg))
            assert ulp_close(sig[t, e], np.float32(s), 2)
            assert ch[t, e] == np.float32(sig[t, e] + bias[e])
    sig0, _ = oracle.router(np.zeros((1, H), np.float32), Wr, bias)
    assert np.all(sig0 == 0.5)


def test_router_rejects_non_finite():
    x = np.zeros((1, 4), np.float32)
    x[0, 1] = np.nan
    with pytest.raises(ValueError):
        oracle.router(x, np.ones((3, 4), np.float32), np.zeros(3, np.float32))


def _parse_route(line):
    parts = [p.split() for p in line.split("|")]
    K, ksel, top_p, norm, rs = parts[0]
    return (int(K), int(ksel), float(top_p), int(norm), float(rs),
            np.array(parts[1], np.float32), np.array(parts[2], np.float32),
            np.array(parts[3], np.int32), np.array(parts[4], np.float32), int(parts[5][0]))


def test_select_golden():
    n_cases = 0
    for line in golden_lines("route.txt"):
        K, ksel, top_p, norm, rs, sig, bias, eidx, ew, ekeff = _parse_route(line)
        ch = (sig + bias).astype(np.float32)
        idx, w, keff = oracle.select(sig[None], ch[None], K, norm, rs, ksel, top_p)
        assert np.array_equal(idx[0], eidx), line
        assert ulp_close(w[0], ew, 1), (line, w)
        assert keff[0] == ekeff
        n_cases += 1
    assert n_cases == 4


def _brute_topk(ch, K):
    order = sorted(range(len(ch)), key=lambda e: (-float(ch[e]), e))
    return order[:K]


@pytest.mark.parametrize("E", [1, 2, 3, 5, 8, 12, 33, 64, 256])
def test_select_matches_brute_force_sort(E):
    rng = np.random.default_rng(E)
    for trial in range(60):
        K = int(rng.integers(1, min(E, 9) + 1))
        T = 4
        if trial % 2:
            # few distinct values: many exact ties
            ch = rng.choice(np.array([0.1, 0.25, 0.5, 0.75], np.float32), size=(T, E))
            sig = ch.copy()
        else:
            sig = rng.uniform(0, 1, (T, E)).astype(np.float32)
            ch = (sig + rng.uniform(-0.1, 0.1, (T, E)).astype(np.float32)).astype(np.float32)
        idx, w, keff = oracle.select(sig, ch, K, 0, 1.0)
        for t in range(T):
            assert list(idx[t]) == _brute_topk(ch[t], K)
            assert np.array_equal(w[t], sig[t, idx[t]])  # weights are scores, not choices
        assert np.all(keff == K)


def test_select_exhaustive_small():
    vals = np.array([0.25, 0.5, 0.75], np.float32)
    E = 5
    import itertools
    for pattern in itertools.product(range(3), repeat=E):
        ch = vals[list(pattern)][None, :]
        for K in range(1, E + 1):
            idx, _, _ = oracle.select(ch, ch, K, 0, 1.0)
            assert list(idx[0]) == _brute_topk(ch[0], K)


@pytest.mark.parametrize("rs", [1.0, 2.5])
def test_renorm_sums_to_routed_scale(rs):
    rng = np.random.default_rng(9)
    T, E, K = 50, 64, 8
    sig = rng.uniform(0.01, 1, (T, E)).astype(np.float32)
    idx, w, _ = oracle.select(sig, sig, K, 1, rs)
    tot = w.astype(np.float64).sum(axis=1)
    assert np.all(np.abs(tot - rs) <= 4 * K * np.spacing(np.float32(rs)))
    _, w0, _ = oracle.select(sig, sig, K, 0, rs)
    assert np.array_equal(w0, (np.take_along_axis(sig, idx, 1) * np.float32(rs)).astype(np.float32))


def test_top_p_prefix_rule_brute_force():
    rng = np.random.default_rng(21)
    T, E, K = 200, 32, 8
    sig = rng.uniform(0, 1, (T, E)).astype(np.float32)
    ch = (sig + rng.uniform(-0.3, 0.3, (T, E))).astype(np.float32)
    p = 0.6
    idx, w, keff = oracle.select(sig, ch, K, 0, 1.0, 0, p)
    for t in range(T):
        sel = _brute_topk(ch[t], K)
        ws = sorted([float(sig[t, e]) for e in sel], reverse=True)
        tot = sum(ws)
        cum = np.cumsum(ws)
        if np.min(np.abs(cum - p * tot)) < 1e-5:
            continue  # too close to the threshold to decide in double
        ke = int(np.argmax(cum >= p * tot)) + 1
        assert keff[t] == ke
        assert np.allclose(w[t, :ke], ws[:ke], rtol=0, atol=0)
        assert np.all(idx[t, ke:] == -1)


# ---------------------------------------------------------------- buckets
def test_buckets_golden():
    for line in golden_lines("buckets.txt"):
        parts = [p.split() for p in line.split("|")]
        T, K, E = map(int, parts[0])
        idx = np.array(parts[1], np.int32).reshape(T, K)
        counts, offsets, perm = oracle.buckets(idx, E)
        assert list(counts) == list(map(int, parts[2]))
        assert list(offsets) == list(map(int, parts[3]))
        assert list(perm) == list(map(int, parts[4]))


@pytest.mark.parametrize("T,K,E", [(1, 8, 64), (32, 8, 256), (100, 3, 7), (2048, 8, 256)])
def test_buckets_invariants(T, K, E):
    rng = np.random.default_rng(T + K + E)
    idx = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    counts, offsets, perm = oracle.buckets(idx, E)
    assert counts.sum() == T * K
    assert np.array_equal(np.sort(perm), np.arange(T * K))
    assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(idx.reshape(-1)[seg] == e)  # perm reproduces idx
        assert np.all(np.diff(seg // K) > 0)  # strictly increasing tokens within a bucket
    # with keff: only the first keff[t] of each row are bucketed
    keff = rng.integers(1, K + 1, T).astype(np.int32)
    c2, o2, p2 = oracle.buckets(idx, E, keff)
    assert c2.sum() == keff.sum() and len(p2) == keff.sum()
    assert np.all(p2 % K < keff[p2 // K])


# ---------------------------------------------------------------- the block
def _silu(z):
    return z / (1.0 + math.exp(-z))


def _tiny_block(routed, shared, Wr, bias, x, E, K, H, I, Is, fmt, norm=1, rs=1.0):
    def slabify(mats):
        return {k: np.ascontiguousarray(v) for k, v in mats.items()}
    cfg = dict(T=x.shape[0], H=H, I=I, E=E, K=K, I_shared=Is, norm_topk=norm, routed_scale=rs,
               routed_fmt=fmt, shared_fmt=fmt)
    return dict(cfg=cfg, x=x, Wr=Wr, bias=bias, routed=[slabify(r) for r in routed],
                shared=None if shared is None else slabify(shared))


def _i8(rows):
    return np.array(rows, np.int8).view(np.uint8)


def test_block_hand_worked():
    """H=2, I=1, E=2, K=1, shared I_s=1, int8 weights.  Router logits are 0 for both experts,
    so sig = 0.5 each; bias (0, 0.25) selects expert 1; renorm gives w = 1, routed_scale 2
    gives w = 2.  Expert 1: g = 1, u = 2, h = 2*silu(1), y = (h, -h/2).  Shared: g = 3, u = 1,
    h = silu(3), y = (h, 2h).  out = 2*y1 + y_sh."""
    H, I, Is = 2, 1, 1
    one = lambda n: np.ones(n, np.float32)
    dummy = dict(gate_w=_i8([[0, 0]]), gate_s=one(1), up_w=_i8([[0, 0]]), up_s=one(1),
                 down_w=_i8([[0], [0]]), down_s=one(2))
    e1 = dict(gate_w=_i8([[1, 0]]), gate_s=one(1), up_w=_i8([[0, 1]]), up_s=one(1),
              down_w=_i8([[1], [-1]]), down_s=np.array([1.0, 0.5], np.float32))
    sh = dict(gate_w=_i8([[1, 1]]), gate_s=one(1), up_w=_i8([[1, 0]]), up_s=one(1),
              down_w=_i8([[1], [2]]), down_s=one(2))
    blk = _tiny_block([dummy, e1], sh, np.zeros((2, H), np.float32),
                      np.array([0.0, 0.25], np.float32), np.array([[1.0, 2.0]], np.float32),
                      2, 1, H, I, Is, F8, norm=1, rs=2.0)
    out, idx, w, keff = oracle.moe_forward(blk)
    assert idx[0, 0] == 1 and w[0, 0] == 2.0 and keff[0] == 1
    h1 = _silu(1.0) * 2.0
    hs = _silu(3.0)
    expect = np.array([2 * h1 + hs, 2 * (-0.5 * h1) + 2 * hs])
    assert np.allclose(out[0], expect, rtol=1e-6, atol=0)


def _torch_ffn(fmt, ex, x, H, Iin):
    """Dense SwiGLU on the dequantised weights, in float64 with torch: down(silu(gate x)*(up x))."""
    Wg = torch.tensor(np_deq(fmt, ex["gate_w"], H) * ex["gate_s"][:, None].astype(np.float64))
    Wu = torch.tensor(np_deq(fmt, ex["up_w"], H) * ex["up_s"][:, None].astype(np.float64))
    Wd = torch.tensor(np_deq(fmt, ex["down_w"], Iin) * ex["down_s"][:, None].astype(np.float64))
    xt = torch.tensor(x.astype(np.float64))
    return (Wd @ (torch.nn.functional.silu(Wg @ xt) * (Wu @ xt))).numpy()


@pytest.mark.parametrize("fmt", [F8, F4, F2])
def test_block_single_expert_is_dense_swiglu(fmt):
    """E=1, K=1, renormalised: the routed weight is s/(s+1e-20) = 1 exactly, so the block is two
    dense SwiGLU FFNs (routed + shared) — a textbook layer, computed here with torch in float64."""
    cfg = dict(T=3, H=96, I=64, E=1, K=1, I_shared=32, norm_topk=1, routed_scale=1.0,
               routed_fmt=fmt, shared_fmt=fmt, zipf=False)
    blk = synth.make_block(cfg, seed=31 + fmt)
    out, idx, w, _ = oracle.moe_forward(blk)
    assert np.all(idx == 0) and np.all(w == 1.0)
    for t in range(cfg["T"]):
        ref = (_torch_ffn(fmt, blk["routed"][0], blk["x"][t], 96, 64) +
               _torch_ffn(fmt, blk["shared"], blk["x"][t], 96, 32))
        assert np.allclose(out[t], ref, rtol=0, atol=2e-5 * np.sqrt(np.mean(ref ** 2)))


def _torch_ffn_grouped(ex, x, H, Iin, gs):
    """Dense SwiGLU on int4-grouped weights (numpy decode, per-group scales), float64 torch."""
    Wg = torch.tensor(np_deq(F4, ex["gate_w"], H) * np_group_scales(ex["gate_s"], Iin, H, gs))
    Wu = torch.tensor(np_deq(F4, ex["up_w"], H) * np_group_scales(ex["up_s"], Iin, H, gs))
    Wd = torch.tensor(np_deq(F4, ex["down_w"], Iin) * np_group_scales(ex["down_s"], H, Iin, gs))
    xt = torch.tensor(x.astype(np.float64))
    return (Wd @ (torch.nn.functional.silu(Wg @ xt) * (Wu @ xt))).numpy()


@pytest.mark.parametrize("gs", [32, 64])
def test_block_grouped_single_expert_is_dense_swiglu(gs):
    """Format 4 through the whole block: E=1, K=1 (weight exactly 1), so routed + shared are two
    dense SwiGLU FFNs whose weights carry one scale per group of gs inputs (H=96 and I=80 leave
    ragged last groups)."""
    cfg = dict(T=3, H=96, I=80, E=1, K=1, I_shared=48, norm_topk=1, routed_scale=1.0,
               routed_fmt=F4G, shared_fmt=F4G, group_size=gs, zipf=False)
    blk = synth.make_block(cfg, seed=41 + gs)
    out, idx, w, _ = oracle.moe_forward(blk)
    assert np.all(idx == 0) and np.all(w == 1.0)
    for t in range(cfg["T"]):
        ref = (_torch_ffn_grouped(blk["routed"][0], blk["x"][t], 96, 80, gs) +
               _torch_ffn_grouped(blk["shared"], blk["x"][t], 96, 48, gs))
        assert np.allclose(out[t], ref, rtol=0, atol=2e-5 * np.sqrt(np.mean(ref ** 2)))


def test_block_grouped_with_equal_group_scales_is_per_row_int4():
    # every group of a row given the row's first scale: the block equals the per-row int4 block
    # on the same weights (same routing; outputs within float rounding)
    gs, H, I, Is = 32, 128, 64, 32
    cfg = dict(T=5, H=H, I=I, E=6, K=3, I_shared=Is, norm_topk=1, routed_scale=2.5,
               routed_fmt=F4G, shared_fmt=F4G, group_size=gs, zipf=False)
    blk = synth.make_block(cfg, seed=77)

    def inputs_of(key, Iin):
        return Iin if key == "down_s" else H

    def equalise(ex, Iin):  # in place: each row's groups all take the row's first scale
        for k in ("gate_s", "up_s", "down_s"):
            rows = ex[k].reshape(-1, (inputs_of(k, Iin) + gs - 1) // gs)
            rows[:] = rows[:, :1]

    def per_row(ex, Iin):  # the same expert with one scale per row
        out = dict(ex)
        for k in ("gate_s", "up_s", "down_s"):
            out[k] = np.ascontiguousarray(ex[k].reshape(-1, (inputs_of(k, Iin) + gs - 1) // gs)[:, 0])
        return out

    for ex in blk["routed"]:
        equalise(ex, I)
    equalise(blk["shared"], Is)
    blk4 = dict(blk, cfg=dict(cfg, routed_fmt=F4, shared_fmt=F4, group_size=0),
                routed=[per_row(ex, I) for ex in blk["routed"]], shared=per_row(blk["shared"], Is))
    o1, i1, w1, _ = oracle.moe_forward(blk)
    o2, i2, w2, _ = oracle.moe_forward(blk4)
    assert np.array_equal(i1, i2) and np.array_equal(w1, w2)
    assert np.allclose(o1, o2, rtol=0, atol=1e-6 * np.sqrt(np.mean(o2 ** 2)))


def test_block_idot_leaves_int2_and_grouped_experts_exact():
    # the engine's matmul_qt takes the IDOT kernels for int8 and int4 weights only
    for fmt, extra in ((F2, {}), (F4G, {"group_size": 32})):
        cfg = dict(T=3, H=128, I=64, E=5, K=2, I_shared=32, norm_topk=1, routed_scale=2.5,
                   routed_fmt=fmt, shared_fmt=fmt, zipf=False, **extra)
        blk = synth.make_block(cfg, seed=91)
        o1 = oracle.moe_forward(blk)[0]
        o2 = oracle.moe_forward(dict(blk, cfg=dict(cfg, idot=1)))[0]
        assert np.array_equal(o1, o2), fmt


def test_block_idot_matches_composed_idot_gemvs():
    # one token through the IDOT block equals the IDOT GEMVs composed by hand (gate and up on
    # qrow_i8(x), SwiGLU in float, down on qrow_i8(h)), weighted and combined in selection order
    cfg = dict(T=1, H=128, I=64, E=4, K=2, I_shared=32, norm_topk=1, routed_scale=2.5,
               routed_fmt=F4, shared_fmt=F8, idot=1, zipf=False)
    blk = synth.make_block(cfg, seed=93)
    out, idx, w, _ = oracle.moe_forward(blk)

    def ffn(fmt, ex, x, Iin):
        qx, sx = oracle.qrow_i8(x)
        g = oracle.qgemv_idot(fmt, ex["gate_w"], ex["gate_s"], qx, sx, Iin, 128)
        u = oracle.qgemv_idot(fmt, ex["up_w"], ex["up_s"], qx, sx, Iin, 128)
        h = (g / (np.float32(1) + np.exp(-g))) * u
        qh, sh = oracle.qrow_i8(h.astype(np.float32))
        return oracle.qgemv_idot(fmt, ex["down_w"], ex["down_s"], qh, sh, 128, Iin)

    x = blk["x"][0]
    ref = np.zeros(128, np.float32)
    for k in range(2):
        ref = ref + w[0, k] * ffn(F4, blk["routed"][idx[0, k]], x, 64)
    ref = ref + ffn(F8, blk["shared"], x, 32)
    assert np.allclose(out[0], ref, rtol=0, atol=1e-5 * np.sqrt(np.mean(ref ** 2)))


def test_block_combine_weights_and_shared_weight_one():
    cfg = dict(T=4, H=64, I=32, E=6, K=3, I_shared=16, norm_topk=1, routed_scale=2.5,
               routed_fmt=F4, shared_fmt=F8, zipf=False)
    blk = synth.make_block(cfg, seed=77, row_filter=gap_filter(3))
    out, idx, w, _ = oracle.moe_forward(blk)
    for t in range(cfg["T"]):
        ref = _torch_ffn(F8, blk["shared"], blk["x"][t], 64, 16)
        for k in range(3):
            ref = ref + float(w[t, k]) * _torch_ffn(F4, blk["routed"][idx[t, k]], blk["x"][t], 64, 32)
        assert np.allclose(out[t], ref, rtol=0, atol=2e-5 * np.sqrt(np.mean(ref ** 2)))
    # and the weights are the renormalised, scaled sigmoid scores of the selected experts
    sig, _ = oracle.router(blk["x"], blk["Wr"], blk["bias"])
    s = np.take_along_axis(sig, idx, 1).astype(np.float64)
    assert np.allclose(w, 2.5 * s / s.sum(1, keepdims=True), rtol=1e-6)


def test_block_rows_are_independent():
    cfg = dict(T=5, H=64, I=32, E=8, K=2, I_shared=32, norm_topk=1, routed_scale=2.5,
               routed_fmt=F4, shared_fmt=F4, zipf=False)
    blk = synth.make_block(cfg, seed=5)
    out, idx, w, _ = oracle.moe_forward(blk)
    for t in range(5):
        o1, i1, w1, _ = oracle.moe_forward(blk, x=blk["x"][t:t + 1])
        assert np.array_equal(o1[0], out[t]) and np.array_equal(i1[0], idx[t])


def test_block_linear_in_down_scales():
    cfg = dict(T=3, H=64, I=32, E=8, K=2, I_shared=32, norm_topk=1, routed_scale=2.5,
               routed_fmt=F8, shared_fmt=F8, zipf=False)
    blk = synth.make_block(cfg, seed=6)
    out, _, _, _ = oracle.moe_forward(blk)
    for ex in blk["routed"] + [blk["shared"]]:
        ex["down_s"][:] *= np.float32(2.0)
    out2, _, _, _ = oracle.moe_forward(blk)
    assert np.array_equal(out2, 2 * out)
    # zero the shared expert: only the routed sum remains
    blk["shared"]["down_s"][:] = 0
    out3, _, _, _ = oracle.moe_forward(blk)
    assert not np.array_equal(out3, out2)


def test_block_expert_relabelling():
    cfg = dict(T=4, H=64, I=32, E=8, K=3, I_shared=0, norm_topk=1, routed_scale=1.0,
               routed_fmt=F4, shared_fmt=F4, zipf=False)
    blk = synth.make_block(cfg, seed=8)
    out, idx, w, _ = oracle.moe_forward(blk)
    pi = np.random.default_rng(1).permutation(8)  # new id of old expert e is pi[e]
    blk2 = dict(blk)
    inv = np.argsort(pi)
    blk2["Wr"] = blk["Wr"][inv]
    blk2["bias"] = blk["bias"][inv]
    blk2["routed"] = [blk["routed"][inv[j]] for j in range(8)]
    out2, idx2, w2, _ = oracle.moe_forward(blk2)
    assert np.array_equal(out2, out)
    assert np.array_equal(idx2, pi[idx])
    assert np.array_equal(w2, w)


# ---------------------------------------------------------------- the input generator
def test_generator_is_deterministic():
    a = synth.make_block(0)
    b = synth.make_block(0)
    assert np.array_equal(a["routed_slabs"], b["routed_slabs"])
    assert np.array_equal(a["x"], b["x"]) and np.array_equal(a["Wr"], b["Wr"])


def test_gap_filter_enforces_margin():
    blk = synth.make_block(1, row_filter=gap_filter(8))
    _, ch = oracle.router(blk["x"], blk["Wr"], blk["bias"])
    top = -np.sort(-ch[0])[:9].astype(np.float64)
    assert np.all(-np.diff(top) > 1e-5)


def test_skewed_bias_concentrates_assignments():
    """The skewed continuous-batch workload: the 20% most-used experts take about half of the
    assignments (measured over many token draws with the same router)."""
    cfg = synth.config(3)
    rng = np.random.Generator(np.random.PCG64(synth.seed_for(3)))
    Wr, bias = synth.make_router(rng, cfg)
    x = np.random.default_rng(0).standard_normal((512, cfg["H"])).astype(np.float32)
    sig, ch = oracle.router(x, Wr, bias)
    idx, _, _ = oracle.select(sig, ch, cfg["K"], 1, 2.5)
    counts = np.bincount(idx.reshape(-1), minlength=cfg["E"])
    top = np.sort(counts)[::-1][: cfg["E"] // 5].sum() / counts.sum()
    assert 0.45 <= top <= 0.55, top


# ------------------------------------------------------------------ RMS normalisation (layer tail)
# glm.c rmsnorm(): r = 1 / sqrtf(mean square + eps) with the mean square accumulated in double,
# out = x * r * w. The block as the tail of a decoder layer: out = resid + moe(rmsnorm(resid)).
def test_rmsnorm_constant_rows_closed_form():
    w = np.ones(16, np.float32)
    # a constant row c has mean square c^2: r = 1 / |c| exactly for these c, eps = 0
    for c in (2.0, 0.25, -4.0):
        out = oracle.rmsnorm(np.full((1, 16), c, np.float32), w, 0.0)
        assert np.array_equal(out[0], np.full(16, np.sign(c), np.float32)), c
    # eps enters under the root: c = 1, eps = 3 gives r = 1 / 2
    out = oracle.rmsnorm(np.ones((1, 16), np.float32), w, 3.0)
    assert np.array_equal(out[0], np.full(16, 0.5, np.float32))


def test_rmsnorm_weights_multiply_elementwise():
    rng = np.random.default_rng(3)
    w = rng.uniform(0.5, 2.0, 64).astype(np.float32)
    out = oracle.rmsnorm(np.full((1, 64), 2.0, np.float32), w, 0.0)  # r * 2 = 1 exactly
    assert np.array_equal(out[0], w)


def test_rmsnorm_matches_float64_definition():
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((5, 300)) * rng.uniform(0.1, 30, (5, 1))).astype(np.float32)
    w = rng.uniform(0.5, 1.5, 300).astype(np.float32)
    eps = 1e-5
    got = oracle.rmsnorm(x, w, eps).astype(np.float64)
    xt = torch.from_numpy(x.astype(np.float64))
    ref = (xt / torch.sqrt((xt * xt).mean(dim=1, keepdim=True) + eps) * torch.from_numpy(w.astype(np.float64))).numpy()
    assert np.max(np.abs(got - ref) / np.abs(ref).max()) < 1e-6


def test_tail_normalises_the_residual_before_the_block():
    # rmsnorm is invariant to scaling its input by 2 (eps = 0), so doubling the residual doubles
    # only the residual term of the tail: tail(2 r) - 2 r == tail(r) - r up to the rounding of
    # the two residual additions. A tail that fed the raw residual to the block, or skipped the
    # norm, would differ by far more.
    cfg = dict(T=3, H=128, I=64, E=8, K=2, I_shared=64, norm_topk=1, routed_scale=2.5,
               routed_fmt=2, shared_fmt=1, zipf=False)
    blk = synth.make_block(cfg, seed=12, row_filter=gap_filter(2))
    rng = np.random.default_rng(12)
    w = rng.uniform(0.5, 1.5, 128).astype(np.float32)
    r = blk["x"] * 3.0
    a, ia, _, _ = oracle.moe_tail(blk, r, w, 0.0)
    b, ib, _, _ = oracle.moe_tail(blk, 2 * r, w, 0.0)
    assert np.array_equal(ia, ib)
    assert np.array_equal(oracle.rmsnorm(2 * r, w, 0.0), oracle.rmsnorm(r, w, 0.0))
    ulp = np.spacing(np.maximum(np.abs(b), 2 * np.abs(r)).astype(np.float32)).astype(np.float64)
    diff = np.abs((b.astype(np.float64) - 2 * r) - (a.astype(np.float64) - r))
    assert np.all(diff <= 2 * ulp)
    assert np.max(np.abs(a - r)) > 1e-3  # the block's part is not negligible


def test_tail_single_expert_is_dense_swiglu_of_the_normalised_residual():
    # E = K = 1 (weight exactly 1), int8 weights with scale 1 and |w| <= 1: the block is two dense
    # SwiGLU FFNs; the tail adds the residual to them, all in float64 here
    H, I = 64, 32
    cfg = dict(T=2, H=H, I=I, E=1, K=1, I_shared=32, norm_topk=1, routed_scale=1.0,
               routed_fmt=1, shared_fmt=1, zipf=False)
    blk = synth.make_block(cfg, seed=21)
    rng = np.random.default_rng(21)
    for ex in [blk["routed"][0], blk["shared"]]:
        for k in ("gate_w", "up_w", "down_w"):
            ex[k][...] = rng.integers(-1, 2, ex[k].shape, dtype=np.int8).view(np.uint8)
        for k in ("gate_s", "up_s", "down_s"):
            ex[k][...] = 1.0
    resid = (rng.standard_normal((2, H)) * 4).astype(np.float32)
    nw = rng.uniform(0.5, 1.5, H).astype(np.float32)
    eps = 1e-6
    out, _, _, _ = oracle.moe_tail(blk, resid, nw, eps)
    r64 = resid.astype(np.float64)
    xn = r64 / np.sqrt((r64 ** 2).mean(axis=1, keepdims=True) + eps) * nw.astype(np.float64)

    def ffn(ex, Iin):
        G = ex["gate_w"].view(np.int8)[:, :H].astype(np.float64)
        U = ex["up_w"].view(np.int8)[:, :H].astype(np.float64)
        D = ex["down_w"].view(np.int8)[:, :Iin].astype(np.float64)
        g, u = xn @ G.T, xn @ U.T
        return (g / (1 + np.exp(-g)) * u) @ D.T

    ref = r64 + ffn(blk["routed"][0], I) + ffn(blk["shared"], 32)
    assert np.max(np.abs(out - ref)) < 1e-4 * np.sqrt(np.mean(ref ** 2))
