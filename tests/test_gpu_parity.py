"""Parity of the CUDA library with the CPU oracle, through the C ABI.

Bars (from the block's definition and fp32 arithmetic): selected expert ids, keff and the
token->expert buckets bit-exact; routing weights within 1e-5 relative (fp32 logit sums in a
different order, then sigmoid / renorm); block outputs max|err| <= 1e-4 * rms(oracle) on the
fp32 CUDA-core path. Inputs are drawn so that the K+1 best router choices of every token are
separated by more than 1e-5 (tests/conftest.py gap_filter), so the selection is decided the
same way on both sides.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
import synth
from conftest import gap_filter, oracle_rows, plant_tie, tail_inputs, top_p_filter, with_heavy_tails

pytestmark = pytest.mark.gpu

OUT_TOL = 1e-4
W_RTOL = 1e-5
# T > 64 runs the expert GEMMs on the tensor cores with bf16 activations and fp32 accumulation
PREFILL_TOL = 2e-2
PREFILL_MIN_T = 65


@pytest.fixture(scope="module")
def qed():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import quantized_expert_decode_gb300 as q
    return q


def rms(a):
    return float(np.sqrt(np.mean(np.asarray(a, np.float64) ** 2)))


def assert_out_close(got, ref, tol=OUT_TOL, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.max(np.abs(got - ref))
    assert np.all(np.isfinite(got)), what
    assert err <= tol * rms(ref), f"{what}: max|err| {err:.3e} > {tol} * rms {rms(ref):.3e}"


def run_forward(q, dev, x_np, check=True):
    T, H = x_np.shape
    K = dev.cfg["K"]
    dev.set_tokens(T)
    x = torch.from_numpy(x_np).to(dev.device)
    out = torch.empty((T, H), dtype=torch.float32, device=dev.device)
    idx = torch.empty((T, K), dtype=torch.int32, device=dev.device)
    w = torch.empty((T, K), dtype=torch.float32, device=dev.device)
    q.coli_moe_forward(dev.desc, x, dev.Wr, dev.bias, dev.table, dev.shared, out, idx, w,
                       dev.ws, dev.ws_bytes)
    if check:
        q.coli_moe_check(dev.ws)
    torch.cuda.synchronize()
    return out.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()


def run_route(q, dev, x_np):
    T, H = x_np.shape
    K, E = dev.cfg["K"], dev.cfg["E"]
    dev.set_tokens(T)
    d = dev.device
    x = torch.from_numpy(x_np).to(d)
    idx = torch.empty((T, K), dtype=torch.int32, device=d)
    w = torch.empty((T, K), dtype=torch.float32, device=d)
    keff = torch.empty(T, dtype=torch.int32, device=d)
    counts = torch.empty(E, dtype=torch.int32, device=d)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=d)
    perm = torch.full((T * K,), -7, dtype=torch.int32, device=d)
    q.coli_moe_route(dev.desc, x, dev.Wr, dev.bias, idx, w, keff, counts, offsets, perm, dev.ws,
                     dev.ws_bytes)
    q.coli_moe_check(dev.ws)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in (idx, w, keff, counts, offsets, perm)]


def check_route(q, blk, dev, ksel=0, top_p=0.0):
    idx, w, keff, counts, offsets, perm = run_route(q, dev, blk["x"])
    sig, ch = oracle.router(blk["x"], blk["Wr"], blk["bias"])
    cfg = blk["cfg"]
    oi, ow, ok = oracle.select(sig, ch, cfg["K"], cfg["norm_topk"], cfg["routed_scale"], ksel, top_p)
    assert np.array_equal(idx, oi)
    assert np.array_equal(keff, ok)
    assert np.allclose(w, ow, rtol=W_RTOL, atol=0)
    oc, oo, op = oracle.buckets(oi, cfg["E"], ok)
    assert np.array_equal(counts, oc) and np.array_equal(offsets, oo)
    assert np.array_equal(perm[: len(op)], op)


def check_forward(q, blk, dev, tokens=None, ksel=0, top_p=0.0, tol=OUT_TOL):
    """Every token (or the listed ones) against its own oracle call, element by element."""
    out, idx, w = run_forward(q, dev, blk["x"])
    rows = range(blk["x"].shape[0]) if tokens is None else tokens
    ref = oracle_rows(blk, rows, ksel=ksel, top_p=top_p)
    for t in rows:
        ro, ri, rw = ref[t]
        assert np.array_equal(idx[t], ri), t
        assert np.allclose(w[t], rw, rtol=W_RTOL, atol=0), t
        assert_out_close(out[t], ro, tol, what=f"token {t}")
    return out


def make(cfg, seed, K=None):
    K = cfg["K"] if K is None else K
    return synth.make_block(cfg, seed=seed, row_filter=gap_filter(K))


# ------------------------------------------------------------------ building block: qgemv
@pytest.mark.parametrize("fmt", [1, 2, 3])
def test_qgemv_unit_vectors_exact(qed, fmt):
    rng = np.random.default_rng(fmt)
    O, In = 37, 2 * {1: 16, 2: 32, 3: 64}[fmt]
    rb = synth.row_bytes(fmt, In)
    W = rng.integers(0, 256, size=(O, rb), dtype=np.uint8)
    s = rng.uniform(0.5, 2, O).astype(np.float32)
    x = np.eye(In, dtype=np.float32)  # T = In unit vectors
    d = torch.device("cuda")
    y = torch.empty((In, O), dtype=torch.float32, device=d)
    q = qed
    q.coli_moe_qgemv(fmt, torch.from_numpy(W).to(d), torch.from_numpy(s).to(d),
                     torch.from_numpy(x).to(d), y, O, In, In)
    got = y.cpu().numpy()
    for i in range(In):
        e = np.zeros(In, np.float32)
        e[i] = 1
        assert np.array_equal(got[i], oracle.qgemv(fmt, W, s, e, O, In)), i


@pytest.mark.parametrize("fmt", [1, 2, 3])
@pytest.mark.parametrize("T", [1, 3, 4, 9])
def test_qgemv_random(qed, fmt, T):
    rng = np.random.default_rng(10 * fmt + T)
    O, In = 70, 6 * {1: 16, 2: 32, 3: 64}[fmt]
    rb = synth.row_bytes(fmt, In)
    W = rng.integers(0, 256, size=(O, rb), dtype=np.uint8)
    s = rng.uniform(0.5, 2, O).astype(np.float32)
    x = rng.standard_normal((T, In)).astype(np.float32)
    d = torch.device("cuda")
    y = torch.empty((T, O), dtype=torch.float32, device=d)
    qed.coli_moe_qgemv(fmt, torch.from_numpy(W).to(d), torch.from_numpy(s).to(d),
                       torch.from_numpy(x).to(d), y, O, In, T)
    got = y.cpu().numpy()
    for t in range(T):
        assert_out_close(got[t], oracle.qgemv(fmt, W, s, x[t], O, In), what=f"t={t}")


# ------------------------------------------------------------------ the five workloads
@pytest.fixture(scope="module")
def blocks(qed):
    cache = {}

    def get(cid):
        if cid not in cache:
            cfg = synth.config(cid)
            blk = make(cfg, synth.seed_for(cid))
            from quantized_expert_decode_gb300.device import DeviceBlock
            cache.clear()  # keep one large block resident at a time
            torch.cuda.empty_cache()
            cache[cid] = (blk, DeviceBlock(blk))
        return cache[cid]
    return get


@pytest.mark.parametrize("cid", [0, 1, 2, 3, 4])
def test_route_workload(qed, blocks, cid):
    blk, dev = blocks(cid)
    check_route(qed, blk, dev)


@pytest.mark.parametrize("cid", [0, 1, 2, 3, 4])
def test_forward_workload(qed, blocks, cid):
    """Every token of every workload (2048 at prefill) against the oracle."""
    blk, dev = blocks(cid)
    tol = PREFILL_TOL if blk["cfg"]["T"] >= PREFILL_MIN_T else OUT_TOL
    check_forward(qed, blk, dev, tol=tol)


def test_forward_is_deterministic(qed, blocks):
    blk, dev = blocks(3)
    a, _, _ = run_forward(qed, dev, blk["x"])
    b, _, _ = run_forward(qed, dev, blk["x"])
    assert np.array_equal(a, b)


def test_forward_host_matches_device(qed, blocks):
    blk, dev = blocks(3)
    out_d, _, _ = run_forward(qed, dev, blk["x"])
    x_h = torch.from_numpy(blk["x"]).pin_memory()
    out_h = torch.empty(blk["x"].shape, dtype=torch.float32).pin_memory()
    qed.coli_moe_forward_host(dev.desc, x_h, dev.Wr, dev.bias, dev.table, dev.shared, out_h,
                              dev.ws, dev.ws_bytes)
    assert np.array_equal(out_h.numpy(), out_d)


# ------------------------------------------------------------------ exact ties in the router
# The pages' scan keeps the first of equal choices, so an exact tie goes to the lower expert id
# (moe() phase A of colibri-strix c/glm.c @98759bf; "ties prefer the LOWER index" in the
# r_top8_par shader). Expert b's router row and bias are copies of expert a's (a < b), so the
# two choices are bitwise equal on both sides; each token's x is moved along W_r[a] so that a
# is pick K - 1 (b just misses the cut: membership) or an earlier pick (b follows a: order).
# Every other gap among the K + 2 best choices exceeds the usual margin. T = 1 runs the
# single-token kernel, T = 4 and 16 the token-group kernel, T = 96 the router launches and the
# tensor-core GEMMs; b sits in another block of 32 experts than a, or in the same one.
TIES = [(1, None), (1, 3), (4, None), (16, None), (16, 5), (96, None)]


@pytest.mark.parametrize("T,b_off", TIES, ids=[f"T{t}-{'same' if o else 'other'}-block" for t, o in TIES])
def test_exact_tie_goes_to_lower_index(qed, T, b_off):
    from quantized_expert_decode_gb300.device import DeviceBlock
    K = 8
    cfg = dict(T=T, H=256, I=128, E=64, K=K, I_shared=64, norm_topk=1, routed_scale=2.5,
               routed_fmt=2, shared_fmt=2, zipf=False)
    blk = make(cfg, seed=700 + T)
    places = [K - 1 if (t % 2 == 0 or T == 1) else t % K for t in range(T)]
    if T == 1 and b_off is not None:
        places = [2]
    blk, a, b = plant_tie(blk, K, places, seed=T, b_off=b_off)
    dev = DeviceBlock(blk)
    check_route(qed, blk, dev)
    out, idx, w = run_forward(qed, dev, blk["x"])
    for t in range(T):
        row = list(idx[t])
        assert row[places[t]] == a, (t, row)  # the lower id takes the contested place
        if places[t] == K - 1:
            assert b not in row, (t, row)
        else:
            assert row[places[t] + 1] == b, (t, row)
    check_forward(qed, blk, dev, tol=PREFILL_TOL if T >= PREFILL_MIN_T else OUT_TOL)


# ------------------------------------------------------------------ heavy-tailed activations
# x = N(0, 1) with three entries per token at 100-1000 times that rms: the fixed-point staging
# of the single-token core (24 bits relative to max|x|), the f16 hi/lo parts of the tensor-core
# core (22 bits relative to each token's max|x|) and the bf16 rounding of the prefill GEMMs
# are all relative to the largest entry, so this is where their error is largest.
@pytest.mark.parametrize("T", [1, 4, 16, 96])
def test_heavy_tailed_activations(qed, T):
    from quantized_expert_decode_gb300.device import DeviceBlock
    cfg = dict(T=T, H=512, I=256, E=32, K=4, I_shared=128, norm_topk=1, routed_scale=2.5,
               routed_fmt=2, shared_fmt=1, zipf=False)
    blk = with_heavy_tails(make(cfg, seed=800 + T), seed=T, K=cfg["K"])
    dev = DeviceBlock(blk)
    check_route(qed, blk, dev)
    check_forward(qed, blk, dev, tol=PREFILL_TOL if T >= PREFILL_MIN_T else OUT_TOL)


# ------------------------------------------------------------------ ragged and degenerate shapes
EDGE = [
    # name, cfg overrides
    ("ragged-int4", dict(T=7, H=352, I=160, E=40, K=3, I_shared=96, routed_fmt=2, shared_fmt=2)),
    ("mixed-fmt", dict(T=5, H=256, I=128, E=24, K=4, I_shared=64, routed_fmt=2, shared_fmt=1)),
    ("int2", dict(T=6, H=384, I=192, E=16, K=2, I_shared=128, routed_fmt=3, shared_fmt=3)),
    ("k1-no-shared", dict(T=3, H=128, I=64, E=5, K=1, I_shared=0, routed_fmt=1, shared_fmt=1)),
    ("k-equals-e", dict(T=4, H=128, I=64, E=6, K=6, I_shared=32, routed_fmt=2, shared_fmt=1)),
    ("one-expert", dict(T=9, H=64, I=32, E=1, K=1, I_shared=0, routed_fmt=2, shared_fmt=2)),
    ("no-renorm", dict(T=3, H=128, I=64, E=12, K=3, I_shared=32, norm_topk=0, routed_scale=1.5)),
    ("hot-bucket", dict(T=23, H=128, I=64, E=3, K=2, I_shared=64)),
    ("max-e-k", dict(T=2, H=64, I=32, E=1024, K=32, I_shared=0)),
    # T > 8: the token images of the tensor-core core, per routed format, ragged segments
    ("int8-t12", dict(T=12, H=256, I=128, E=6, K=3, I_shared=64, routed_fmt=1, shared_fmt=2)),
    ("int2-t16", dict(T=16, H=256, I=128, E=5, K=2, I_shared=64, routed_fmt=3, shared_fmt=1)),
    ("ragged-t20", dict(T=20, H=352, I=160, E=7, K=3, I_shared=96, routed_fmt=2, shared_fmt=2)),
]


@pytest.mark.parametrize("name,over", EDGE, ids=[e[0] for e in EDGE])
def test_edge_shapes(qed, name, over):
    from quantized_expert_decode_gb300.device import DeviceBlock
    cfg = dict(T=4, H=128, I=64, E=8, K=2, I_shared=64, norm_topk=1, routed_scale=2.5,
               routed_fmt=2, shared_fmt=2, zipf=False)
    cfg.update(over)
    blk = make(cfg, seed=zlib.crc32(name.encode()) % 1000)
    dev = DeviceBlock(blk)
    check_route(qed, blk, dev)
    check_forward(qed, blk, dev)


@pytest.mark.parametrize("ksel,top_p", [(3, 0.0), (0, 0.5), (5, 0.8)])
def test_topk_override_and_top_p(qed, ksel, top_p):
    from quantized_expert_decode_gb300.device import DeviceBlock
    cfg = dict(T=16, H=256, I=128, E=32, K=8, I_shared=64, norm_topk=1, routed_scale=2.5,
               routed_fmt=2, shared_fmt=2, zipf=False)
    blk = synth.make_block(cfg, seed=ksel * 10 + int(top_p * 10),
                           row_filter=top_p_filter(8, ksel, top_p))
    dev = DeviceBlock(blk, ksel=ksel, top_p=top_p)
    check_route(qed, blk, dev, ksel=ksel, top_p=top_p)
    check_forward(qed, blk, dev, ksel=ksel, top_p=top_p)


# ------------------------------------------------------------------ one token (the single-token kernel)
# T = 1 runs its own kernel: every routed/shared format pair, ragged sizes, fewer output-row
# blocks than CTAs, E not a multiple of 4, K at its maximum, no shared expert, no renorm.
EDGE1 = [
    ("i8-i8", dict(H=512, I=256, E=16, K=4, I_shared=128, routed_fmt=1, shared_fmt=1)),
    ("i4-i8", dict(H=768, I=384, E=40, K=6, I_shared=256, routed_fmt=2, shared_fmt=1)),
    ("i2-i4", dict(H=384, I=192, E=16, K=2, I_shared=128, routed_fmt=3, shared_fmt=2)),
    ("i8-i2", dict(H=320, I=128, E=9, K=3, I_shared=192, routed_fmt=1, shared_fmt=3)),
    ("ragged-e37", dict(H=352, I=160, E=37, K=5, I_shared=96, routed_fmt=2, shared_fmt=2)),
    ("few-rows", dict(H=64, I=64, E=6, K=2, I_shared=64, routed_fmt=2, shared_fmt=2)),
    ("k32", dict(H=256, I=128, E=64, K=32, I_shared=0, routed_fmt=2, shared_fmt=2)),
    ("k1-no-shared", dict(H=128, I=64, E=5, K=1, I_shared=0, routed_fmt=2, shared_fmt=2)),
    ("no-renorm", dict(H=256, I=128, E=12, K=3, I_shared=64, norm_topk=0, routed_scale=1.5)),
    ("e1024", dict(H=128, I=64, E=1024, K=8, I_shared=64, routed_fmt=2, shared_fmt=2)),
]


@pytest.mark.parametrize("name,over", EDGE1, ids=[e[0] for e in EDGE1])
def test_one_token_shapes(qed, name, over):
    from quantized_expert_decode_gb300.device import DeviceBlock
    cfg = dict(T=1, H=128, I=64, E=8, K=2, I_shared=64, norm_topk=1, routed_scale=2.5,
               routed_fmt=2, shared_fmt=2, zipf=False)
    cfg.update(over)
    blk = make(cfg, seed=zlib.crc32(("one-" + name).encode()) % 1000)
    dev = DeviceBlock(blk)
    check_route(qed, blk, dev)
    check_forward(qed, blk, dev)


@pytest.mark.parametrize("ksel,top_p", [(3, 0.0), (0, 0.5), (5, 0.8)])
def test_one_token_topk_and_top_p(qed, ksel, top_p):
    from quantized_expert_decode_gb300.device import DeviceBlock
    cfg = dict(T=1, H=256, I=128, E=32, K=8, I_shared=64, norm_topk=1, routed_scale=2.5,
               routed_fmt=2, shared_fmt=2, zipf=False)
    blk = synth.make_block(cfg, seed=100 + ksel * 10 + int(top_p * 10),
                           row_filter=top_p_filter(8, ksel, top_p))
    dev = DeviceBlock(blk, ksel=ksel, top_p=top_p)
    check_route(qed, blk, dev, ksel=ksel, top_p=top_p)
    check_forward(qed, blk, dev, ksel=ksel, top_p=top_p)


def test_one_token_many_calls(qed, blocks):
    """Fresh tokens through the same block, back to back: counters and scratch start clean."""
    blk, dev = blocks(1)
    cfg = blk["cfg"]
    xs = synth.make_x_batches(cfg, 515, 6)
    for i in range(6):
        out, idx, w = run_forward(qed, dev, xs[i])
        ro, ri, rw, rk = oracle.moe_forward(blk, x=xs[i])
        assert np.array_equal(idx[0], ri[0]), i
        assert_out_close(out[0], ro[0], what=f"call {i}")


# ------------------------------------------------------------------ prefill (tensor-core GEMMs)
# T > 64: every format pair, token counts that leave ragged N tiles, more tokens per expert than
# one N tile holds, no shared expert, and a 16-bit-unfriendly activation scale.
PREFILL = [
    ("i4-i4", dict(T=96, H=256, I=128, E=8, K=2, I_shared=128)),
    ("i8-i8", dict(T=80, H=192, I=128, E=6, K=2, I_shared=64, routed_fmt=1, shared_fmt=1)),
    ("i2-i4", dict(T=70, H=128, I=192, E=5, K=2, I_shared=128, routed_fmt=3, shared_fmt=2)),
    ("i4-i8", dict(T=130, H=320, I=64, E=4, K=3, I_shared=192, routed_fmt=2, shared_fmt=1)),
    ("hot-expert", dict(T=300, H=128, I=128, E=3, K=1, I_shared=0)),
    ("no-shared", dict(T=100, H=256, I=256, E=16, K=4, I_shared=0)),
    # T >= 128: the router partials run as 128 x 128 tiles; 200 experts leave a ragged second
    # expert tile and 160 tokens a ragged second token tile
    ("wide-router", dict(T=160, H=256, I=128, E=200, K=4, I_shared=64)),
]


@pytest.mark.parametrize("name,over", PREFILL, ids=[e[0] for e in PREFILL])
def test_prefill_shapes(qed, name, over):
    from quantized_expert_decode_gb300.device import DeviceBlock
    cfg = dict(H=128, I=64, E=8, K=2, I_shared=64, norm_topk=1, routed_scale=2.5,
               routed_fmt=2, shared_fmt=2, zipf=False)
    cfg.update(over)
    blk = make(cfg, seed=zlib.crc32(("pf-" + name).encode()) % 1000)
    dev = DeviceBlock(blk)
    check_route(qed, blk, dev)
    check_forward(qed, blk, dev, tol=PREFILL_TOL)


def test_prefill_is_deterministic(qed):
    from quantized_expert_decode_gb300.device import DeviceBlock
    cfg = dict(T=96, H=256, I=128, E=8, K=2, I_shared=128, norm_topk=1, routed_scale=2.5,
               routed_fmt=2, shared_fmt=2, zipf=False)
    blk = make(cfg, seed=5)
    dev = DeviceBlock(blk)
    a, _, _ = run_forward(qed, dev, blk["x"])
    b, _, _ = run_forward(qed, dev, blk["x"])
    assert np.array_equal(a, b)


def test_one_token_dirty_workspace(qed, blocks):
    """The single-token kernel resets its own counters from a per-call id: a workspace full of
    garbage (here: random bytes, then the bytes of the previous call's counter block) between
    calls must not change the result."""
    blk, dev = blocks(1)
    cfg = blk["cfg"]
    xs = synth.make_x_batches(cfg, 717, 3)
    ref = []
    for i in range(3):
        out, _, _ = run_forward(qed, dev, xs[i])
        ref.append(out)
    ctrl = dev.ws[:4096].clone()
    g = torch.Generator(device="cpu").manual_seed(5)
    for i in range(3):
        noise = torch.randint(0, 256, (dev.ws.numel(),), dtype=torch.uint8, generator=g)
        dev.ws.copy_(noise.to(dev.ws.device))  # the workspace is a byte buffer
        if i == 1:
            dev.ws[:4096].copy_(ctrl)  # the counter block exactly as a finished call left it
        out, _, _ = run_forward(qed, dev, xs[i])
        assert np.array_equal(out, ref[i]), i


# ------------------------------------------------------------------ int4-grouped tensors (format 4)
def rand_grouped(rng, O, In, gs):
    W = rng.integers(0, 256, size=(O, In // 2), dtype=np.uint8)
    s = rng.uniform(0.5, 2, O * ((In + gs - 1) // gs)).astype(np.float32)
    return W, s


@pytest.mark.parametrize("gs", [32, 64, 128])
def test_qgemv_grouped_unit_vectors_exact(qed, gs):
    rng = np.random.default_rng(900 + gs)
    O, In = 21, 160  # gs = 64, 128: a ragged last group
    W, s = rand_grouped(rng, O, In, gs)
    x = np.eye(In, dtype=np.float32)
    d = torch.device("cuda")
    y = torch.empty((In, O), dtype=torch.float32, device=d)
    qed.coli_moe_qgemv_grouped(torch.from_numpy(W).to(d), torch.from_numpy(s).to(d), gs,
                               torch.from_numpy(x).to(d), y, O, In, In)
    got = y.cpu().numpy()
    for i in range(In):
        assert np.array_equal(got[i], oracle.qgemv_grouped(W, s, gs, x[i], O, In)), i


@pytest.mark.parametrize("gs", [32, 96, 128])
@pytest.mark.parametrize("T", [1, 4, 9])
def test_qgemv_grouped_random(qed, gs, T):
    rng = np.random.default_rng(950 + gs + T)
    O, In = 70, 6 * 32
    W, s = rand_grouped(rng, O, In, gs)
    x = rng.standard_normal((T, In)).astype(np.float32)
    d = torch.device("cuda")
    y = torch.empty((T, O), dtype=torch.float32, device=d)
    qed.coli_moe_qgemv_grouped(torch.from_numpy(W).to(d), torch.from_numpy(s).to(d), gs,
                               torch.from_numpy(x).to(d), y, O, In, T)
    got = y.cpu().numpy()
    for t in range(T):
        assert_out_close(got[t], oracle.qgemv_grouped(W, s, gs, x[t], O, In), what=f"t={t}")


GROUPED = [
    ("g32-one-token", dict(T=1, H=256, I=128, E=16, K=4, I_shared=64, group_size=32)),
    ("g64-ragged", dict(T=5, H=352, I=160, E=12, K=3, I_shared=96, group_size=64)),
    ("g128-routed-only", dict(T=4, H=256, I=192, E=10, K=2, I_shared=64, shared_fmt=1, group_size=128)),
    ("g32-shared-only", dict(T=3, H=256, I=128, E=8, K=2, I_shared=128, routed_fmt=2, shared_fmt=4,
                             group_size=32)),
    ("g64-long", dict(T=70, H=128, I=64, E=9, K=2, I_shared=64, group_size=64)),
    # T = 1 runs the single-token kernel, each chunk's integer sum scaled by its group
    ("g128-one-token-large", dict(T=1, H=6144, I=2048, E=256, K=8, I_shared=2048, group_size=128)),
    ("g96-one-token-ragged", dict(T=1, H=352, I=160, E=12, K=3, I_shared=96, group_size=96)),
    ("g64-one-token-int8-shared", dict(T=1, H=256, I=128, E=16, K=4, I_shared=128, shared_fmt=1,
                                       group_size=64)),
    ("g32-one-token-int2-routed", dict(T=1, H=256, I=128, E=16, K=4, I_shared=128, routed_fmt=3,
                                       shared_fmt=4, group_size=32)),
]


@pytest.mark.parametrize("name,over", GROUPED, ids=[e[0] for e in GROUPED])
def test_grouped_blocks(qed, name, over):
    from quantized_expert_decode_gb300.device import DeviceBlock
    cfg = dict(norm_topk=1, routed_scale=2.5, routed_fmt=4, shared_fmt=4, zipf=False)
    cfg.update(over)
    blk = make(cfg, seed=zlib.crc32(name.encode()) % 1000)
    dev = DeviceBlock(blk)
    check_route(qed, blk, dev)
    tokens = None if cfg["T"] <= 9 else [0, 33, 69]
    check_forward(qed, blk, dev, tokens)


# ------------------------------------------------------------------ IDOT kernels (int8 activations)
# Up to x's quantisation the gate/up products are bit-identical to the oracle's (same IEEE
# quantiser, exact integer sums, the same two products); SiLU's expf may differ by an ulp
# between CUDA and the C library, which can move an element of h across a rounding boundary
# of its int8 grid (one step of 1/127 of max|h|) before the down product. The bar allows a few
# such steps: max|err| <= 2e-3 * rms(ref); the IDOT error itself (vs the exact block) is ~0.3 %.
IDOT_TOL = 2e-3
IDOT = [
    # T = 1 runs the single-token kernel on int8 activations (both sides, one side, none when a
    # grouped expert is present: the general kernels then)
    ("idot-one-token", dict(T=1, H=256, I=128, E=16, K=4, I_shared=64, routed_fmt=2, shared_fmt=1)),
    ("idot-one-token-large", dict(T=1, H=6144, I=2048, E=256, K=8, I_shared=2048, routed_fmt=2, shared_fmt=2)),
    ("idot-one-token-int2-routed", dict(T=1, H=512, I=256, E=16, K=4, I_shared=128, routed_fmt=3, shared_fmt=1)),
    ("idot-one-token-int2-shared", dict(T=1, H=512, I=256, E=16, K=4, I_shared=128, routed_fmt=1, shared_fmt=3)),
    ("idot-one-token-int8", dict(T=1, H=512, I=256, E=16, K=4, I_shared=0, routed_fmt=1, shared_fmt=1)),
    ("idot-one-token-grouped-shared", dict(T=1, H=512, I=256, E=16, K=4, I_shared=128, routed_fmt=2,
                                           shared_fmt=4, group_size=64)),
    ("idot-int8", dict(T=5, H=256, I=128, E=12, K=3, I_shared=128, routed_fmt=1, shared_fmt=1)),
    ("idot-int2-shared", dict(T=4, H=256, I=128, E=8, K=2, I_shared=64, routed_fmt=2, shared_fmt=3)),
    ("idot-long", dict(T=70, H=128, I=64, E=9, K=2, I_shared=64, routed_fmt=2, shared_fmt=2)),
]


@pytest.mark.parametrize("name,over", IDOT, ids=[e[0] for e in IDOT])
def test_idot_blocks(qed, name, over):
    from quantized_expert_decode_gb300.device import DeviceBlock
    cfg = dict(norm_topk=1, routed_scale=2.5, zipf=False, idot=1)
    cfg.update(over)
    blk = make(cfg, seed=zlib.crc32(name.encode()) % 1000)
    dev = DeviceBlock(blk)
    check_route(qed, blk, dev)
    tokens = None if cfg["T"] <= 9 else [0, 33, 69]
    out = check_forward(qed, blk, dev, tokens, tol=IDOT_TOL)
    # the IDOT kernels ran: the result departs from the exact block's by what the IDOT definition
    # itself departs (the oracle's IDOT block against its exact block; a few percent at the
    # large shapes, where max|h| / rms(h) is large and the int8 grid coarse)
    exact = oracle.moe_forward(dict(blk, cfg=dict(cfg, idot=0)))[0]
    ref = oracle.moe_forward(blk)[0]
    rows = list(range(cfg["T"])) if tokens is None else tokens
    rel = rms(out[rows] - exact[rows]) / rms(exact[rows])
    ref_rel = rms(ref[rows] - exact[rows]) / rms(exact[rows])
    assert rel > 1e-4 and abs(rel - ref_rel) <= 0.1 * ref_rel, (rel, ref_rel)


# ------------------------------------------------------------------ the layer tail (RMSNorm folded in)
# coli_moe_forward_tail: out = resid + block(rmsnorm(resid) * norm_w), the post-attention norm
# and residual of the layer forward (colibri-strix c/glm.c @98759bf). T = 1 normalises inside the
# single-token kernel; other T through a prologue launch. Compared with oracle.moe_tail token by
# token at the path's bar (the residual is added after, so rms(out) includes it: the bar is taken
# on the block part, out - resid, against the oracle's block part).
TAILS = [
    ("one-token", dict(T=1, H=512, I=256, E=32, K=4, I_shared=128, routed_fmt=2, shared_fmt=1), False),
    ("one-token-in-place", dict(T=1, H=512, I=256, E=32, K=4, I_shared=128, routed_fmt=2, shared_fmt=2), True),
    ("token-group", dict(T=6, H=512, I=256, E=32, K=4, I_shared=128, routed_fmt=2, shared_fmt=1), True),
    ("tensor-core", dict(T=96, H=256, I=128, E=16, K=2, I_shared=128, routed_fmt=2, shared_fmt=2), False),
    ("grouped", dict(T=3, H=256, I=128, E=8, K=2, I_shared=64, routed_fmt=4, shared_fmt=4, group_size=64), False),
    ("grouped-one-token", dict(T=1, H=256, I=128, E=8, K=2, I_shared=64, routed_fmt=4, shared_fmt=4,
                               group_size=64), True),
    ("idot-one-token", dict(T=1, H=512, I=256, E=16, K=4, I_shared=128, routed_fmt=2, shared_fmt=1, idot=1), False),
]


@pytest.mark.parametrize("name,over,in_place", TAILS, ids=[t[0] for t in TAILS])
def test_layer_tail(qed, name, over, in_place):
    from quantized_expert_decode_gb300.device import DeviceBlock
    cfg = dict(norm_topk=1, routed_scale=2.5, zipf=False)
    cfg.update(over)
    blk = make(cfg, seed=zlib.crc32(("tail-" + name).encode()) % 1000)
    resid, nw, eps = tail_inputs(blk, seed=31, K=cfg["K"])
    dev = DeviceBlock(blk)
    T, H, K = cfg["T"], cfg["H"], cfg["K"]
    d = dev.device
    r = torch.from_numpy(resid).to(d)
    w = torch.from_numpy(nw).to(d)
    out = r if in_place else torch.empty((T, H), dtype=torch.float32, device=d)
    idx = torch.empty((T, K), dtype=torch.int32, device=d)
    wt = torch.empty((T, K), dtype=torch.float32, device=d)
    qed.coli_moe_forward_tail(dev.desc, r, w, eps, dev.Wr, dev.bias, dev.table, dev.shared, out, idx, wt,
                              dev.ws, dev.ws_bytes)
    qed.coli_moe_check(dev.ws)
    torch.cuda.synchronize()
    got, gi = out.cpu().numpy(), idx.cpu().numpy()
    ro, ri, rw, _ = oracle.moe_tail(blk, resid, nw, eps)
    assert np.array_equal(gi, ri)
    assert np.allclose(wt.cpu().numpy(), rw, rtol=W_RTOL, atol=0)
    tol = IDOT_TOL if cfg.get("idot", 0) else (PREFILL_TOL if T >= PREFILL_MIN_T else OUT_TOL)
    for t in range(T):
        block_ref = ro[t].astype(np.float64) - resid[t]
        block_got = got[t].astype(np.float64) - resid[t]
        # the residual's own rounding in the final add is one ulp of |out|
        slack = 2 * np.max(np.spacing(np.abs(ro[t])))
        err = np.max(np.abs(block_got - block_ref))
        assert err <= tol * rms(block_ref) + slack, (name, t, err, rms(block_ref))


def test_rmsnorm_entry_point(qed):
    rng = np.random.default_rng(8)
    T, H = 5, 768
    x = (rng.standard_normal((T, H)) * rng.uniform(0.1, 40, (T, 1))).astype(np.float32)
    w = rng.uniform(0.5, 1.5, H).astype(np.float32)
    d = torch.device("cuda")
    xn = torch.empty((T, H), dtype=torch.float32, device=d)
    qed.coli_moe_rmsnorm(torch.from_numpy(x).to(d), torch.from_numpy(w).to(d), 1e-5, xn, T, H)
    torch.cuda.synchronize()
    ref = oracle.rmsnorm(x, w, 1e-5)
    # the same float operations; only the order of the double sum differs, which can move r by
    # at most an ulp
    assert np.max(np.abs(xn.cpu().numpy() - ref) / np.abs(ref).max()) < 4e-7
