"""Host-side checks of the C ABI: the library loads, exports every symbol include/colimoe.h
declares, and rejects bad arguments with the documented codes before touching the GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def q():
    import __graft_entry__
    __graft_entry__._builder().build()
    import quantized_expert_decode_gb300 as q
    return q


def header_functions():
    with open(os.path.join(ROOT, "include", "colimoe.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(coli_moe_[a-z_]+)\s*\(", text,
                                 re.M)))


def test_header_and_binding_agree(q):
    names = header_functions()
    assert names == sorted(q.EXPORTS), names
    for n in names:
        assert hasattr(q.lib(), n), n


def test_library_exports_every_header_symbol(q):
    lib = ctypes.CDLL(q.LIB_PATH)
    for n in header_functions():
        getattr(lib, n)  # raises AttributeError if missing


def test_strerror_covers_codes(q):
    for code in range(-7, 1):
        assert q.coli_moe_strerror(code) != "unknown error code"
    assert q.coli_moe_strerror(-99) == "unknown error code"


def good_desc(q, **over):
    d = dict(T=4, H=256, I=128, E=8, K=2, I_shared=128, norm_topk=1, routed_scale=2.5,
             routed_fmt=2, shared_fmt=1)
    d.update(over)
    return q.make_desc(**d)


def test_workspace_bytes(q):
    n = q.coli_moe_workspace_bytes(good_desc(q))
    assert n > 0 and n % 256 == 0
    assert q.coli_moe_workspace_bytes(good_desc(q, T=8)) > n
    for bad in (dict(T=0), dict(K=0), dict(K=9), dict(E=2000), dict(K=33, E=64), dict(I_shared=-1),
                dict(norm_topk=2), dict(top_p=1.0), dict(top_p=-0.1), dict(ksel=3),
                dict(routed_fmt=7), dict(H=48), dict(I=40, routed_fmt=3), dict(routed_scale=float("nan"))):
        assert q.coli_moe_workspace_bytes(good_desc(q, **bad)) == 0, bad


FAKE = 1 << 40  # a 256-byte aligned address never dereferenced: validation fails first


def call_forward(q, desc, x=FAKE, wr=FAKE, bias=FAKE, experts=FAKE, shared="default", out=FAKE,
                 ws=FAKE, ws_bytes=None):
    if shared == "default":
        shared = q.coli_moe_expert(*[FAKE] * 6) if desc.I_shared > 0 else None
    if ws_bytes is None:
        ws_bytes = max(q.coli_moe_workspace_bytes(desc), 1)
    return q.coli_moe_forward(desc, x, wr, bias, experts, shared, out, None, None, ws, ws_bytes,
                              raise_on_error=False)


def test_forward_rejects_bad_arguments(q):
    d = good_desc(q)
    assert call_forward(q, d, x=None) == q.COLI_MOE_EINVAL
    assert call_forward(q, d, out=None) == q.COLI_MOE_EINVAL
    assert call_forward(q, d, experts=None) == q.COLI_MOE_EINVAL
    assert call_forward(q, d, shared=None) == q.COLI_MOE_EINVAL  # I_shared > 0 needs it
    assert call_forward(q, good_desc(q, I_shared=0), shared=q.coli_moe_expert(*[FAKE] * 6)) == q.COLI_MOE_EINVAL
    assert call_forward(q, d, ws=None) == q.COLI_MOE_EWORKSPACE
    assert call_forward(q, d, ws=FAKE + 16) == q.COLI_MOE_EWORKSPACE
    assert call_forward(q, d, ws_bytes=q.coli_moe_workspace_bytes(d) - 1) == q.COLI_MOE_EWORKSPACE
    assert call_forward(q, d, wr=FAKE + 4) == q.COLI_MOE_EALIGN
    bad_shared = q.coli_moe_expert(FAKE + 8, FAKE, FAKE, FAKE, FAKE, FAKE)
    assert call_forward(q, d, shared=bad_shared) == q.COLI_MOE_EALIGN
    assert call_forward(q, good_desc(q, routed_fmt=0)) == q.COLI_MOE_ENOTSUP
    assert call_forward(q, good_desc(q, H=272)) == q.COLI_MOE_ENOTSUP  # int4 needs H % 32 == 0
    assert call_forward(q, good_desc(q, K=9)) == q.COLI_MOE_EINVAL


def test_route_rejects_bad_arguments(q):
    d = good_desc(q)
    n = q.coli_moe_workspace_bytes(d)
    r = lambda **kw: q.coli_moe_route(d, kw.get("x", FAKE), FAKE, FAKE, kw.get("idx", FAKE), FAKE,
                                      None, None, None, None, kw.get("ws", FAKE), n,
                                      raise_on_error=False)
    assert r(x=None) == q.COLI_MOE_EINVAL
    assert r(idx=None) == q.COLI_MOE_EINVAL
    assert r(x=FAKE + 4) == q.COLI_MOE_EALIGN
    assert r(ws=None) == q.COLI_MOE_EWORKSPACE


def test_qgemv_rejects_bad_arguments(q):
    g = lambda fmt=2, W=FAKE, O=8, In=64, T=1: q.coli_moe_qgemv(fmt, W, FAKE, FAKE, FAKE, O, In, T,
                                                                raise_on_error=False)
    assert g(fmt=9) == q.COLI_MOE_EINVAL
    assert g(fmt=0) == q.COLI_MOE_ENOTSUP
    assert g(W=None) == q.COLI_MOE_EINVAL
    assert g(O=0) == q.COLI_MOE_EINVAL
    assert g(In=48) == q.COLI_MOE_ENOTSUP
    assert g(W=FAKE + 8) == q.COLI_MOE_EALIGN


def test_grouped_format_validation(q):
    # int4-grouped blocks need a group size that is a positive multiple of 32 (whole chunks)
    G = q.COLI_FMT_INT4G
    assert q.coli_moe_workspace_bytes(good_desc(q, routed_fmt=G, group_size=32)) > 0
    assert q.coli_moe_workspace_bytes(good_desc(q, routed_fmt=G, shared_fmt=G, group_size=128)) > 0
    for gs in (0, -32, 16, 48, 1 << 20):
        assert q.coli_moe_workspace_bytes(good_desc(q, routed_fmt=G, group_size=gs)) == 0, gs
        assert q.coli_moe_workspace_bytes(good_desc(q, shared_fmt=G, group_size=gs)) == 0, gs
    # without a grouped expert the field is ignored; a grouped shared slot without a shared
    # expert is not a grouped block
    assert q.coli_moe_workspace_bytes(good_desc(q, group_size=7)) > 0
    assert q.coli_moe_workspace_bytes(good_desc(q, I_shared=0, shared_fmt=G, group_size=0)) > 0
    assert call_forward(q, good_desc(q, routed_fmt=G, group_size=48)) == q.COLI_MOE_EINVAL
    assert call_forward(q, good_desc(q, routed_fmt=G, group_size=64, H=272)) == q.COLI_MOE_ENOTSUP


def test_qgemv_grouped_rejects_bad_arguments(q):
    g = lambda W=FAKE, gs=64, O=8, In=64, T=1: q.coli_moe_qgemv_grouped(W, FAKE, gs, FAKE, FAKE, O, In, T,
                                                                         raise_on_error=False)
    # the plain entry point needs the group size for format 4
    assert q.coli_moe_qgemv(q.COLI_FMT_INT4G, FAKE, FAKE, FAKE, FAKE, 8, 64, 1,
                            raise_on_error=False) == q.COLI_MOE_ENOTSUP
    assert g(gs=0) == q.COLI_MOE_EINVAL
    assert g(gs=48) == q.COLI_MOE_EINVAL
    assert g(W=None) == q.COLI_MOE_EINVAL
    assert g(O=0) == q.COLI_MOE_EINVAL
    assert g(In=48) == q.COLI_MOE_ENOTSUP
    assert g(W=FAKE + 8) == q.COLI_MOE_EALIGN


def test_idot_flag_validation(q):
    assert q.coli_moe_workspace_bytes(good_desc(q, idot=1)) > 0
    for bad in (2, -1):
        assert q.coli_moe_workspace_bytes(good_desc(q, idot=bad)) == 0, bad


def test_noalloc_scratch_bound_at_block_shapes(q):
    # the fixed scratch of coli_moe_forward_noalloc admits T <= 89 at the GLM-5.2 block shapes
    # (the bound the header states); the workspace grows with T on both sides of it, also where
    # the router partials switch to the 128 x 128 tiles (T = 128)
    shapes = dict(H=6144, I=2048, E=256, K=8, I_shared=2048, routed_scale=2.5)
    ws = {T: q.coli_moe_workspace_bytes(q.make_desc(T=T, **shapes)) for T in (1, 64, 89, 90, 127, 128, 2048)}
    assert ws[89] <= q.COLI_MOE_NOALLOC_SCRATCH_BYTES < ws[90]
    order = sorted(ws)
    assert all(ws[a] < ws[b] for a, b in zip(order, order[1:])), ws
