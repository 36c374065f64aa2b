"""CPU oracle for the quantized MoE feed-forward block (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may import
this package. It wraps ``colimoe_oracle.c`` — plain single-threaded C with double accumulation —
through ctypes, building it with gcc on first use. The CUDA library never imports, links or calls
anything here, and nothing here imports the CUDA library.

The definitions are restated from the colibri pages: c/glm.c (QT formats, matmul_q / matmul_i4 /
matmul_i2, sigmoidf / siluf, moe() phases A–E) and c/backend_metal.mm (mm_gemv, moe_gemv,
moe_silu, r_router, r_top8). Each C function cites the part it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "colimoe_oracle.c")
_HDR = os.path.join(_HERE, "colimoe_oracle.h")
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "libcolimoe_oracle.so")
_lock = threading.Lock()
_lib = None

FMT_F32, FMT_INT8, FMT_INT4, FMT_INT2, FMT_INT4G = 0, 1, 2, 3, 4


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, no contraction of a*b+c into fused multiply-adds, so
    x86 and Arm hosts round identically). Returns the path of the shared library."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= newest:
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P, I, F, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_int64
        lib.oracle_row_bytes.argtypes = [I, I64]
        lib.oracle_row_bytes.restype = I64
        lib.oracle_deq.argtypes = [I, P, I64]
        lib.oracle_deq.restype = F
        lib.oracle_qgemv.argtypes = [I, P, P, P, I, I, P]
        lib.oracle_qgemv.restype = None
        lib.oracle_qgemv_grouped.argtypes = [P, P, I, P, I, I, P]
        lib.oracle_qgemv_grouped.restype = None
        lib.oracle_qrow_i8.argtypes = [P, P, I]
        lib.oracle_qrow_i8.restype = F
        lib.oracle_qgemv_idot.argtypes = [I, P, P, P, F, I, I, P]
        lib.oracle_qgemv_idot.restype = None
        lib.oracle_router.argtypes = [P, I, I, P, P, I, P, P]
        lib.oracle_router.restype = I
        lib.oracle_select.argtypes = [P, P, I, I, I, I, F, I, F, P, P, P]
        lib.oracle_select.restype = I
        lib.oracle_buckets.argtypes = [P, P, I, I, I, P, P, P]
        lib.oracle_buckets.restype = I
        lib.oracle_expert.argtypes = [I, I, I, P, P, P, P, P, P, I, I, P, P]
        lib.oracle_expert.restype = None
        lib.oracle_rmsnorm.argtypes = [P, P, I, F, P]
        lib.oracle_rmsnorm.restype = None
        lib.oracle_moe_forward.argtypes = ([I, I, I, I, I, I, F, I, F, I, P, P, P] + [P] * 6 +
                                           [I, I, I, I] + [P] * 6 + [P, P, P, P])
        lib.oracle_moe_forward.restype = I
        _lib = lib
        return lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def row_bytes(fmt: int, n: int) -> int:
    return int(_load().oracle_row_bytes(fmt, n))


def deq_row(fmt: int, row: np.ndarray, n: int) -> np.ndarray:
    """Dequantised values of the first n elements of one packed row (no scale)."""
    row = np.ascontiguousarray(row, dtype=np.uint8)
    lib = _load()
    return np.array([lib.oracle_deq(fmt, _p(row), i) for i in range(n)], dtype=np.float32)


def qgemv(fmt: int, W: np.ndarray, s, v: np.ndarray, O: int, In: int) -> np.ndarray:
    W = np.ascontiguousarray(W)
    v = _f32(v)
    s = None if s is None else _f32(s)
    y = np.empty(O, np.float32)
    _load().oracle_qgemv(fmt, _p(W), _p(s), _p(v), O, In, _p(y))
    return y


def qgemv_grouped(W: np.ndarray, s, gs: int, v: np.ndarray, O: int, In: int) -> np.ndarray:
    """int4-grouped GEMV: s is [O, ceil(In/gs)] fp32."""
    W = np.ascontiguousarray(W)
    v, s = _f32(v), _f32(s)
    y = np.empty(O, np.float32)
    _load().oracle_qgemv_grouped(_p(W), _p(s), int(gs), _p(v), O, In, _p(y))
    return y


def qrow_i8(x):
    """IDOT activation quantiser: (q int8 [n], s)."""
    x = _f32(x)
    q = np.empty(len(x), np.int8)
    s = _load().oracle_qrow_i8(_p(x), _p(q), len(x))
    return q, float(np.float32(s))


def qgemv_idot(fmt, W, s, q, sx, O, In):
    """IDOT GEMV on int8 activations q with their scale sx (int8 / int4 weights)."""
    W = np.ascontiguousarray(W)
    s = _f32(s)
    q = np.ascontiguousarray(q, dtype=np.int8)
    y = np.empty(O, np.float32)
    _load().oracle_qgemv_idot(fmt, _p(W), _p(s), _p(q), float(sx), O, In, _p(y))
    return y


def router(x, Wr, bias):
    x, Wr, bias = _f32(x), _f32(Wr), _f32(bias)
    T, H = x.shape
    E = Wr.shape[0]
    sig = np.empty((T, E), np.float32)
    ch = np.empty((T, E), np.float32)
    rc = _load().oracle_router(_p(x), T, H, _p(Wr), _p(bias), E, _p(sig), _p(ch))
    if rc != 0:
        raise ValueError("oracle_router: non-finite router score")
    return sig, ch


def select(sig, ch, K, norm_topk=1, routed_scale=1.0, ksel=0, top_p=0.0):
    sig, ch = _f32(sig), _f32(ch)
    T, E = sig.shape
    idx = np.empty((T, K), np.int32)
    w = np.empty((T, K), np.float32)
    keff = np.empty(T, np.int32)
    rc = _load().oracle_select(_p(sig), _p(ch), T, E, K, ksel, float(top_p), int(norm_topk),
                               float(routed_scale), _p(idx), _p(w), _p(keff))
    if rc != 0:
        raise ValueError("oracle_select: bad arguments")
    return idx, w, keff


def buckets(idx, E, keff=None):
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    T, K = idx.shape
    kf = None if keff is None else np.ascontiguousarray(keff, dtype=np.int32)
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(max(T * K, 1), np.int32)
    n = _load().oracle_buckets(_p(idx), _p(kf), T, K, E, _p(counts), _p(offsets), _p(perm))
    if n < 0:
        raise ValueError("oracle_buckets: expert index out of range")
    return counts, offsets, perm[:n].copy()


def expert(fmt, ex, x, H, Iin, group_size=0, idot=0):
    """One SwiGLU expert on one vector; ex is a dict with gate_w/gate_s/up_w/up_s/down_w/down_s."""
    y = np.empty(H, np.float32)
    arrs = [np.ascontiguousarray(ex[k]) for k in ("gate_w", "gate_s", "up_w", "up_s", "down_w", "down_s")]
    _load().oracle_expert(fmt, int(group_size), int(idot), *[_p(a) for a in arrs], H, Iin, _p(_f32(x)), _p(y))
    return y


def moe_forward(blk, x=None, ksel=0, top_p=0.0):
    """The whole block on the host. ``blk`` is the dict made by ``synth.make_block``.
    Returns (out [T,H], idx [T,K], w [T,K], keff [T])."""
    lib = _load()
    cfg = blk["cfg"]
    x = _f32(blk["x"] if x is None else x)
    T, H = x.shape
    E, K, I = cfg["E"], cfg["K"], cfg["I"]
    rt = blk["routed"]
    keep = []

    def table(key):
        arrs = [np.ascontiguousarray(rt[e][key]) for e in range(E)]
        keep.append(arrs)
        t = (ctypes.c_void_p * E)(*[a.ctypes.data for a in arrs])
        keep.append(t)
        return t

    tabs = [table(k) for k in ("gate_w", "gate_s", "up_w", "up_s", "down_w", "down_s")]
    sh = blk.get("shared")
    Is = cfg["I_shared"] if sh is not None else 0
    if sh is not None:
        sh_arrs = [np.ascontiguousarray(sh[k]) for k in ("gate_w", "gate_s", "up_w", "up_s", "down_w", "down_s")]
    else:
        sh_arrs = [None] * 6
    out = np.empty((T, H), np.float32)
    idx = np.empty((T, K), np.int32)
    w = np.empty((T, K), np.float32)
    keff = np.empty(T, np.int32)
    Wr, bias = _f32(blk["Wr"]), _f32(blk["bias"])
    rc = lib.oracle_moe_forward(T, H, I, E, K, ksel, float(top_p), int(cfg["norm_topk"]),
                                float(cfg["routed_scale"]), cfg["routed_fmt"], _p(x), _p(Wr), _p(bias),
                                *[ctypes.cast(t, ctypes.c_void_p) for t in tabs],
                                Is, cfg["shared_fmt"], int(cfg.get("group_size", 0)), int(cfg.get("idot", 0)),
                                *[_p(a) for a in sh_arrs],
                                _p(out), _p(idx), _p(w), _p(keff))
    if rc != 0:
        raise ValueError("oracle_moe_forward failed (bad arguments or non-finite router score)")
    return out, idx, w, keff


def rmsnorm(x, w, eps):
    """RMS normalisation of each row of x (glm.c rmsnorm): rows * r * w, r from the row's mean
    square accumulated in double."""
    x = np.atleast_2d(_f32(x))
    w = _f32(w)
    out = np.empty_like(x)
    lib = _load()
    for t in range(x.shape[0]):
        row = np.ascontiguousarray(x[t])
        o = np.empty_like(row)
        lib.oracle_rmsnorm(_p(row), _p(w), x.shape[1], float(eps), _p(o))
        out[t] = o
    return out


def moe_tail(blk, resid, norm_w, eps, ksel=0, top_p=0.0):
    """The block as the tail of a decoder layer (glm.c layer forward after the attention
    residual): xn = rmsnorm(resid, post_ln); out = resid + moe(xn), the residual added in float
    as `x[j] += tmp[j]` does. Returns (out, idx, w, keff) like moe_forward."""
    resid = np.atleast_2d(_f32(resid))
    xn = rmsnorm(resid, norm_w, eps)
    y, idx, w, keff = moe_forward(blk, x=xn, ksel=ksel, top_p=top_p)
    return (resid + y).astype(np.float32), idx, w, keff
