"""Python binding of libcolimoe (include/colimoe.h): argument marshalling only.

Every function here has the name of the C entry point it calls and passes device pointers
(ints, or torch tensors whose data_ptr() is taken) and a CUDA stream handle straight through.
All arithmetic of the MoE block runs in the library's CUDA kernels; there is no fallback: if
the shared library is missing this module raises on import.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libcolimoe.so")

COLI_FMT_INT8, COLI_FMT_INT4, COLI_FMT_INT2, COLI_FMT_INT4G = 1, 2, 3, 4
COLI_MOE_OK = 0
COLI_MOE_EINVAL = -1
COLI_MOE_ENOTSUP = -2
COLI_MOE_EALIGN = -3
COLI_MOE_EWORKSPACE = -4
COLI_MOE_ECUDA = -5
COLI_MOE_EDEVICE = -6
COLI_MOE_EKERNEL = -7

# every symbol include/colimoe.h declares
EXPORTS = ("coli_moe_workspace_bytes", "coli_moe_route", "coli_moe_forward", "coli_moe_forward_profiled",
           "coli_moe_forward_host", "coli_moe_qgemv", "coli_moe_qgemv_grouped", "coli_moe_check",
           "coli_moe_strerror",
           "coli_moe_last_cuda_error", "coli_moe_forward_noalloc", "coli_moe_noalloc_check",
           "coli_moe_forward_tail", "coli_moe_rmsnorm")

COLI_MOE_NOALLOC_SCRATCH_BYTES = 32 << 20


class coli_moe_desc(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32),
                ("E", ctypes.c_int32), ("K", ctypes.c_int32), ("I_shared", ctypes.c_int32),
                ("norm_topk", ctypes.c_int32), ("routed_scale", ctypes.c_float),
                ("routed_fmt", ctypes.c_int32), ("shared_fmt", ctypes.c_int32),
                ("ksel", ctypes.c_int32), ("top_p", ctypes.c_float), ("group_size", ctypes.c_int32),
                ("idot", ctypes.c_int32)]


class coli_moe_expert(ctypes.Structure):
    _fields_ = [("gate_w", ctypes.c_void_p), ("up_w", ctypes.c_void_p), ("down_w", ctypes.c_void_p),
                ("gate_s", ctypes.c_void_p), ("up_s", ctypes.c_void_p), ("down_s", ctypes.c_void_p)]


class ColiMoeError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        msg = _lib.coli_moe_strerror(code).decode() if _lib is not None else str(code)
        if code == COLI_MOE_ECUDA and _lib is not None:
            msg += f" (cudaError {_lib.coli_moe_last_cuda_error()})"
        super().__init__(f"{where}: {msg} [{code}]")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libcolimoe.so not built ({LIB_PATH}); run quantized_expert_decode_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    D = ctypes.POINTER(coli_moe_desc)
    X = ctypes.POINTER(coli_moe_expert)
    lib.coli_moe_workspace_bytes.argtypes = [D]
    lib.coli_moe_workspace_bytes.restype = SZ
    lib.coli_moe_route.argtypes = [D, P, P, P, P, P, P, P, P, P, P, SZ, P]
    lib.coli_moe_route.restype = ctypes.c_int
    lib.coli_moe_forward.argtypes = [D, P, P, P, P, X, P, P, P, P, SZ, P]
    lib.coli_moe_forward.restype = ctypes.c_int
    lib.coli_moe_forward_profiled.argtypes = [D, P, P, P, P, X, P, P, ctypes.c_int, P, SZ, P]
    lib.coli_moe_forward_profiled.restype = ctypes.c_int
    lib.coli_moe_forward_host.argtypes = [D, P, P, P, P, X, P, P, SZ, P]
    lib.coli_moe_forward_host.restype = ctypes.c_int
    lib.coli_moe_qgemv.argtypes = [I32, P, P, P, P, I32, I32, I32, P]
    lib.coli_moe_qgemv.restype = ctypes.c_int
    lib.coli_moe_qgemv_grouped.argtypes = [P, P, I32, P, P, I32, I32, I32, P]
    lib.coli_moe_qgemv_grouped.restype = ctypes.c_int
    lib.coli_moe_check.argtypes = [P, P]
    lib.coli_moe_check.restype = ctypes.c_int
    lib.coli_moe_strerror.argtypes = [ctypes.c_int]
    lib.coli_moe_strerror.restype = ctypes.c_char_p
    lib.coli_moe_forward_noalloc.argtypes = [D, P, P, P, P, X, P, P]
    lib.coli_moe_forward_noalloc.restype = ctypes.c_int
    lib.coli_moe_forward_tail.argtypes = [D, P, P, ctypes.c_float, P, P, P, X, P, P, P, P, SZ, P]
    lib.coli_moe_forward_tail.restype = ctypes.c_int
    lib.coli_moe_rmsnorm.argtypes = [P, P, ctypes.c_float, P, I32, I32, P]
    lib.coli_moe_rmsnorm.restype = ctypes.c_int
    lib.coli_moe_noalloc_check.argtypes = [P]
    lib.coli_moe_noalloc_check.restype = ctypes.c_int
    lib.coli_moe_last_cuda_error.argtypes = []
    lib.coli_moe_last_cuda_error.restype = ctypes.c_int
    return lib


_lib = _load()


def lib():
    return _lib


def _ptr(a):
    """Device/host address of a torch tensor, a numpy array, an int or None."""
    if a is None:
        return None
    if isinstance(a, int):
        return a
    if hasattr(a, "data_ptr"):
        return a.data_ptr()
    if hasattr(a, "ctypes"):
        return a.ctypes.data
    raise TypeError(f"cannot take the address of {type(a)}")


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream  # torch.cuda.Stream


def _check(rc, where, raise_on_error):
    if raise_on_error and rc != COLI_MOE_OK:
        raise ColiMoeError(rc, where)
    return rc


def make_desc(T, H, I, E, K, I_shared=0, norm_topk=1, routed_scale=1.0, routed_fmt=COLI_FMT_INT4,
              shared_fmt=COLI_FMT_INT4, ksel=0, top_p=0.0, group_size=0, idot=0):
    return coli_moe_desc(T, H, I, E, K, I_shared, norm_topk, routed_scale, routed_fmt, shared_fmt,
                         ksel, top_p, group_size, idot)


def coli_moe_workspace_bytes(desc) -> int:
    return int(_lib.coli_moe_workspace_bytes(ctypes.byref(desc)))


def coli_moe_route(desc, x, W_r, bias, idx, w, keff=None, counts=None, offsets=None, perm=None,
                   ws=None, ws_bytes=0, stream=None, raise_on_error=True):
    rc = _lib.coli_moe_route(ctypes.byref(desc), _ptr(x), _ptr(W_r), _ptr(bias), _ptr(idx), _ptr(w),
                             _ptr(keff), _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(ws),
                             ws_bytes, _stream(stream))
    return _check(rc, "coli_moe_route", raise_on_error)


def coli_moe_forward(desc, x, W_r, bias, experts, shared, out, idx_out=None, w_out=None, ws=None,
                     ws_bytes=0, stream=None, raise_on_error=True):
    sh = ctypes.byref(shared) if shared is not None else None
    rc = _lib.coli_moe_forward(ctypes.byref(desc), _ptr(x), _ptr(W_r), _ptr(bias), _ptr(experts), sh,
                               _ptr(out), _ptr(idx_out), _ptr(w_out), _ptr(ws), ws_bytes,
                               _stream(stream))
    return _check(rc, "coli_moe_forward", raise_on_error)


def coli_moe_forward_profiled(desc, x, W_r, bias, experts, shared, out, events, ws=None,
                              ws_bytes=0, stream=None, raise_on_error=True):
    """events: five torch.cuda.Event objects (already created, e.g. recorded once) or raw
    cudaEvent_t handles; recorded at the stage boundaries."""
    handles = [e if isinstance(e, int) else e.cuda_event for e in events]
    arr = (ctypes.c_void_p * len(handles))(*handles)
    sh = ctypes.byref(shared) if shared is not None else None
    rc = _lib.coli_moe_forward_profiled(ctypes.byref(desc), _ptr(x), _ptr(W_r), _ptr(bias),
                                        _ptr(experts), sh, _ptr(out), arr, len(handles), _ptr(ws),
                                        ws_bytes, _stream(stream))
    return _check(rc, "coli_moe_forward_profiled", raise_on_error)


def coli_moe_forward_tail(desc, resid, norm_w, eps, W_r, bias, experts, shared, out, idx_out=None,
                          w_out=None, ws=None, ws_bytes=0, stream=None, raise_on_error=True):
    sh = ctypes.byref(shared) if shared is not None else None
    rc = _lib.coli_moe_forward_tail(ctypes.byref(desc), _ptr(resid), _ptr(norm_w), float(eps), _ptr(W_r),
                                    _ptr(bias), _ptr(experts), sh, _ptr(out), _ptr(idx_out), _ptr(w_out),
                                    _ptr(ws), ws_bytes, _stream(stream))
    return _check(rc, "coli_moe_forward_tail", raise_on_error)


def coli_moe_rmsnorm(resid, norm_w, eps, xn, T, H, stream=None, raise_on_error=True):
    rc = _lib.coli_moe_rmsnorm(_ptr(resid), _ptr(norm_w), float(eps), _ptr(xn), T, H, _stream(stream))
    return _check(rc, "coli_moe_rmsnorm", raise_on_error)


def coli_moe_forward_host(desc, x_host, W_r, bias, experts, shared, out_host, ws=None, ws_bytes=0,
                          stream=None, raise_on_error=True):
    sh = ctypes.byref(shared) if shared is not None else None
    rc = _lib.coli_moe_forward_host(ctypes.byref(desc), _ptr(x_host), _ptr(W_r), _ptr(bias),
                                    _ptr(experts), sh, _ptr(out_host), _ptr(ws), ws_bytes,
                                    _stream(stream))
    return _check(rc, "coli_moe_forward_host", raise_on_error)


def coli_moe_qgemv(fmt, W, s, x, y, O, In, T, stream=None, raise_on_error=True):
    rc = _lib.coli_moe_qgemv(fmt, _ptr(W), _ptr(s), _ptr(x), _ptr(y), O, In, T, _stream(stream))
    return _check(rc, "coli_moe_qgemv", raise_on_error)


def coli_moe_qgemv_grouped(W, s, group_size, x, y, O, In, T, stream=None, raise_on_error=True):
    rc = _lib.coli_moe_qgemv_grouped(_ptr(W), _ptr(s), group_size, _ptr(x), _ptr(y), O, In, T, _stream(stream))
    return _check(rc, "coli_moe_qgemv_grouped", raise_on_error)


def coli_moe_check(ws, stream=None, raise_on_error=True):
    rc = _lib.coli_moe_check(_ptr(ws), _stream(stream))
    return _check(rc, "coli_moe_check", raise_on_error)


def coli_moe_strerror(code) -> str:
    return _lib.coli_moe_strerror(code).decode()


def coli_moe_forward_noalloc(desc, x, W_r, bias, experts, shared, out, stream=None,
                             raise_on_error=True):
    """The block without a workspace, for callers that cannot allocate device memory: the
    library's fixed COLI_MOE_NOALLOC_SCRATCH_BYTES device array serves as scratch. Calls share
    that array, so calls that overlap on the GPU race; the first call on a device should come
    before any stream capture."""
    sh = ctypes.byref(shared) if shared is not None else None
    rc = _lib.coli_moe_forward_noalloc(ctypes.byref(desc), _ptr(x), _ptr(W_r), _ptr(bias),
                                       _ptr(experts), sh, _ptr(out), _stream(stream))
    return _check(rc, "coli_moe_forward_noalloc", raise_on_error)


def coli_moe_noalloc_check(stream=None, raise_on_error=True):
    """Reads and clears the error word of coli_moe_forward_noalloc's fixed array (synchronises
    the stream)."""
    rc = _lib.coli_moe_noalloc_check(_stream(stream))
    return _check(rc, "coli_moe_noalloc_check", raise_on_error)
