"""Seeded synthetic inputs for the quantized MoE block.

This module only draws random numbers into the shapes and value distributions of the five
workloads; it holds none of the block's arithmetic (no routing, no dequantisation, no GEMV).
Both the CUDA library's tests/benchmark and the CPU oracle's tests take their inputs from here.

Weights of one expert live in one contiguous "slab" (the same idea as the coalesced per-expert
read of glm.c's expert loader): gate [I][row_bytes(H)], up [I][row_bytes(H)],
down [H][row_bytes(I)], then the fp32 row scales of gate [I], up [I] and down [H]. Every section
starts on a 256-byte boundary. All routed experts form one [E, slab_bytes] array.

Distributions (one numpy PCG64 stream per seed):
  x      ~ N(0, 1)                        [T, H] fp32
  W_r    ~ N(0, 1/H)                      [E, H] fp32
  bias   ~ U(-0.1, 0.1)                   [E]    (+ a Zipf(s=1.1) term over a seeded expert
                                                   permutation for the skewed workload)
  int8   weight bytes uniform in [-127, 127], row scale ~ U(0.5, 1.5) / (127 * sqrt(in))
  int4   weight bytes uniform in [0, 255] (both nibbles uniform in 0..15),
         row scale ~ U(0.5, 1.5) / (8 * sqrt(in))
  int2   weight bytes uniform in [0, 255], row scale ~ U(0.5, 1.5) / (2 * sqrt(in))
  int4-grouped (format 4): int4 bytes, one scale ~ U(0.5, 1.5) / (8 * sqrt(in)) per group of
         `group_size` inputs of a row, stored [rows][ceil(in / group_size)]
where "in" is the number of input features of that matrix (H for gate/up, I for down).
"""
from __future__ import annotations

import numpy as np

FMT_INT8, FMT_INT4, FMT_INT2, FMT_INT4G = 1, 2, 3, 4
_QMAX = {FMT_INT8: 127.0, FMT_INT4: 8.0, FMT_INT2: 2.0, FMT_INT4G: 8.0}
ALIGN = 256

# Zipf amplitude added to the router bias of the skewed continuous-batch workload. Chosen so
# that the 20% most-used experts receive about half of the T*K assignments (checked by a test).
ZIPF_S = 1.1
ZIPF_ALPHA = 0.1

CONFIGS = {
    0: dict(name="tiny-int8", T=4, H=256, I=128, E=8, K=2, I_shared=128, norm_topk=1,
            routed_scale=2.5, routed_fmt=FMT_INT8, shared_fmt=FMT_INT8, zipf=False),
    1: dict(name="small-decode-int4", T=1, H=2048, I=1024, E=64, K=8, I_shared=0, norm_topk=1,
            routed_scale=1.0, routed_fmt=FMT_INT4, shared_fmt=FMT_INT4, zipf=False),
    2: dict(name="large-decode-int4", T=1, H=6144, I=2048, E=256, K=8, I_shared=2048, norm_topk=1,
            routed_scale=2.5, routed_fmt=FMT_INT4, shared_fmt=FMT_INT4, zipf=False),
    3: dict(name="batch32-decode-int4-shared-int8", T=32, H=6144, I=2048, E=256, K=8, I_shared=2048,
            norm_topk=1, routed_scale=2.5, routed_fmt=FMT_INT4, shared_fmt=FMT_INT8, zipf=True),
    4: dict(name="prefill-int4", T=2048, H=6144, I=2048, E=256, K=8, I_shared=2048, norm_topk=1,
            routed_scale=2.5, routed_fmt=FMT_INT4, shared_fmt=FMT_INT4, zipf=False),
}


def seed_for(cfg_id: int) -> int:
    return 0xC0110000 + int(cfg_id)


def config(cfg_id: int, **over) -> dict:
    c = dict(CONFIGS[cfg_id])
    c.update(over)
    return c


def row_bytes(fmt: int, n: int) -> int:
    if fmt == FMT_INT8:
        return n
    if fmt in (FMT_INT4, FMT_INT4G):
        return (n + 1) // 2
    if fmt == FMT_INT2:
        return (n + 3) // 4
    raise ValueError(f"unknown weight format {fmt}")


def _up(n: int) -> int:
    return (n + ALIGN - 1) // ALIGN * ALIGN


def groups(fmt: int, n: int, gs: int) -> int:
    """Scales per row of a matrix with n inputs: ceil(n / gs) for int4-grouped, else 1."""
    return (n + gs - 1) // gs if fmt == FMT_INT4G else 1


def slab_layout(fmt: int, H: int, I: int, gs: int = 0) -> dict:
    """Byte offsets of the six sections of one expert slab, and the slab size."""
    rb_h, rb_i = row_bytes(fmt, H), row_bytes(fmt, I)
    ng_h, ng_i = groups(fmt, H, gs), groups(fmt, I, gs)
    off = {}
    p = 0
    for key, nbytes in (("gate_w", I * rb_h), ("up_w", I * rb_h), ("down_w", H * rb_i),
                        ("gate_s", 4 * I * ng_h), ("up_s", 4 * I * ng_h), ("down_s", 4 * H * ng_i)):
        off[key] = p
        p += _up(nbytes)
    off["bytes"] = p
    off["rb_h"], off["rb_i"] = rb_h, rb_i
    off["ng_h"], off["ng_i"] = ng_h, ng_i
    return off


def _fill_weights(rng, fmt: int, out: np.ndarray) -> None:
    if fmt == FMT_INT8:
        out[...] = rng.integers(-127, 128, size=out.shape, dtype=np.int8).view(np.uint8)
    else:
        out[...] = rng.integers(0, 256, size=out.shape, dtype=np.uint8)


def _scales(rng, fmt: int, n: int, fan_in: int) -> np.ndarray:
    return (rng.uniform(0.5, 1.5, size=n) / (_QMAX[fmt] * np.sqrt(fan_in))).astype(np.float32)


def expert_views(slab_row: np.ndarray, fmt: int, H: int, I: int, gs: int = 0) -> dict:
    """Numpy views of the six sections of one expert slab (no copy). Scales are flat:
    [rows * groups] (row-major [rows][groups] for int4-grouped)."""
    L = slab_layout(fmt, H, I, gs)
    rb_h, rb_i, ng_h, ng_i = L["rb_h"], L["rb_i"], L["ng_h"], L["ng_i"]
    return {
        "gate_w": slab_row[L["gate_w"]:L["gate_w"] + I * rb_h].reshape(I, rb_h),
        "up_w": slab_row[L["up_w"]:L["up_w"] + I * rb_h].reshape(I, rb_h),
        "down_w": slab_row[L["down_w"]:L["down_w"] + H * rb_i].reshape(H, rb_i),
        "gate_s": slab_row[L["gate_s"]:L["gate_s"] + 4 * I * ng_h].view(np.float32),
        "up_s": slab_row[L["up_s"]:L["up_s"] + 4 * I * ng_h].view(np.float32),
        "down_s": slab_row[L["down_s"]:L["down_s"] + 4 * H * ng_i].view(np.float32),
    }


def make_slabs(rng, n: int, fmt: int, H: int, I: int, gs: int = 0) -> np.ndarray:
    """n expert slabs [n, slab_bytes] of random packed weights and scales."""
    L = slab_layout(fmt, H, I, gs)
    slabs = np.zeros((n, L["bytes"]), np.uint8)
    for e in range(n):
        v = expert_views(slabs[e], fmt, H, I, gs)
        for key in ("gate_w", "up_w", "down_w"):
            _fill_weights(rng, fmt, v[key])
        v["gate_s"][:] = _scales(rng, fmt, I * L["ng_h"], H)
        v["up_s"][:] = _scales(rng, fmt, I * L["ng_h"], H)
        v["down_s"][:] = _scales(rng, fmt, H * L["ng_i"], I)
    return slabs


def draw_x(rng, T: int, H: int) -> np.ndarray:
    return rng.standard_normal((T, H)).astype(np.float32)


def zipf_bias_term(rng, E: int) -> np.ndarray:
    perm = rng.permutation(E)
    return (ZIPF_ALPHA * (perm + 1.0) ** (-ZIPF_S)).astype(np.float32)


def make_router(rng, cfg: dict):
    E, H = cfg["E"], cfg["H"]
    Wr = (rng.standard_normal((E, H)) / np.sqrt(H)).astype(np.float32)
    bias = rng.uniform(-0.1, 0.1, size=E).astype(np.float32)
    if cfg.get("zipf"):
        bias = (bias + zipf_bias_term(rng, E)).astype(np.float32)
    return Wr, bias


def make_block(cfg, seed=None, T=None, row_filter=None, max_redraws=1000) -> dict:
    """All inputs of one block call.

    cfg: a workload id (0..4) or a config dict.  T overrides the token count.
    row_filter: optional callable(x, Wr, bias) -> bool mask of acceptable rows; rejected rows
    are redrawn from the same stream (used by tests to demand a margin between router scores).
    """
    if not isinstance(cfg, dict):
        cid = int(cfg)
        cfg = config(cid)
        seed = seed_for(cid) if seed is None else seed
    cfg = dict(cfg)
    if T is not None:
        cfg["T"] = int(T)
    rng = np.random.Generator(np.random.PCG64(0 if seed is None else seed))
    H, I, E = cfg["H"], cfg["I"], cfg["E"]
    Wr, bias = make_router(rng, cfg)
    gs = int(cfg.get("group_size", 0))
    slabs = make_slabs(rng, E, cfg["routed_fmt"], H, I, gs)
    routed = [expert_views(slabs[e], cfg["routed_fmt"], H, I, gs) for e in range(E)]
    shared_slab, shared = None, None
    if cfg["I_shared"] > 0:
        shared_slab = make_slabs(rng, 1, cfg["shared_fmt"], H, cfg["I_shared"], gs)
        shared = expert_views(shared_slab[0], cfg["shared_fmt"], H, cfg["I_shared"], gs)
    x = draw_x(rng, cfg["T"], H)
    if row_filter is not None:
        for _ in range(max_redraws):
            ok = np.asarray(row_filter(x, Wr, bias), dtype=bool)
            if ok.all():
                break
            bad = np.nonzero(~ok)[0]
            x[bad] = draw_x(rng, len(bad), H)
        else:
            raise RuntimeError("make_block: could not draw rows that pass the filter")
    return dict(cfg=cfg, seed=seed, x=x, Wr=Wr, bias=bias, routed_slabs=slabs, routed=routed,
                shared_slab=shared_slab, shared=shared)


def make_x_batches(cfg: dict, seed: int, n: int, T=None) -> np.ndarray:
    """n independent activation batches [n, T, H] from their own stream (benchmark rotation)."""
    rng = np.random.Generator(np.random.PCG64(seed ^ 0x5EED5EED))
    T = cfg["T"] if T is None else T
    return rng.standard_normal((n, T, cfg["H"])).astype(np.float32)
