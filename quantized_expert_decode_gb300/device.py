"""Device-memory plumbing with PyTorch: place a block's weights in HBM and build the tables
the C ABI takes (a device array of coli_moe_expert, a host coli_moe_expert for the shared
expert, the workspace). Allocation and copies only; no arithmetic of the block."""
from __future__ import annotations

import numpy as np
import torch

from . import coli_moe_expert, coli_moe_workspace_bytes, make_desc

_SECTIONS = ("gate_w", "up_w", "down_w", "gate_s", "up_s", "down_s")


def slab_offsets(views: dict, slab_row: np.ndarray) -> list:
    base = slab_row.ctypes.data
    return [views[k].ctypes.data - base for k in _SECTIONS]


class DeviceBlock:
    """Weights of one block resident on `device`. ``blk`` is a dict made by ``synth.make_block``
    (or any dict with the same keys: cfg, Wr, bias, routed_slabs, routed, shared_slab, shared)."""

    def __init__(self, blk: dict, device="cuda", ksel=0, top_p=0.0, T=None):
        cfg = blk["cfg"]
        self.cfg = cfg
        self.device = torch.device(device)
        E = cfg["E"]
        self.desc = make_desc(cfg["T"] if T is None else T, cfg["H"], cfg["I"], E, cfg["K"],
                              cfg["I_shared"], cfg["norm_topk"], cfg["routed_scale"],
                              cfg["routed_fmt"], cfg["shared_fmt"], ksel, top_p, cfg.get("group_size", 0),
                              cfg.get("idot", 0))
        self.Wr = torch.from_numpy(np.ascontiguousarray(blk["Wr"])).to(self.device)
        self.bias = torch.from_numpy(np.ascontiguousarray(blk["bias"])).to(self.device)
        slabs = blk["routed_slabs"]
        self.slabs = torch.from_numpy(slabs).to(self.device)
        offs = slab_offsets(blk["routed"][0], slabs[0])
        base = self.slabs.data_ptr()
        stride = slabs.shape[1]
        tab = np.array([[base + e * stride + o for o in offs] for e in range(E)], dtype=np.int64)
        self.table = torch.from_numpy(tab).to(self.device)  # [E, 6] = coli_moe_expert[E]
        self.shared = None
        self.shared_slab = None
        if cfg["I_shared"] > 0:
            self.shared_slab = torch.from_numpy(blk["shared_slab"]).to(self.device)
            so = slab_offsets(blk["shared"], blk["shared_slab"][0])
            sb = self.shared_slab.data_ptr()
            self.shared = coli_moe_expert(*[sb + o for o in so])
        self.weight_bytes_per_expert = int(stride)
        self.alloc_workspace()

    def set_tokens(self, T: int):
        self.desc.T = int(T)
        self.alloc_workspace()

    def alloc_workspace(self):
        n = coli_moe_workspace_bytes(self.desc)
        if n == 0:
            raise ValueError("invalid block description")
        if getattr(self, "ws", None) is None or self.ws.numel() < n:
            self.ws = torch.empty(n, dtype=torch.uint8, device=self.device)
        self.ws_bytes = self.ws.numel()
