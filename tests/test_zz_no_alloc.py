"""coli_moe_forward_noalloc — the forward for callers that cannot allocate device memory.

Such callers (a host whose memory pool owns the whole device, a plugin that may only launch
work, a loop that must never enter the allocator) cannot hand the library a workspace. This
entry point runs the same block on a fixed scratch array inside the library's device image.
The tests compare it with coli_moe_forward on the same inputs, two calls in a row (the second
on fresh activations, so stale scratch from the first call would show), on every path the
fixed array can serve: the single-token kernel, the token-group kernel, the tensor-core GEMMs
(T > 64, which reuse the scratch for bf16 activations), the general kernels of an
int4-grouped block and the single-token kernel on int4-grouped weights and on int8 activations
(IDOT). Both entry points run the same deterministic kernels, so the outputs must
be identical bit for bit; the fixed array's error word must read clear afterwards. A
description needing more than the fixed scratch is refused. The tests build their own inputs,
so they pass alone in a fresh process as well as after the rest of the suite; the file name
keeps them last in collection order.
"""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

CASES = [
    ("token-group", dict(T=6, H=512, I=256, E=16, K=3, I_shared=128, norm_topk=1, routed_scale=2.5,
                         routed_fmt=2, shared_fmt=1, zipf=False)),
    ("one-token", synth.config(1)),
    ("tensor-core-gemms", dict(T=80, H=512, I=256, E=16, K=2, I_shared=128, norm_topk=1, routed_scale=2.5,
                               routed_fmt=2, shared_fmt=2, zipf=False)),
    ("int4-grouped", dict(T=5, H=512, I=256, E=12, K=3, I_shared=128, norm_topk=1, routed_scale=2.5,
                          routed_fmt=4, shared_fmt=4, group_size=64, zipf=False)),
    ("int4-grouped-one-token", dict(T=1, H=512, I=256, E=12, K=3, I_shared=128, norm_topk=1, routed_scale=2.5,
                                    routed_fmt=4, shared_fmt=4, group_size=64, zipf=False)),
    ("idot-one-token", dict(T=1, H=512, I=256, E=12, K=3, I_shared=128, norm_topk=1, routed_scale=2.5,
                            routed_fmt=2, shared_fmt=1, idot=1, zipf=False)),
]


@pytest.mark.parametrize("name,cfg", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_forward_twice(name, cfg):
    assert torch.cuda.is_available(), "needs a CUDA device"
    import quantized_expert_decode_gb300 as q
    from quantized_expert_decode_gb300.device import DeviceBlock

    blk = synth.make_block(cfg, seed=4242)
    dev = DeviceBlock(blk)
    assert q.coli_moe_workspace_bytes(dev.desc) <= q.COLI_MOE_NOALLOC_SCRATCH_BYTES
    T, H = cfg["T"], cfg["H"]
    xs = synth.make_x_batches(cfg, 4242, 2)
    for call in range(2):  # two calls in a row share the fixed scratch
        x = torch.from_numpy(xs[call]).cuda()
        ref = torch.empty((T, H), dtype=torch.float32, device="cuda")
        got = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
        q.coli_moe_forward(dev.desc, x, dev.Wr, dev.bias, dev.table, dev.shared, ref,
                           ws=dev.ws, ws_bytes=dev.ws_bytes)
        q.coli_moe_check(dev.ws)
        q.coli_moe_forward_noalloc(dev.desc, x, dev.Wr, dev.bias, dev.table, dev.shared, got)
        q.coli_moe_noalloc_check()  # raises if a kernel flagged an error in the fixed array
        r = ref.cpu().numpy()
        g = got.cpu().numpy()
        assert np.all(np.isfinite(g)), (name, call)
        assert np.array_equal(g, r), (name, call, float(np.max(np.abs(g.astype(np.float64) - r))))


def test_noalloc_refuses_oversize_description():
    import quantized_expert_decode_gb300 as q
    # at these shapes the fixed array admits T <= 89
    fits = q.make_desc(T=89, H=6144, I=2048, E=256, K=8, I_shared=2048, routed_scale=2.5)
    big = q.make_desc(T=90, H=6144, I=2048, E=256, K=8, I_shared=2048, routed_scale=2.5)
    assert q.coli_moe_workspace_bytes(fits) <= q.COLI_MOE_NOALLOC_SCRATCH_BYTES
    assert q.coli_moe_workspace_bytes(big) > q.COLI_MOE_NOALLOC_SCRATCH_BYTES
    dummy = torch.empty(16, dtype=torch.float32, device="cuda")
    ex = q.coli_moe_expert(*[dummy.data_ptr()] * 6)
    rc = q.coli_moe_forward_noalloc(big, dummy, dummy, dummy, dummy, ex, dummy,
                                    raise_on_error=False)
    assert rc == q.COLI_MOE_EWORKSPACE
