#!/usr/bin/env python
"""Benchmark of the quantized MoE feed-forward block on GB300.

A step is one whole block (router, selection, buckets, gate/up + SiLU*mul, down, combine) over
one batch of synthetic tokens, through the C ABI. Default workload: large decode at GLM-5.2
block shapes (T=1, H=6144, I=2048, 256 int4 experts top-8 + an int4 shared expert of 2048,
~176.5 MB of packed weights, scales and router weights per token). Inputs are resident in HBM;
activations rotate through 16 pre-drawn batches and a 512 MiB buffer is written between timed
steps so that no step finds its expert weights in the 129 MB L2.

Prints one JSON line (rank 0). `--impl reference` times the CPU oracle instead, on the host
cores, on the same workload.

Under torchrun (N > 1) every rank runs an independent replica on its own GPU (the block has no
cross-GPU exchange on this path): value = tokens of all ranks / max time over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "MoE-block tokens/s"
UNIT = "tokens/s"
ROTATE = 16
FLUSH_BYTES = 512 << 20
DECODE_MAX_T = 64  # the library runs T <= 64 as one persistent decode kernel

# DRAM bytes (read + write) per launch of the roofline kernel measured by ncu
# (dram__bytes_read.sum + dram__bytes_write.sum), keyed by workload, with the hash of the kernel
# sources they were taken on; a changed kernel reports null until it is measured again.
NCU_TRAFFIC = {
    # moe_decode1_kernel, small decode: a full-size capture (single-pass DRAM counters)
    1: {"bytes": 25958656 + 0, "src": "0e3695ff713bdd7e"},
    # moe_decode1_kernel, large decode: a full-size capture (256 experts; single-pass DRAM
    # counters) of a call whose algorithmic bytes are 176530432
    2: {"bytes": 176697600 + 2807040, "src": "0e3695ff713bdd7e"},
    # moe_decode_kernel, batch-32 decode: a full-size capture (single-pass DRAM counters) of a
    # call whose algorithmic bytes were 2402205696; its ratio applies to each bench launch
    3: {"ratio": (2456358656 + 12191232) / 2402205696, "src": "0e3695ff713bdd7e"},
    # moe_prefill_tc_kernel, prefill: the gate/up GEMM launch, a full-size capture (single-pass
    # DRAM counters; 248 routed experts + the shared one, the f16 activations and h)
    4: {"bytes": 3376586240 + 68475904, "src": "8f8ba21abc55adc7"},
}


def recorded_traffic(cfg, cid, general, src, mean_kernel_bytes):
    """DRAM bytes per launch of the dominant kernel from the recorded ncu captures, or None.
    The captures are of the plain workloads (per-row scales, exact products) on the general-free
    paths: a variant's kernel instance (int4-grouped, IDOT) or the general kernels read other
    bytes, and a capture taken on other kernel sources (src) no longer describes this kernel.
    A full-size capture gives bytes per launch; one of a smaller case gives the ratio of DRAM
    bytes to algorithmic bytes, applied to this run's mean launch."""
    variant = bool(cfg.get("group_size", 0)) or bool(cfg.get("idot", 0))
    tr = None if (general or variant) else NCU_TRAFFIC.get(cid)
    if not tr or tr["src"] != src:
        return None
    return tr["bytes"] if "bytes" in tr else tr["ratio"] * mean_kernel_bytes


def kernel_source_hash(kind: str = "decode") -> str:
    """Hash of the sources a roofline kernel is compiled from (its translation units and
    everything they include): the persistent decode kernels, or the prefill GEMM."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "quantized_expert_decode_gb300", "csrc")
    names = (("prefill.cu", "tc.cuh", "kernels.h", "common.cuh", "ptx.cuh") if kind == "prefill" else
             ("decode.cu", "decode1.cu", "decode_parts.cuh", "idot.cuh", "mma.cuh", "qdot.cuh", "select.cuh",
              "kernels.h", "common.cuh", "ptx.cuh"))
    paths = [os.path.join(csrc, n) for n in names]
    paths.append(os.path.join(ROOT, "include", "colimoe.h"))
    for path in paths:
        with open(path, "rb") as f:
            h.update(_code_only(f.read().decode()).encode())
    return h.hexdigest()[:16]


def _code_only(src: str) -> str:
    """C/C++ source without comments and blank lines (a comment edit does not change a kernel)."""
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    lines = (re.sub(r"//.*$", "", l).rstrip() for l in src.splitlines())
    return "\n".join(l for l in lines if l)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="colimoe", choices=["colimoe", "reference"])
    ap.add_argument("--workload", type=int, default=2, choices=sorted(synth.CONFIGS))
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU work budget of the oracle baseline sample")
    ap.add_argument("--calls", type=int, default=0,
                    help="profiling mode: only run this many forward calls (L2 flushed between "
                         "them) and exit; for ncu captures")
    ap.add_argument("--experts", type=int, default=0, help="profiling mode: override E")
    ap.add_argument("--tokens", type=int, default=0, help="profiling mode: override T")
    ap.add_argument("--idot", action="store_true",
                    help="int8 and int4 experts through the IDOT kernels (int8 activations, lossy)")
    ap.add_argument("--tail", action="store_true",
                    help="also time the block as a decoder-layer tail (RMSNorm folded in, residual "
                         "added) against the same work as a separate RMSNorm launch plus the block")
    ap.add_argument("--group-size", type=int, default=0,
                    help="run the workload's int4 experts as int4-grouped tensors (format 4) with "
                         "this many inputs per scale")
    return ap.parse_args()


def run_calls(args):
    """Profiling mode: N plain forward calls of the workload (optionally with fewer experts or
    tokens, to keep an ncu capture small), a 64 MiB buffer written between them."""
    import torch
    import quantized_expert_decode_gb300 as q
    from quantized_expert_decode_gb300.device import DeviceBlock
    over = {}
    if args.experts:
        over["E"] = args.experts
    if args.tokens:
        over["T"] = args.tokens
    cfg = workload_cfg(args, **over)
    blk = synth.make_block(cfg, seed=synth.seed_for(args.workload))
    dev = DeviceBlock(blk)
    T, H = cfg["T"], cfg["H"]
    xs = torch.from_numpy(synth.make_x_batches(cfg, 7, 4)).cuda()
    out = torch.empty((T, H), dtype=torch.float32, device="cuda")
    flush = torch.empty(16 << 20, dtype=torch.float32, device="cuda")
    for i in range(args.calls):
        flush.fill_(float(i))
        q.coli_moe_forward(dev.desc, xs[i % 4], dev.Wr, dev.bias, dev.table, dev.shared, out,
                           ws=dev.ws, ws_bytes=dev.ws_bytes)
    q.coli_moe_check(dev.ws)
    torch.cuda.synchronize()
    # distinct experts of each call and the algorithmic bytes of its decode kernel (for scaling
    # the DRAM traffic of a capture to the benchmark's launches)
    K = cfg["K"]
    idx = torch.empty((T, K), dtype=torch.int32, device="cuda")
    wts = torch.empty((T, K), dtype=torch.float32, device="cuda")
    active, kbytes = [], []
    for i in range(args.calls):
        q.coli_moe_route(dev.desc, xs[i % 4], dev.Wr, dev.bias, idx, wts, None, None, None, None,
                         dev.ws, dev.ws_bytes)
        ids = idx.cpu().numpy()
        active.append(int(len(np.unique(ids[ids >= 0]))))
        kbytes.append(decode_kernel_bytes(cfg, T, active[-1]))
    print(json.dumps({"calls": args.calls, "workload": cfg["name"], "T": T, "E": cfg["E"],
                      "out_abs_sum": float(out.abs().sum()), "active": active,
                      "decode_kernel_bytes": kbytes}))


# ------------------------------------------------------------------ algorithmic bytes
def workload_cfg(args, **over):
    """The workload's config; with --group-size its int4 experts become int4-grouped."""
    cfg = synth.config(args.workload, **over)
    gs = getattr(args, "group_size", 0)
    if gs:
        g = {f: (synth.FMT_INT4G if cfg[f] == synth.FMT_INT4 else cfg[f]) for f in ("routed_fmt", "shared_fmt")}
        cfg.update(g, group_size=gs, name=f"{cfg['name']}-grouped{gs}")
    if getattr(args, "idot", False):
        cfg.update(idot=1, name=f"{cfg['name']}-idot")
    return cfg


def expert_bytes(fmt, H, I, gs=0):
    """(gate+up bytes, down bytes) of one expert: packed weights + fp32 scales (one per row, or
    one per group of gs inputs for int4-grouped)."""
    gu = 2 * (I * synth.row_bytes(fmt, H) + 4 * I * synth.groups(fmt, H, gs))
    dn = H * synth.row_bytes(fmt, I) + 4 * H * synth.groups(fmt, I, gs)
    return gu, dn


def step_bytes(cfg, n_active):
    """Algorithmic bytes one block call must read: each distinct selected expert once, the
    shared expert, the router weights and bias (activations excluded)."""
    gs = cfg.get("group_size", 0)
    gu, dn = expert_bytes(cfg["routed_fmt"], cfg["H"], cfg["I"], gs)
    b = n_active * (gu + dn)
    gu_s = dn_s = 0
    if cfg["I_shared"] > 0:
        gu_s, dn_s = expert_bytes(cfg["shared_fmt"], cfg["H"], cfg["I_shared"], gs)
    router = cfg["E"] * cfg["H"] * 4 + cfg["E"] * 4
    return dict(total=b + gu_s + dn_s + router, experts=b + gu_s + dn_s,
                gateup=n_active * gu + gu_s, down=n_active * dn + dn_s)


def decode_kernel_bytes(cfg, T, n_active):
    """Algorithmic bytes of one persistent decode launch: the experts it streams, plus the
    router weights when the launch computes the logits itself (T <= 8)."""
    b = step_bytes(cfg, n_active)
    return b["experts"] + (b["total"] - b["experts"] if T <= 8 else 0)


def load_peaks(kind="hbm"):
    """(peak, 'measured'|'fallback'): HBM copy GB/s, or dense bf16 TFLOP/s (burst)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return (float(p["hbm_gbs"]) if kind == "hbm" else float(p["bf16_tflops"])), "measured"
    except Exception:
        return (6800.0 if kind == "hbm" else 1900.0), "fallback"


def gateup_flops(cfg, assignments):
    """FLOPs of the gate and up products of one block call (2 per multiply-add)."""
    return 2 * cfg["H"] * 2 * (assignments * cfg["I"] + cfg["T"] * cfg["I_shared"])


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "200"], stdout=open(self.path, "w"),
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ distributed plumbing
def dist_init(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def dist_max(v, world, device="cpu"):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_sum(v, world, device="cpu"):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------ CPU oracle (baseline)
def oracle_sample(cfg, blk, xs, budget_s):
    """Time the CPU oracle, as it stands, on whole tokens of the workload until `budget_s`
    seconds of work are done (at least one token). Returns (tokens/s, tokens, seconds)."""
    import oracle
    oracle.build()
    flat = xs.reshape(-1, cfg["H"])
    n, t0 = 0, time.perf_counter()
    while True:
        oracle.moe_forward(blk, x=flat[n % len(flat)][None, :])
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            return n / el, n, el


def cpu_cores_used():
    return 1  # the oracle is single-threaded C


# ------------------------------------------------------------------ the GPU arm
def run_colimoe(args, rank, world, local):
    import torch
    import quantized_expert_decode_gb300 as q
    from quantized_expert_decode_gb300.device import DeviceBlock

    dev_name = f"cuda:{local}"
    torch.cuda.set_device(local)
    cid = args.workload
    cfg = workload_cfg(args)
    blk = synth.make_block(cfg, seed=synth.seed_for(cid))
    dev = DeviceBlock(blk, device=dev_name)
    T, H, K = cfg["T"], cfg["H"], cfg["K"]
    xs_np = synth.make_x_batches(cfg, synth.seed_for(cid) + 97 * rank, ROTATE)
    xs = torch.from_numpy(xs_np).to(dev_name)
    out = torch.empty((T, H), dtype=torch.float32, device=dev_name)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev_name)
    stream = torch.cuda.current_stream()

    def events():
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        for e in evs:
            e.record(stream)  # creates the underlying cudaEvent_t
        return evs

    step_ev = [events() for _ in range(args.steps)]
    warm_ev = events()
    torch.cuda.synchronize()

    for i in range(args.warmup):
        flush.fill_(float(i))
        q.coli_moe_forward_profiled(dev.desc, xs[i % ROTATE], dev.Wr, dev.bias, dev.table,
                                    dev.shared, out, warm_ev, dev.ws, dev.ws_bytes, stream)
    q.coli_moe_check(dev.ws, stream)
    torch.cuda.synchronize()
    dist_barrier(world)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    for i in range(args.steps):
        flush.fill_(float(i))
        q.coli_moe_forward_profiled(dev.desc, xs[i % ROTATE], dev.Wr, dev.bias, dev.table,
                                    dev.shared, out, step_ev[i], dev.ws, dev.ws_bytes, stream)
    torch.cuda.synchronize()
    dist_barrier(world)
    time.sleep(0.2)
    clk = clocks.stop()
    q.coli_moe_check(dev.ws, stream)

    stage = np.array([[step_ev[i][j].elapsed_time(step_ev[i][j + 1]) for j in range(4)]
                      for i in range(args.steps)])  # ms
    # decode (T <= 64) does all its work between events 0 and 2 (the counter memset, the router
    # launch for T > 8, the persistent kernel); events 3 and 4 follow with no work between them
    # and only add the recording overhead of an event pair, so they are not part of the step
    # int4-grouped and IDOT blocks run the single-token kernel at T = 1 (not both at once) and
    # the general launches (router, gate/up, down, combine) for other T
    grouped = bool(cfg.get("group_size", 0)) and synth.FMT_INT4G in (cfg["routed_fmt"], cfg["shared_fmt"])
    idot = bool(cfg.get("idot", 0))
    general = (T != 1 and (grouped or idot)) or (grouped and idot)
    fused = T <= DECODE_MAX_T and not general
    step_ms = stage[:, :2].sum(axis=1) if fused else stage.sum(axis=1)
    total_s = float(step_ms.sum()) / 1e3
    # distinct routed experts each rotated batch reads (from the library's own routing)
    idx = torch.empty((T, K), dtype=torch.int32, device=dev_name)
    wts = torch.empty((T, K), dtype=torch.float32, device=dev_name)
    uniq = []
    for b in range(ROTATE):
        q.coli_moe_route(dev.desc, xs[b], dev.Wr, dev.bias, idx, wts, None, None, None, None,
                         dev.ws, dev.ws_bytes, stream)
        ids = idx.cpu().numpy()
        uniq.append(len(np.unique(ids[ids >= 0])))
    n_active = np.array([uniq[i % ROTATE] for i in range(args.steps)])
    max_s = dist_max(total_s, world, dev_name if world > 1 else "cpu")
    tokens = dist_sum(T * args.steps, world, dev_name if world > 1 else "cpu")
    value = tokens / max_s

    bytes_per = [step_bytes(cfg, int(u)) for u in n_active]
    hbm_peak, peak_kind = load_peaks()
    if fused:
        # one persistent kernel does the whole block (T = 1: the single-token kernel); for
        # T > 8 the router logits come from a separate launch before it
        kname = "moe_decode1_kernel" if T == 1 else "moe_decode_kernel"
        k_ms = stage[:, 1]
        k_bytes = np.array([decode_kernel_bytes(cfg, T, int(u)) for u in n_active], np.float64)
        launches = 1 if T <= 8 else 2
    elif general:
        kname = "gateup_kernel"
        k_ms = stage[:, 1]
        k_bytes = np.array([b["gateup"] for b in bytes_per], np.float64)
        launches = 6  # router partial, select, bucket, gate/up, down, combine
    else:
        # T > 64: the expert products run as tcgen05 GEMMs; the gate/up launch (with its bf16
        # activation pre-pass) is the dominant kernel and its bound is the tensor pipe
        kname = "moe_prefill_tc_kernel"
        k_ms = stage[:, 1]
        k_bytes = np.array([b["gateup"] for b in bytes_per], np.float64)
        launches = 7  # router partial, select, bucket, pre-pass, two GEMMs, combine
    achieved = float(k_bytes.sum() / (k_ms.sum() / 1e3) / 1e9)
    hbm_bound = fused or general
    if not hbm_bound:
        flops = gateup_flops(cfg, T * K)
        tc_peak, tc_kind = load_peaks("tensor")
        tc_achieved = flops / (float(k_ms.mean()) / 1e3) / 1e12
    block_gbs = float(sum(b["total"] for b in bytes_per) / total_s / 1e9)
    expert_gbs = float(sum(b["experts"] for b in bytes_per) / total_s / 1e9)
    src = kernel_source_hash("decode" if fused else "prefill")
    traffic = recorded_traffic(cfg, cid, general, src, float(k_bytes.mean()))

    # end to end through the host-buffer entry point: H2D of x and D2H of out inside each step
    x_host = torch.from_numpy(xs_np).pin_memory()
    out_host = torch.empty((T, H), dtype=torch.float32).pin_memory()
    for i in range(args.warmup):
        q.coli_moe_forward_host(dev.desc, x_host[i % ROTATE], dev.Wr, dev.bias, dev.table,
                                dev.shared, out_host, dev.ws, dev.ws_bytes, stream)
    e2e_s = 0.0
    for i in range(args.steps):
        flush.fill_(float(i))
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        q.coli_moe_forward_host(dev.desc, x_host[i % ROTATE], dev.Wr, dev.bias, dev.table,
                                dev.shared, out_host, dev.ws, dev.ws_bytes, stream)
        e2e_s += time.perf_counter() - t0
    e2e_max = dist_max(e2e_s, world, dev_name if world > 1 else "cpu")

    tail = measure_tail(q, dev, cfg, xs, flush, stream, args) if args.tail else None

    cpu = None
    if rank == 0:
        v, n, el = oracle_sample(cfg, blk, xs_np, args.cpu_seconds)
        cpu = {"value": v, "unit": UNIT, "cores": cpu_cores_used(), "kind": "oracle",
               "sample": f"{n} tokens of the workload's rotating batches, single-threaded C "
                         f"oracle, {el:.1f} s"}

    if rank != 0:
        return None
    k_launch_ms = float(k_ms.mean())
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": float(step_ms.mean()), "higher_is_better": True,
        "step_ms": {"mean": float(step_ms.mean()), "median": float(np.median(step_ms)),
                    "p10": float(np.percentile(step_ms, 10)), "p90": float(np.percentile(step_ms, 90))},
        "scaling": "weak", "vs_baseline": None, "dtype": ("i8 activations x int4/int8 weights, exact int32 sums (IDOT)" if cfg.get("idot", 0)
                  else "f32 (int4/int8 weights dequantised exactly)"),
        "data": "synthetic (seeded; random-init int weights with the workload's shapes)",
        "config": {"workload": f"{cfg['name']} (T={T}, H={H}, I={cfg['I']}, E={cfg['E']}, K={K}, "
                               f"I_shared={cfg['I_shared']})",
                   "tokens_per_step": T, "l2": "512 MiB buffer written between timed steps; "
                                              "activations rotate over 16 batches",
                   "parallelism": f"replicas x{world}"},
        "weight_stream_gbs": expert_gbs, "block_bytes_gbs": block_gbs,
        "frac_of_8tbs": expert_gbs / 8000.0,
        "active_experts_mean": float(np.mean(n_active)),
        "stages_ms": ({"prologue": float(stage[:, 0].mean()), kname: k_launch_ms}
                      if fused else
                      {"route": float(stage[:, 0].mean()), kname: k_launch_ms,
                       "down_kernel": float(stage[:, 2].mean()), "combine": float(stage[:, 3].mean())}
                      if general else
                      {"route": float(stage[:, 0].mean()), "prepass_gateup_gemm": k_launch_ms,
                       "down_gemm": float(stage[:, 2].mean()), "combine": float(stage[:, 3].mean())}),
        "roofline": ({"kernel": kname, "bound": "hbm", "achieved": achieved,
                      "peak": hbm_peak, "peak_kind": peak_kind, "unit": "GB/s",
                      "frac": achieved / hbm_peak, "traffic": traffic,
                      "algorithmic_bytes_per_launch": float(k_bytes.mean()),
                      "avg_launch_ms": k_launch_ms, "kernel_src": src}
                     if hbm_bound else
                     {"kernel": kname, "bound": "tensor", "achieved": tc_achieved,
                      "peak": tc_peak, "peak_kind": tc_kind + " bf16 burst", "unit": "TFLOP/s",
                      "frac": tc_achieved / tc_peak, "traffic": traffic,
                      "algorithmic_flops_per_launch": float(gateup_flops(cfg, T * K)),
                      "weight_bytes_per_launch": float(k_bytes.mean()),
                      "avg_launch_ms": k_launch_ms, "kernel_src": src}),
        "cpu_baseline": cpu,
        "e2e": {"value": tokens / e2e_max, "unit": UNIT, "h2d_bytes_per_step": T * H * 4,
                "d2h_bytes_per_step": T * H * 4},
        "gpu_launches": launches * args.steps,
        **({"layer_tail": tail} if tail else {}),
        "clocks": clk,
    }


def measure_tail(q, dev, cfg, xs, flush, stream, args):
    """The block as a decoder-layer tail: coli_moe_forward_tail (RMSNorm folded into the
    single-token kernel at T = 1) against coli_moe_rmsnorm + coli_moe_forward (one launch more),
    CUDA events around each step, L2 flushed between steps. The residual rows are the workload's
    rotating activation batches times 3; the norm weight is U(0.5, 1.5)."""
    import torch
    T, H = cfg["T"], cfg["H"]
    rng = np.random.default_rng(5)
    nw = torch.from_numpy(rng.uniform(0.5, 1.5, H).astype(np.float32)).to(xs.device)
    resid = xs * 3.0
    out = torch.empty((T, H), dtype=torch.float32, device=xs.device)
    xn = torch.empty((T, H), dtype=torch.float32, device=xs.device)
    eps = 1e-5

    def fused(i):
        q.coli_moe_forward_tail(dev.desc, resid[i % ROTATE], nw, eps, dev.Wr, dev.bias, dev.table, dev.shared,
                                out, ws=dev.ws, ws_bytes=dev.ws_bytes, stream=stream)

    def separate(i):
        q.coli_moe_rmsnorm(resid[i % ROTATE], nw, eps, xn, T, H, stream=stream)
        q.coli_moe_forward(dev.desc, xn, dev.Wr, dev.bias, dev.table, dev.shared, out, ws=dev.ws,
                           ws_bytes=dev.ws_bytes, stream=stream)

    res = {}
    for name, fn in (("fused", fused), ("separate", separate)):
        for i in range(args.warmup):
            fn(i)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for i in range(args.steps):
            flush.fill_(float(i))
            ev[i][0].record(stream)
            fn(i)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        ms = np.array([a.elapsed_time(b) for a, b in ev])
        res[name + "_ms_median"] = float(np.median(ms))
    q.coli_moe_check(dev.ws, stream)
    res["launches_fused"] = 1 if T == 1 else None
    res["saved_ms"] = res["separate_ms_median"] - res["fused_ms_median"]
    return res


# ------------------------------------------------------------------ the reference arm
def run_reference(args, rank, world):
    if rank != 0:
        return None
    cid = args.workload
    cfg = workload_cfg(args)
    blk = synth.make_block(cfg, seed=synth.seed_for(cid))
    xs = synth.make_x_batches(cfg, synth.seed_for(cid), ROTATE)
    import oracle
    oracle.build()
    flat = xs.reshape(-1, cfg["H"])
    # each step: one token of the workload (the oracle's per-token loop), bounded so that
    # warmup + steps finish in minutes
    for i in range(args.warmup):
        oracle.moe_forward(blk, x=flat[i % len(flat)][None, :])
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle.moe_forward(blk, x=flat[i % len(flat)][None, :])
    el = time.perf_counter() - t0
    v = args.steps / el
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 accumulate",
        "data": "synthetic (seeded)",
        "config": {"workload": f"{cfg['name']} (T={cfg['T']}, H={cfg['H']}, I={cfg['I']}, "
                               f"E={cfg['E']}, K={cfg['K']}, I_shared={cfg['I_shared']})",
                   "tokens_per_step": 1, "parallelism": "host cores"},
        "cpu_baseline": {"kind": "oracle", "cores": cpu_cores_used(), "value": v, "unit": UNIT,
                         "sample": f"{args.steps} single tokens of the workload"},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    if args.calls:
        run_calls(args)
        return
    rank, world, local = dist_init(args.gpus)
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_colimoe(args, rank, world, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
