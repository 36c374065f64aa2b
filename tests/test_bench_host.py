"""Host-side arithmetic of the benchmark: algorithmic bytes per call, the option that turns a
workload's int4 experts into int4-grouped ones, and the comment-free source hash that keys the
recorded DRAM traffic (no GPU)."""
import argparse

import bench
import synth


def test_expert_bytes_at_glm_shapes():
    # gate+up: 2 * (I rows of H/2 bytes + I fp32 scales); down: H rows of I/2 bytes + H scales
    gu, dn = bench.expert_bytes(synth.FMT_INT4, 6144, 2048)
    assert gu == 2 * (2048 * 3072 + 4 * 2048) == 12599296
    assert dn == 6144 * 1024 + 4 * 6144 == 6316032
    gu8, dn8 = bench.expert_bytes(synth.FMT_INT8, 6144, 2048)
    assert gu8 == 2 * (2048 * 6144 + 4 * 2048) and dn8 == 6144 * 2048 + 4 * 6144


def test_grouped_expert_bytes_count_one_scale_per_group():
    gu, dn = bench.expert_bytes(synth.FMT_INT4G, 6144, 2048, 128)
    assert gu == 2 * (2048 * 3072 + 4 * 2048 * 48)
    assert dn == 6144 * 1024 + 4 * 6144 * 16


def test_step_and_decode_kernel_bytes():
    cfg = synth.config(2)
    b = bench.step_bytes(cfg, 8)
    router = cfg["E"] * cfg["H"] * 4 + cfg["E"] * 4
    assert b["total"] == b["experts"] + router
    assert b["experts"] == b["gateup"] + b["down"]
    assert bench.decode_kernel_bytes(cfg, 1, 8) == b["total"]       # T <= 8: logits in-kernel
    assert bench.decode_kernel_bytes(cfg, 32, 8) == b["experts"]    # T > 8: a router launch first


def test_group_size_option_converts_int4_experts_only():
    args = argparse.Namespace(workload=3, group_size=64, idot=False)
    cfg = bench.workload_cfg(args)
    assert cfg["routed_fmt"] == synth.FMT_INT4G and cfg["shared_fmt"] == synth.FMT_INT8
    assert cfg["group_size"] == 64
    plain = bench.workload_cfg(argparse.Namespace(workload=3, group_size=0, idot=False))
    assert plain == synth.config(3)


def test_source_hash_ignores_comments_only():
    code = "int f(int a) {\n    return a + 1;  // one more\n}\n/* block\n comment */\n"
    assert bench._code_only(code) == bench._code_only(code.replace("one more", "plus one"))
    assert bench._code_only(code) != bench._code_only(code.replace("a + 1", "a + 2"))


def test_recorded_traffic_only_for_the_captured_plain_kernels():
    src = bench.NCU_TRAFFIC[2]["src"]
    plain = synth.config(2)
    assert bench.recorded_traffic(plain, 2, False, src, 1.0) == bench.NCU_TRAFFIC[2]["bytes"]
    # another kernel source, a variant instance or the general kernels: no recorded traffic
    assert bench.recorded_traffic(plain, 2, False, "0" * 16, 1.0) is None
    assert bench.recorded_traffic(dict(plain, group_size=128, routed_fmt=synth.FMT_INT4G), 2, False, src, 1.0) is None
    assert bench.recorded_traffic(dict(plain, idot=1), 2, False, src, 1.0) is None
    assert bench.recorded_traffic(plain, 2, True, src, 1.0) is None
    # a ratio capture scales with this run's algorithmic bytes
    r3 = bench.NCU_TRAFFIC[3]
    got = bench.recorded_traffic(synth.config(3), 3, False, r3["src"], 2.0e9)
    assert abs(got - r3["ratio"] * 2.0e9) < 1.0 and 1.0 < r3["ratio"] < 1.1
