"""Generator determinism / recipe checks and the byte/FLOP accounting pinned to
the figures printed on the source pages (tests/golden/page_figures.json)."""
import json
import os

import numpy as np
import pytest

import oracle
import synth
from moe_expert_ffn_02_gb300 import roofline

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_figures.json")


def test_generator_is_counter_based_and_deterministic():
    a = synth.bf16_normal(0, synth.STREAM_X, (4, 1024))
    b = synth.bf16_normal(0, synth.STREAM_X, (4, 1024))
    assert np.array_equal(a, b)
    c = synth.bf16_normal(0, synth.STREAM_X, (8, 1024))
    assert np.array_equal(c[:4], a)                           # prefix-stable
    assert not np.array_equal(synth.bf16_normal(1, synth.STREAM_X, (4, 1024)), a)
    assert not np.array_equal(synth.bf16_normal(0, synth.STREAM_ROUTER_W, (4, 1024)), a)
    q1, s1 = synth.fp8_blocks(0, synth.STREAM_GATE, 3, 256, 384)
    q2, s2 = synth.fp8_blocks(0, synth.STREAM_GATE, 2, 256, 384)
    assert np.array_equal(q1[:2], q2) and np.array_equal(s1[:2], s2)


def test_generator_distributions():
    x = synth.bf16_to_f32(synth.bf16_normal(0, synth.STREAM_X, (256, 1024))).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01 and np.abs(x).max() <= 6.0
    q, s = synth.fp8_blocks(0, synth.STREAM_GATE, 2, 256, 512, std=0.02)
    w = oracle.e4m3_decode(q) * np.repeat(np.repeat(s.astype(np.float64), 128, 1), 128, 2)
    assert abs(w.std() - 0.02) < 0.001
    # every block's multiplier is its amax / 448, so its largest code is +-448
    blk = q.reshape(2, 2, 128, 4, 128).transpose(0, 1, 3, 2, 4).reshape(2, 2, 4, -1)
    assert np.all((blk & 0x7F).max(-1) == 0x7E)


def test_zipf_bias_recipe_gives_skewed_load():
    """Skewed 32K prefill workload: popularity must put hot experts above
    10x the mean row count and leave some experts with no rows."""
    wl = synth.WORKLOADS["skew_32k"]
    b = synth.router_bias(wl, seed=0)
    assert b.shape == (wl.n_experts,) and np.isclose(b.max(), 0.0)
    # logits ~ N(0,1) (router std 1/sqrt(H) on N(0,1) activations) plus the bias
    L = (np.random.default_rng(0).normal(0, 1, (wl.T, wl.n_experts)) + b).astype(np.float32)
    r = oracle.route_from_logits(L, wl.top_k)
    counts = np.diff(r["offsets"])
    mean = wl.T * wl.top_k / wl.n_experts
    assert counts.max() > 10 * mean
    assert np.count_nonzero(counts == 0) > 0


def test_page_figures_pin_accounting():
    fig = {e["name"]: e for e in json.load(open(GOLDEN))["entries"]}

    def close(name, got):
        e = fig[name]
        assert abs(got - e["value"]) <= e["rel_tol"] * e["value"] + 1e-9, (name, got, e["value"])

    close("params_per_expert", roofline.expert_params(7168, 2048))
    close("active_routed_params_per_token", 58 * 8 * roofline.expert_params(7168, 2048))
    close("routed_params_model", 58 * 256 * roofline.expert_params(7168, 2048))
    close("layer_expert_bytes_deepseek_v3", roofline.layer_expert_bytes(7168, 2048, 256))
    close("layer_expert_bytes_kimi_k2", roofline.layer_expert_bytes(7168, 2048, 384))
    close("weight_tensor_count_deepseek_v3", 58 * 256 * 3)
    close("tokens_per_routed_expert_b64", roofline.tokens_per_routed_expert(64, 8, 256))
    close("active_routed_bytes_per_token_4p5bit", 58 * 8 * roofline.expert_params(7168, 2048) * 4.5 / 8)


def test_flop_and_touched_byte_accounting():
    # 2 * 3 * H * I per (token, expert) pair, k routed + 1 shared per token
    assert roofline.layer_flops(8192, 7168, 2048, 8, 1) == 88_080_384 * 8192 * 9
    assert abs(roofline.expected_distinct_experts(16, 8, 256) - 256 * (1 - (31 / 32) ** 16)) < 1e-9
    ids = np.array([[0, 3], [3, 5]])
    assert roofline.touched_experts(ids, 8) == 3
    eb = roofline.expert_bytes(7168, 2048)
    assert eb == 44_040_192 + 3 * 56 * 16 * 4
    assert roofline.decode_weight_bytes(ids, 7168, 2048, 8, 1) == 4 * eb


def test_bench_reference_arm_prints_the_contract_line():
    """bench.py --impl reference times the CPU oracle (no GPU needed) and prints
    one JSON line with the contract's keys; a non-zero rank prints nothing."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--workload", "tiny",
           "--steps", "1", "--warmup", "3"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=root)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 1 and d["warmup"] == 3 and d["value"] > 0
    assert d["config"]["workload"] == "tiny"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=root, env=env)
    assert out.returncode == 0 and not [l for l in out.stdout.splitlines() if l.startswith("{")]


def test_bench_metric_helpers():
    """The bench line's value and CPU-baseline arithmetic, and the rule that
    the roofline's traffic figure is used only for the sources it was taken on."""
    import json
    import os
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    dec, pre = synth.WORKLOADS["ds_decode_t16"], synth.WORKLOADS["ds_prefill_8k"]
    assert bench.metric_of(dec) == ("moe_layer_decode_us_per_layer", "us/layer", False)
    assert bench.metric_of(pre) == ("moe_layer_prefill_tokens_per_s", "tokens/s", True)
    # one replica: the step time itself / T tokens per step time; N replicas: the whole job
    assert bench.value_of(dec, 764e-6) == 764e-6 * 1e6
    assert abs(bench.value_of(dec, 800e-6, 4) - 200.0) < 1e-9
    assert abs(bench.value_of(pre, 4e-3) - 8192 / 4e-3) < 1e-6
    assert abs(bench.value_of(pre, 4e-3, 2) - 2 * 8192 / 4e-3) < 1e-6
    # oracle sample scaled to the workload's unit
    assert abs(bench.cpu_value(dec, 2.0, 4) - 2.0 / 4 * 16 * 1e6) < 1e-3
    assert abs(bench.cpu_value(pre, 2.0, 100) - 50.0) < 1e-12
    # traffic: only when the committed capture was taken on the current sources of that kernel
    hd, hp = bench.kernel_source_hash("decode"), bench.kernel_source_hash("prefill")
    assert hd == bench.kernel_source_hash("decode") and len(hd) == 16 and hd != hp
    d = json.load(open(bench.TRAFFIC_FILE))
    for wl_name, per in d.items():
        kind = "decode" if "decode" in wl_name else "prefill"
        h = hd if kind == "decode" else hp
        for kernel, e in per.items():
            got = bench.traffic_for(kernel, wl_name, kind)
            assert got == (e["dram_bytes_per_launch"] if e["source_hash"] == h else None)
            # a record never applies to the other path's kernel
            if e["source_hash"] == h:
                assert bench.traffic_for(kernel, wl_name, "prefill" if kind == "decode" else "decode") is None
    assert bench.traffic_for("gate_up", "no_such_workload", "decode") is None
