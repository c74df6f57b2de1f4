"""The benchmark's byte and flop accounting (the roofline numerators),
checked against counts written out from the model shapes."""
import os
import sys

import pytest

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_8b_q8_0_decode_bytes_per_token():
    cfg = synth.get_config("8b")
    # Llama-3.1-8B shapes: hidden 4096, 32 query heads and 8 KV heads of 128,
    # FFN 14336, vocab 128256; Q8_0 = 34 bytes per 32 weights
    blk = 34
    qkv = (4096 + 2 * 1024) * (4096 // 32) * blk
    o = 4096 * (4096 // 32) * blk
    gate_up = 2 * 14336 * (4096 // 32) * blk
    down = 4096 * (14336 // 32) * blk
    head = 128256 * (4096 // 32) * blk
    assert qkv + o + gate_up + down == 231_735_296            # one layer's weights
    weights = 32 * (qkv + o + gate_up + down) + head
    assert weights == 7_973_699_584
    ctx = 2048
    kv = 32 * 2 * ctx * 1024 * 2                              # K and V of every layer, fp16
    # each GEMV reads its fp32 input vector and writes its fp32 output vector
    act = 32 * 4 * ((4096 + 6144) + (4096 + 4096) + (4096 + 28672) + (14336 + 4096)) + 4 * (4096 + 128256)
    assert bench.step_bytes(cfg, ctx) == weights + kv + act == 8_251_577_344


def test_q4_0_bytes_and_kind_split():
    cfg = synth.get_config("fork8b")
    assert cfg.wtype == 4
    # Q4_0 = 18 bytes per 32 weights
    assert bench.gemv_bytes(14336 * 2, 4096, 4) == 28672 * 128 * 18 + 4 * (4096 + 28672)
    # the per-kind bytes of a step add up to the step (attention counts q and o besides K/V)
    ctx = 4096
    kinds = sum(bench.kind_bytes(cfg, k, ctx) for k in (2, 4, 5, 6)) * cfg.n_layers + bench.kind_bytes(cfg, 7, ctx)
    kv = cfg.n_layers * 2 * ctx * cfg.kv_dim * 2
    assert kinds + kv == pytest.approx(bench.step_bytes(cfg, ctx), rel=2e-3)


def test_prefill_flops_closed_form():
    cfg = synth.get_config("8b")
    T = 2048
    layer_params = (4096 + 2048) * 4096 + 4096 * 4096 + 3 * 14336 * 4096
    pairs = T * (T + 1) // 2                                   # causal (query, key) pairs
    att = 2 * 2 * 32 * 128 * pairs                             # QK^T and PV, 2 flops per multiply-add
    want = 32 * (2 * layer_params * T + att) + 2 * 128256 * 4096
    assert bench.prefill_flops(cfg, T) == want


def test_reference_arm_prints_one_contract_line():
    # the reference arm (the oracle on the host cores) on the tiny shape: one
    # JSON line with the keys the driver reads, the steps and warmup it ran
    import json
    import subprocess
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
                          "--steps", "3", "--warmup", "1", "--ctx", "64"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "impl"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 3 and d["warmup"] == 1
    assert d["value"] > 0 and d["unit"] == "tok/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert abs(d["ms_per_step"] - 1000.0 / d["value"]) <= 0.01 * d["ms_per_step"]


def test_reference_arm_runs_on_rank_0_only():
    import subprocess
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
                          "--steps", "2", "--warmup", "0", "--ctx", "64", "--gpus", "2"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert out.returncode == 0, out.stderr[-2000:]
    assert not [l for l in out.stdout.splitlines() if l.startswith("{")]
