"""GPU parity with seeded non-unit RMSNorm gains (every attn_norm, ffn_norm
and output_norm drawn N(1, 0.2)), through every decode path: the persistent
step kernel (its own per-layer residuals captured), the separate kernels,
batched steps through the multi-row GEMV and through the small-batch
tensor-core GEMM, prefill, and streamed layers.  With unit gains a kernel
that skipped the gain or read the other norm's gain would still pass; here
it cannot.  (The engine page, section 4.4: fused RMSNorm with its gain.)
Tolerances as everywhere: max|gpu - oracle| <= 2e-3 * max|oracle|.
"""
import dataclasses
import os

import numpy as np
import pytest

import synth
from oracle import OracleModel
from synth.configs import ModelConfig

from parity import assert_close, check_greedy

pytestmark = pytest.mark.gpu

TINY = synth.get_config("tiny")
TINY_Q4 = ModelConfig("tinyq4", 2, 256, 4, 2, 64, 688, 1024, 10000.0, 4, 0.02)
GB = 1 << 30


def _model(cfg, w, env, **kw):
    """A model created with the given DLS_* switches set (they are read at
    creation)."""
    import torch
    from decode_llama_step_gb300 import dls
    old = {k: os.environ.get(k) for k in env}
    os.environ.update(env)
    try:
        stream = torch.cuda.Stream()
        return dls.Model(cfg, w, stream=stream, **kw), stream
    finally:
        for k, v in old.items():
            if v is None:
                del os.environ[k]
            else:
                os.environ[k] = v


def _single_row(cfg, w, orc, env, n_prompt=20, n_decode=6, resident=None):
    """Prefill then batch-1 decode steps, every layer's residual and the
    logits against the oracle."""
    import torch
    m, stream = _model(cfg, w, env, max_seqs=2, max_ctx=n_prompt + n_decode + 8, page_tokens=32)
    try:
        if resident is not None:
            m.set_resident_layers(resident)
        elif env.get("DLS_STEP_KERNEL") == "1":
            used, why = m.step_kernel_in_use()
            assert used, why
        prompt = synth.prompt_tokens(cfg, n_prompt, seed=21)
        seq = m.seq_create()
        lg = torch.empty(cfg.vocab, device="cuda")
        cap = torch.empty(cfg.n_layers, cfg.hidden, device="cuda")
        m.debug_capture(cap)
        m.prefill(seq, prompt, lg)
        stream.synchronize()
        oseq = orc.new_seq(capacity=n_prompt + n_decode)
        ocap = []
        ref = orc.prefill(oseq, prompt, capture=ocap)
        for l in range(cfg.n_layers):
            assert_close(cap[l].cpu().numpy(), ocap[l], f"{env} prefill layer {l}")
        assert_close(lg.cpu().numpy(), ref, f"{env} prefill logits")
        tok = check_greedy(lg.cpu().numpy(), ref, "prefill")
        for i in range(n_decode):
            pos = n_prompt + i
            m.debug_capture(cap)
            m.decode_step(seq, tok, pos, lg)
            stream.synchronize()
            ocap = []
            ref = orc.decode_step(oseq, tok, pos, capture=ocap)
            for l in range(cfg.n_layers):
                assert_close(cap[l].cpu().numpy(), ocap[l], f"{env} step {i} layer {l}")
            got = lg.cpu().numpy()
            assert_close(got, ref, f"{env} step {i} logits")
            # the same step replayed from a graph (no capture) continues the sequence
            tok = check_greedy(got, ref, f"{env} step {i}")
    finally:
        m.close()


def _batched(cfg, w, orc, env, rows, n_prompt=24, n_decode=3):
    """`rows` sequences with their own prompts, decoded together."""
    import torch
    m, stream = _model(cfg, w, env, max_seqs=rows, max_ctx=n_prompt + n_decode + 8, max_batch=rows,
                       page_tokens=32)
    try:
        seqs, oseqs, toks = [], [], []
        for r in range(rows):
            prompt = synth.prompt_tokens(cfg, n_prompt + r, seed=40 + r)
            s = m.seq_create()
            m.prefill(s, prompt)
            seqs.append(s)
            o = orc.new_seq(capacity=n_prompt + rows + n_decode)
            orc.prefill(o, prompt)
            oseqs.append(o)
            toks.append(int(synth.prompt_tokens(cfg, 1, seed=60 + r)[0]))
        out = torch.empty(rows, cfg.vocab, device="cuda")
        for i in range(n_decode):
            pos = [n_prompt + r + i for r in range(rows)]
            m.decode_batch(seqs, toks, pos, out)
            stream.synchronize()
            got = out.cpu().numpy()
            for r in range(rows):
                ref = orc.decode_step(oseqs[r], toks[r], pos[r])
                assert_close(got[r], ref, f"{env} rows={rows} row {r} step {i}")
                toks[r] = check_greedy(got[r], ref, f"{env} row {r} step {i}")
    finally:
        m.close()


@pytest.fixture(scope="module", params=[TINY, TINY_Q4], ids=["q8_0", "q4_0"])
def tiny_gains(request, gpu_lib):
    cfg = request.param
    w = synth.with_random_gains(synth.model_weights(cfg), cfg)
    return cfg, w, OracleModel(cfg, w)


def test_gains_reach_the_oracle(tiny_gains):
    # the drawn gains change the output: the oracle with unit gains differs
    cfg, w, orc = tiny_gains
    unit = OracleModel(cfg, synth.model_weights(cfg))
    a, b = orc.new_seq(), unit.new_seq()
    p = synth.prompt_tokens(cfg, 8, seed=2)
    la, lb = orc.prefill(a, p), unit.prefill(b, p)
    assert np.max(np.abs(la - lb)) > 0.05 * np.max(np.abs(lb))


@pytest.mark.parametrize("env", [{"DLS_STEP_KERNEL": "1"}, {"DLS_STEP_KERNEL": "0"}],
                         ids=["persistent", "separate"])
def test_tiny_gains_single_row(tiny_gains, env):
    cfg, w, orc = tiny_gains
    _single_row(cfg, w, orc, env)


def test_tiny_gains_streamed(tiny_gains):
    cfg, w, orc = tiny_gains
    for n in (0, 1):
        _single_row(cfg, w, orc, {"DLS_STEP_KERNEL": "1"}, resident=n)


@pytest.mark.parametrize("path,rows", [("rg", 2), ("rg", 4), ("tc", 5), ("tc", 8)])
def test_tiny_gains_batched(tiny_gains, path, rows):
    cfg, w, orc = tiny_gains
    _batched(cfg, w, orc, {"DLS_BATCH_GEMM": path}, rows)


@pytest.fixture(scope="module")
def gains_8b_2layers(gpu_lib):
    cfg = dataclasses.replace(synth.get_config("8b"), n_layers=2)
    w = synth.with_random_gains(synth.model_weights(cfg), cfg)
    return cfg, w, OracleModel(cfg, w, cache_bytes=12 * GB)


@pytest.mark.parametrize("env,resident", [({"DLS_STEP_KERNEL": "1"}, None), ({"DLS_STEP_KERNEL": "0"}, None),
                                          ({"DLS_STEP_KERNEL": "1"}, 1)],
                         ids=["persistent", "separate", "streamed"])
def test_8b_two_layers_gains_single_row(gains_8b_2layers, env, resident):
    """Full width and vocabulary (hidden 4096, 32/8 heads, FFN 14336, vocab
    128256), the first two layers of the 8B shape with drawn gains."""
    cfg, w, orc = gains_8b_2layers
    _single_row(cfg, w, orc, env, n_prompt=300, n_decode=3, resident=resident)


@pytest.mark.parametrize("path,rows", [("rg", 3), ("tc", 6)])
def test_8b_two_layers_gains_batched(gains_8b_2layers, path, rows):
    cfg, w, orc = gains_8b_2layers
    _batched(cfg, w, orc, {"DLS_BATCH_GEMM": path}, rows, n_prompt=100, n_decode=2)
