"""Prefill on the tensor cores, through the C ABI, against the oracle:
the GEMM on every matrix (one to three 128-token tiles, ragged tails), the
per-layer residual of the last prompt token, the fp16 K/V it writes, the
logits, a prefill that continues a sequence, and chunk-size independence.

The GEMM feeds each dequantised weight d*q and each activation to the
tensor cores as two fp16 planes (hi = fp16(v), lo = fp16(v - hi)) and sums
w_hi x_hi + w_hi x_lo + w_lo x_hi in fp32, so it must track the exact fp64
product to about 1e-5; the layers must meet the layer tolerance (2e-3 of
L-inf).
"""
import os

import numpy as np
import pytest

import synth
from oracle import OracleModel, quant
from synth.configs import ModelConfig

from parity import assert_close, check_greedy, rel_err

pytestmark = pytest.mark.gpu

TINY = synth.get_config("tiny")
# hidden 224 and ffn 720 end in half a 64-column K tile; ffn, vocab and q
# rows end in partial 128-row tiles; hidden != n_heads * head_dim
RAGGED = ModelConfig("ragged", 2, 224, 4, 2, 64, 720, 1000, 10000.0, 8, 0.02)
# Q4_0, head_dim 32 (CUDA-core prefill attention), 4 query heads per KV head
RAGGED_Q4 = ModelConfig("raggedq4", 2, 224, 8, 2, 32, 720, 1000, 10000.0, 4, 0.02)
# head_dim 128 with 4 query heads per KV head (the 8B attention shape), 256-token pages
WIDE = ModelConfig("wide", 2, 256, 8, 2, 128, 512, 512, 500000.0, 8, 0.02)
CFGS = [(TINY, 32), (RAGGED, 32), (RAGGED_Q4, 32), (WIDE, 256)]


def _torch():
    import torch
    return torch


def _make(cfg, w, chunk=None, page_tokens=32, **kw):
    from decode_llama_step_gb300 import dls
    torch = _torch()
    old = os.environ.get("DLS_PREFILL_CHUNK")
    if chunk is not None:
        os.environ["DLS_PREFILL_CHUNK"] = str(chunk)
    try:
        stream = torch.cuda.Stream()
        m = dls.Model(cfg, w, max_seqs=4, max_ctx=kw.get("max_ctx", 200), max_batch=1, page_tokens=page_tokens,
                      stream=stream)
    finally:
        if old is None:
            os.environ.pop("DLS_PREFILL_CHUNK", None)
        else:
            os.environ["DLS_PREFILL_CHUNK"] = old
    return m, stream


@pytest.fixture(scope="module", params=CFGS, ids=[f"{c.name}-pt{pt}" for c, pt in CFGS])
def setup(request, gpu_lib):
    cfg, pt = request.param
    w = synth.model_weights(cfg)
    m, stream = _make(cfg, w, chunk=48, page_tokens=pt)   # several chunks per prompt below
    orc = OracleModel(cfg, w)
    yield cfg, w, m, orc, stream
    m.close()


def _f16(a):
    return np.asarray(a, dtype=np.float32).astype(np.float16).astype(np.float64)


@pytest.mark.parametrize("T", [1, 8, 16, 17, 300])
def test_gemm_every_matrix(setup, T):
    torch = _torch()
    cfg, w, m, orc, stream = setup
    shapes = synth.matrix_shapes(cfg)
    shapes["output"] = (cfg.vocab, cfg.hidden)
    shapes["tok_embd"] = (cfg.vocab, cfg.hidden)
    for name, (rows, cols) in shapes.items():
        x = synth.normal(synth.stream_key("gemm-x", name, T), T * cols, 1.0).astype(np.float32).reshape(T, cols)
        y = torch.empty(T, rows, device="cuda")
        m.debug_gemm(1, name, torch.from_numpy(x).cuda(), y)
        got = y.cpu().numpy()
        if name in ("output", "tok_embd"):
            W = quant.matrix(w[name], cfg.vocab, cfg.hidden, cfg.wtype)
        else:
            W = quant.matrix(w["layers"][1][name], rows, cols, cfg.wtype)
        # activations and dequantised weights enter the tensor cores as
        # hi + lo fp16 planes (about 22 bits each): the result tracks the
        # exact product, far inside what single fp16 operands give (~3e-4)
        exact = x.astype(np.float64) @ W.T
        e = rel_err(got, exact)
        assert e <= 1e-5, f"{name} T={T}: vs the exact product {e:.3e}"
        assert rel_err(_f16(x) @ _f16(W).T, exact) > 10 * e or e < 1e-6


@pytest.mark.parametrize("T", [256, 300, 520])
def test_gemm_256_token_tiles(gpu_lib, T, monkeypatch):
    """Prompt chunks on 256-token tiles (DLS_PREFILL_BN=256; large matrices
    choose them by themselves): every matrix of the ragged shapes, token
    counts on and off a tile boundary, against the exact product."""
    torch = _torch()
    monkeypatch.setenv("DLS_PREFILL_BN", "256")
    for cfg in (RAGGED, RAGGED_Q4):
        w = synth.model_weights(cfg)
        m, stream = _make(cfg, w, max_ctx=600)
        try:
            shapes = synth.matrix_shapes(cfg)
            for name, (rows, cols) in shapes.items():
                x = synth.normal(synth.stream_key("gemm256-x", name, T), T * cols, 1.0).astype(np.float32)
                x = x.reshape(T, cols)
                y = torch.empty(T, rows, device="cuda")
                m.debug_gemm(1, name, torch.from_numpy(x).cuda(), y)
                W = quant.matrix(w["layers"][1][name], rows, cols, cfg.wtype)
                e = rel_err(y.cpu().numpy(), x.astype(np.float64) @ W.T)
                assert e <= 1e-5, f"{cfg.name} {name} T={T}: vs the exact product {e:.3e}"
        finally:
            m.close()


def _read_kv(m, cfg, seq, n, layer):
    torch = _torch()
    kvd = cfg.n_kv_heads * cfg.head_dim
    k = torch.empty(n, kvd, dtype=torch.float16, device="cuda")
    v = torch.empty_like(k)
    m.debug_read_kv(seq, layer, k, v)
    return k, v


def test_prefill_layers_kv_logits(setup):
    """A 100-token prompt (three 48-token chunks), then 41 more tokens
    continuing the same sequence: per-layer residual of the last token, all
    K/V, logits and greedy token against the oracle after each call."""
    torch = _torch()
    cfg, w, m, orc, stream = setup
    seq = m.seq_create()
    oseq = orc.new_seq()
    try:
        n0 = 0
        for n, seed in ((100, 3), (41, 4)):
            prompt = synth.prompt_tokens(cfg, n, seed=seed)
            cap = torch.empty(cfg.n_layers, cfg.hidden, device="cuda")
            logits = torch.empty(cfg.vocab, device="cuda")
            m.debug_capture(cap)
            m.prefill(seq, prompt, logits)
            ocap = []
            ref = orc.prefill(oseq, prompt, capture=ocap)
            n0 += n
            assert m.seq_length(seq) == n0
            got_cap = cap.cpu().numpy()
            for l in range(cfg.n_layers):
                assert_close(got_cap[l], ocap[l], f"n={n} layer {l} residual")
                k, v = _read_kv(m, cfg, seq, n0, l)
                shape = (n0, cfg.n_kv_heads, cfg.head_dim)
                assert_close(k.cpu().numpy().astype(np.float64).reshape(shape), oseq.keys(l), f"layer {l} K")
                assert_close(v.cpu().numpy().astype(np.float64).reshape(shape), oseq.values(l), f"layer {l} V")
            assert_close(logits.cpu().numpy(), ref, f"n={n} logits")
            check_greedy(logits.cpu().numpy(), ref, f"n={n}")
    finally:
        m.seq_free(seq)


def test_prefill_then_decode(setup):
    """Decode steps attend over the K/V the prefill wrote."""
    torch = _torch()
    cfg, w, m, orc, stream = setup
    prompt = synth.prompt_tokens(cfg, 77, seed=6)
    seq = m.seq_create()
    oseq = orc.new_seq()
    try:
        logits = torch.empty(cfg.vocab, device="cuda")
        m.prefill(seq, prompt, logits)
        ref = orc.prefill(oseq, prompt)
        tok = check_greedy(logits.cpu().numpy(), ref, "prefill")
        for i in range(6):
            m.decode_step(seq, tok, 77 + i, logits)
            ref = orc.decode_step(oseq, tok, 77 + i)
            assert_close(logits.cpu().numpy(), ref, f"step {i} logits")
            tok = check_greedy(logits.cpu().numpy(), ref, f"step {i}")
    finally:
        m.seq_free(seq)


def test_chunk_size_does_not_change_results(gpu_lib):
    """A token's arithmetic does not depend on which chunk carries it as long
    as the chunks run the same GEMM tiling: one chunk of 150 and three chunks
    of 50 (128-token tiles) give bit-identical K/V and logits.  Chunks of 7 run the
    16-token tiles with K split across CTAs: the fp32 summation order
    changes, and where that moves an activation or a K/V entry across an
    fp16 rounding boundary the difference is one fp16 step there."""
    torch = _torch()
    cfg = TINY
    w = synth.model_weights(cfg)
    prompt = synth.prompt_tokens(cfg, 150, seed=12)
    outs = []
    for chunk in (None, 50, 7):
        m, stream = _make(cfg, w, chunk=chunk)
        try:
            s = m.seq_create()
            lg = torch.empty(cfg.vocab, device="cuda")
            m.prefill(s, prompt, lg)
            kv = [_read_kv(m, cfg, s, 150, l) for l in range(cfg.n_layers)]
            stream.synchronize()
            outs.append((lg.clone(), [(k.clone(), v.clone()) for k, v in kv]))
        finally:
            m.close()
    lg, kv = outs[1]
    assert torch.equal(lg, outs[0][0])
    for (k, v), (k0, v0) in zip(kv, outs[0][1]):
        assert torch.equal(k.view(torch.int16), k0.view(torch.int16))
        assert torch.equal(v.view(torch.int16), v0.view(torch.int16))
    lg, kv = outs[2]
    assert_close(lg.cpu().numpy(), outs[0][0].cpu().numpy(), "chunks of 7 vs one chunk", tol=1e-3)
    for (k, v), (k0, v0) in zip(kv, outs[0][1]):
        assert_close(k.float().cpu().numpy(), k0.float().cpu().numpy(), "K, chunks of 7", tol=1e-3)
        assert_close(v.float().cpu().numpy(), v0.float().cpu().numpy(), "V, chunks of 7", tol=1e-3)


@pytest.mark.parametrize("cfg,pt", [(TINY, 32), (RAGGED, 32), (RAGGED_Q4, 32)], ids=["tiny", "ragged", "raggedq4"])
def test_exact_code_gemm_prefill(gpu_lib, cfg, pt, monkeypatch):
    """The prompt-chunk GEMM with the codes as exact MMA operands and the
    block scales applied per 32 columns after the MMA (DLS_PREFILL_GEMM=codes,
    read at model creation): every projection of a 300-token chunk against
    the exact product, then a prefill's residuals and logits against the
    oracle."""
    torch = _torch()
    monkeypatch.setenv("DLS_PREFILL_GEMM", "codes")
    w = synth.model_weights(cfg)
    m, stream = _make(cfg, w, chunk=120, page_tokens=pt, max_ctx=320)
    monkeypatch.delenv("DLS_PREFILL_GEMM")
    orc = OracleModel(cfg, w)
    try:
        shapes = synth.matrix_shapes(cfg)
        shapes["output"] = (cfg.vocab, cfg.hidden)
        T = 300
        for name, (rows, cols) in shapes.items():
            x = synth.normal(synth.stream_key("gemm-x", name, T), T * cols, 1.0).astype(np.float32).reshape(T, cols)
            y = torch.empty(T, rows, device="cuda")
            m.debug_gemm(1, name, torch.from_numpy(x).cuda(), y)
            W = quant.matrix(w[name] if name == "output" else w["layers"][1][name], rows, cols, cfg.wtype)
            assert rel_err(y.cpu().numpy(), x.astype(np.float64) @ W.T) <= 1e-5, name
        prompt = synth.prompt_tokens(cfg, 250, seed=6)
        seq = m.seq_create()
        lg = torch.empty(cfg.vocab, device="cuda")
        cap = torch.empty(cfg.n_layers, cfg.hidden, device="cuda")
        m.debug_capture(cap)
        m.prefill(seq, prompt, lg)
        stream.synchronize()
        oseq = orc.new_seq(capacity=260)
        ocap = []
        ref = orc.prefill(oseq, prompt, capture=ocap)
        for l in range(cfg.n_layers):
            assert_close(cap[l].cpu().numpy(), ocap[l], f"codes GEMM prefill layer {l}")
        assert_close(lg.cpu().numpy(), ref, "codes GEMM prefill logits")
    finally:
        m.close()
