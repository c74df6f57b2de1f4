"""K-quant weights inside the model (the engine page, section 1: the 70B
runs quoted on Q4_K_M and Q6_K files): per-matrix weight types through the
C ABI, the mixed-format decode path (per-matrix dequant-GEMVs), prefill,
batched steps and streamed layers, against the fp64 oracle reading the same
super-blocks.  Tolerances as everywhere: max|gpu - oracle| <= 2e-3 *
max|oracle|; dequantised weights are the fp32 rounding of the exact value.
"""
import dataclasses

import numpy as np
import pytest

import synth
from oracle import OracleModel, ops
from synth.configs import ModelConfig

from parity import assert_close, check_greedy

pytestmark = pytest.mark.gpu

# the tiny shape with FFN 768 (a K-quant matrix's input width is a multiple of 256)
TINYK = ModelConfig("tinyk", 2, 256, 4, 2, 64, 768, 1024, 10000.0, 8, 0.02)
PARTIAL = {"wv": "q6_k", "w_down": "q6_k", "w_up": "q5_k"}   # the rest stay Q8_0
GB = 1 << 30


def _torch():
    import torch
    return torch


@pytest.fixture(scope="module", params=["q4_k_m", "partial"])
def tiny(request, gpu_lib):
    fm = synth.Q4_K_M if request.param == "q4_k_m" else PARTIAL
    w = synth.model_weights_k(TINYK, fm)
    return request.param, w, OracleModel(TINYK, w)


def _model(w, **kw):
    torch = _torch()
    from decode_llama_step_gb300 import dls
    stream = torch.cuda.Stream()
    return dls.Model(TINYK, w, stream=stream, page_tokens=32, **kw), stream


def test_dequant_matches_the_oracle(tiny):
    torch = _torch()
    name, w, orc = tiny
    m, stream = _model(w, max_seqs=1, max_ctx=64)
    try:
        shapes = synth.matrix_shapes(TINYK)
        for l in range(TINYK.n_layers):
            for t in synth.LAYER_MATRICES:
                rows, cols = shapes[t]
                out = torch.empty(rows, cols, device="cuda")
                m.debug_dequant(l, t, out)
                stream.synchronize()
                ref = orc.matrix(l, t).astype(np.float32)
                assert np.array_equal(out.cpu().numpy(), ref), f"{name} layer {l} {t}"
        for t in ("tok_embd", "output"):
            out = torch.empty(TINYK.vocab, TINYK.hidden, device="cuda")
            m.debug_dequant(0, t, out)
            stream.synchronize()
            assert np.array_equal(out.cpu().numpy(), orc.matrix(None, t).astype(np.float32)), f"{name} {t}"
    finally:
        m.close()


@pytest.mark.parametrize("resident", [2, 1, 0])
def test_prefill_and_decode_against_the_oracle(tiny, resident):
    """Prefill of 19 tokens (three passes of up to 8), then 6 greedy decode
    steps, every layer's residual and the logits; resident, one layer and no
    layer resident (streamed through the staging buffers)."""
    torch = _torch()
    name, w, orc = tiny
    m, stream = _model(w, max_seqs=1, max_ctx=64)
    try:
        m.set_resident_layers(resident)
        prompt = synth.prompt_tokens(TINYK, 19, seed=4)
        seq = m.seq_create()
        lg = torch.empty(TINYK.vocab, device="cuda")
        cap = torch.empty(TINYK.n_layers, TINYK.hidden, device="cuda")
        m.debug_capture(cap)
        m.prefill(seq, prompt, lg)
        stream.synchronize()
        oseq = orc.new_seq()
        ocap = []
        ref = orc.prefill(oseq, prompt, capture=ocap)
        for l in range(TINYK.n_layers):
            assert_close(cap[l].cpu().numpy(), ocap[l], f"{name} prefill layer {l}")
        assert_close(lg.cpu().numpy(), ref, f"{name} prefill logits")
        tok = check_greedy(lg.cpu().numpy(), ref, "prefill")
        for i in range(6):
            pos = 19 + i
            m.debug_capture(cap)
            m.decode_step(seq, tok, pos, lg)
            stream.synchronize()
            ocap = []
            ref = orc.decode_step(oseq, tok, pos, capture=ocap)
            for l in range(TINYK.n_layers):
                assert_close(cap[l].cpu().numpy(), ocap[l], f"{name} step {i} layer {l}")
            assert_close(lg.cpu().numpy(), ref, f"{name} step {i} logits")
            tok = check_greedy(lg.cpu().numpy(), ref, f"{name} step {i}")
    finally:
        m.close()


def test_batched_steps_and_generation(tiny):
    """Three sequences decoded together (each row through the per-matrix
    GEMVs), then greedy generation on the device (graph replay), against the
    oracle's own greedy run."""
    torch = _torch()
    name, w, orc = tiny
    m, stream = _model(w, max_seqs=3, max_ctx=96, max_batch=3)
    try:
        seqs, oseqs, toks = [], [], []
        for r in range(3):
            p = synth.prompt_tokens(TINYK, 10 + r, seed=20 + r)
            s = m.seq_create()
            m.prefill(s, p)
            o = orc.new_seq()
            orc.prefill(o, p)
            seqs.append(s)
            oseqs.append(o)
            toks.append(7 + r)
        out = torch.empty(3, TINYK.vocab, device="cuda")
        for i in range(3):
            pos = [10 + r + i for r in range(3)]
            m.decode_batch(seqs, toks, pos, out)
            stream.synchronize()
            for r in range(3):
                ref = orc.decode_step(oseqs[r], toks[r], pos[r])
                assert_close(out[r].cpu().numpy(), ref, f"{name} batch row {r} step {i}")
                toks[r] = check_greedy(out[r].cpu().numpy(), ref, f"{name} batch row {r} step {i}")
        gen = m.generate([seqs[0]], [toks[0]], 5)
        ref_toks, _ = orc.greedy_decode(oseqs[0], toks[0], 5)
        assert list(gen[:, 0]) == ref_toks
    finally:
        m.close()


def test_types_are_checked_before_anything_is_allocated(gpu_lib):
    from decode_llama_step_gb300 import dls
    w = synth.model_weights_k(TINYK, {"wq": "q4_k"})
    w["formats"][(1, "wq")] = "q6_k"          # layer 1 differs from layer 0
    with pytest.raises(dls.DlsError) as e:
        _model(w, max_seqs=1, max_ctx=32)
    assert e.value.code == dls.DLS_ERR_ARG and "differs from layer 0" in str(e.value)
    cfg = TINYK
    bad = dataclasses.replace(cfg, ffn=688)   # down projection input 688: not a multiple of 256
    wb = synth.model_weights(bad)
    wb["formats"] = {(l, "w_down"): "q6_k" for l in range(bad.n_layers)}
    from decode_llama_step_gb300 import dls as d2
    torch = _torch()
    with pytest.raises(d2.DlsError) as e:
        d2.Model(bad, wb, max_seqs=1, max_ctx=32, stream=torch.cuda.Stream())
    assert e.value.code == d2.DLS_ERR_ARG and "multiple of 256" in str(e.value)


@pytest.mark.slow
def test_70b_q4_k_m_first_layer_resident_and_streamed(gpu_lib):
    """The 70B shape as a Q4_K_M-style file (value and down projections and
    the LM head Q6_K, the rest Q4_K), cut to its first layer at full width
    (hidden 8192, 64/8 heads, FFN 28672, vocab 128256): a 40-token prefill
    and three decode steps, resident and streamed, against the oracle (the
    layer's residual in full, the logits on sampled rows plus the GPU's
    argmax)."""
    torch = _torch()
    from decode_llama_step_gb300 import dls
    cfg = dataclasses.replace(synth.get_config("70b"), n_layers=1)
    w = synth.model_weights_k(cfg, synth.Q4_K_M)
    orc = OracleModel(cfg, w, cache_bytes=24 * GB)
    P, D = 40, 3
    prompt = synth.prompt_tokens(cfg, P, seed=1)
    rng = np.random.default_rng(5)
    sample = np.unique(rng.integers(0, cfg.vocab, 48))
    # oracle: prefill, then decode with its own greedy picks over the sample
    oseq = orc.new_seq(capacity=P + D)
    X = orc.embed(prompt)
    X = orc.layer_forward(0, X, 0, oseq)
    oseq.n = P
    steps = [(None, X[-1])]
    toks = [int(synth.prompt_tokens(cfg, 1, seed=9)[0]) + i for i in range(D)]
    for i in range(D):
        x = orc.layer_forward(0, orc.embed(toks[i]), P + i, oseq)
        oseq.n = P + i + 1
        steps.append((toks[i], x))
    stream = torch.cuda.Stream()
    m = dls.Model(cfg, w, max_seqs=1, max_ctx=P + D + 8, stream=stream)
    try:
        for n_res in (1, 0):
            m.set_resident_layers(n_res)
            seq = m.seq_create()
            lg = torch.empty(cfg.vocab, device="cuda")
            cap = torch.empty(1, cfg.hidden, device="cuda")
            for i, (tok, ref_x) in enumerate(steps):
                m.debug_capture(cap)
                if tok is None:
                    m.prefill(seq, prompt, lg)
                else:
                    m.decode_step(seq, tok, P + i - 1, lg)
                stream.synchronize()
                got_x = cap[0].cpu().numpy()
                assert_close(got_x, ref_x, f"resident={n_res} step {i} residual")
                got = lg.cpu().numpy()
                rows = np.unique(np.concatenate([sample, [int(np.argmax(got))]]))
                ref = orc.final_logits(ref_x, rows=rows)
                assert_close(got[rows], ref, f"resident={n_res} step {i} sampled logits")
            m.seq_free(seq)
    finally:
        m.close()
