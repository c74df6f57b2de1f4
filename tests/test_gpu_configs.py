"""GPU parity at the workloads' full sizes, through the C ABI.

The five model shapes and their workloads (the 1B, 8B, fork and 70B shapes;
the tiny one is covered in test_gpu_tiny.py) run here in the launch
configuration the benchmark times.  Where the fp64 oracle cannot follow the
whole model in seconds, it checks a sample it can compute on its own from the
same seeded inputs: the first layers of the model at full width and full
context.  Weights are drawn per (shape, layer, tensor), so a model cut to its
first n layers holds exactly the first n layers of the full model, and the
GPU's residual stream after those layers in the full model must match the
oracle's.  Properties that hold at any size cover the rest: the KV fork
copies bytes exactly, a forked branch decodes exactly like an independent
prefill, and streamed layers compute what resident layers compute.

Decode inputs come from the oracle: either seeded token ids, or the oracle's
own greedy token at every step (teacher forcing), so that no input of the
oracle ever comes from the GPU.  Tolerances: max|gpu - oracle| <= 2e-3 *
max|oracle| for residuals and logits, identical greedy tokens wherever the
oracle's top-2 gap exceeds 1e-2, bit-exact fork copies.
"""
import dataclasses

import numpy as np
import pytest

import synth
from oracle import OracleModel, ops

from parity import assert_close, check_greedy

pytestmark = pytest.mark.gpu

GB = 1 << 30


def _torch():
    import torch
    return torch


def cut(cfg, n_layers):
    """The first n_layers of a shape (same weights for those layers)."""
    return dataclasses.replace(cfg, n_layers=n_layers)


def gpu_model(cfg, w, **kw):
    from decode_llama_step_gb300 import dls
    torch = _torch()
    stream = torch.cuda.Stream()
    return dls.Model(cfg, w, stream=stream, **kw), stream


def captured(m, stream, cfg, fn):
    """Run fn() with the per-layer capture armed; residuals [n_layers, hidden]."""
    torch = _torch()
    cap = torch.empty(cfg.n_layers, cfg.hidden, device="cuda")
    m.debug_capture(cap)
    fn()
    stream.synchronize()
    return cap.cpu().numpy().astype(np.float64)


def host(t, stream):
    """A device tensor as fp64 numpy, after the model's stream has finished."""
    stream.synchronize()
    return t.cpu().numpy().astype(np.float64)


def release(*models):
    torch = _torch()
    for m in models:
        if m is not None:
            m.close()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def test_1b_prefill_512_then_128_greedy_steps(gpu_lib):
    """Llama-3.2-1B shape (16 layers, tied embeddings, Q8_0): prefill of 512
    seeded tokens, then 128 greedy decode steps, every layer and every
    step's logits against the full fp64 oracle."""
    torch = _torch()
    cfg = synth.get_config("1b")
    P, D = cfg.workload["prompt"], cfg.workload["decode"]
    w = synth.model_weights(cfg)
    m, stream = gpu_model(cfg, w, max_seqs=1, max_ctx=P + D + 8)
    orc = OracleModel(cfg, w, cache_bytes=16 * GB)
    try:
        prompt = synth.prompt_tokens(cfg, P, seed=1)
        seq = m.seq_create()
        logits = torch.empty(cfg.vocab, device="cuda")
        got_layers = captured(m, stream, cfg, lambda: m.prefill(seq, prompt, logits))
        oseq = orc.new_seq(capacity=P + D)
        ref_layers = []
        ref = orc.prefill(oseq, prompt, capture=ref_layers)
        for l in range(cfg.n_layers):
            assert_close(got_layers[l], ref_layers[l], f"prefill layer {l}")
        got = host(logits, stream)
        assert_close(got, ref, "prefill logits")
        tok = check_greedy(got, ref, "prefill")
        worst = 0.0
        for i in range(D):
            pos = P + i
            m.decode_step(seq, tok, pos, logits)
            ref = orc.decode_step(oseq, tok, pos)
            got = host(logits, stream)
            worst = max(worst, assert_close(got, ref, f"decode step {i}"))
            tok = check_greedy(got, ref, f"decode step {i}")  # the oracle's token feeds both sides
        assert m.seq_length(seq) == P + D
    finally:
        release(m)


@pytest.fixture(scope="module")
def w8b():
    cfg = synth.get_config("8b")
    return cfg, synth.model_weights(cfg)


@pytest.mark.parametrize("ctx", [2048, 8192])
def test_8b_decode_at_context(gpu_lib, w8b, ctx):
    """Llama-3.1-8B shape, Q8_0, batch-1 decode at KV context 2048 and 8192
    (the KV filled by prefill of seeded tokens).  The full 32-layer model's
    residual stream after layers 0 and 1 is checked against the oracle for
    the last prompt token and each decode step; the model cut to 2 layers
    (same kernels and launch shapes, full width and vocabulary) is checked
    end to end, logits included."""
    torch = _torch()
    cfg, w = w8b
    D = 4
    prompt = synth.prompt_tokens(cfg, ctx, seed=1)
    toks = synth.prompt_tokens(cfg, D, seed=5)          # seeded decode inputs
    c2 = cut(cfg, 2)
    w2 = dict(w, layers=w["layers"][:2])
    orc = OracleModel(c2, w2, cache_bytes=12 * GB)
    oseq = orc.new_seq(capacity=ctx + D)
    ref_pre_layers = []
    ref_pre = orc.prefill(oseq, prompt, capture=ref_pre_layers)
    ref_layers, ref_logits = [], []
    for i in range(D):
        cap = []
        ref_logits.append(orc.decode_step(oseq, int(toks[i]), ctx + i, capture=cap))
        ref_layers.append(cap)

    # the full model: layers 0 and 1 of its residual stream
    m, stream = gpu_model(cfg, w, max_seqs=1, max_ctx=ctx + D + 8)
    try:
        seq = m.seq_create()
        got = captured(m, stream, cfg, lambda: m.prefill(seq, prompt))
        for l in range(2):
            assert_close(got[l], ref_pre_layers[l], f"32-layer model, prefill, layer {l}")
        for i in range(D):
            got = captured(m, stream, cfg, lambda: m.decode_step(seq, int(toks[i]), ctx + i))
            for l in range(2):
                assert_close(got[l], ref_layers[i][l], f"32-layer model, decode step {i}, layer {l}")
        # graph-replayed steps (the benchmark's path) continue from the same cache
        lg = torch.empty(cfg.vocab, device="cuda")
        m.decode_step(seq, 7, ctx + D, lg)
        assert np.all(np.isfinite(host(lg, stream)))
    finally:
        release(m)

    # the model cut to 2 layers: every output
    m, stream = gpu_model(c2, w2, max_seqs=1, max_ctx=ctx + D + 8)
    try:
        seq = m.seq_create()
        lg = torch.empty(cfg.vocab, device="cuda")
        got = captured(m, stream, c2, lambda: m.prefill(seq, prompt, lg))
        for l in range(2):
            assert_close(got[l], ref_pre_layers[l], f"2-layer model, prefill, layer {l}")
        assert_close(host(lg, stream), ref_pre, "2-layer model, prefill logits")
        kv = torch.empty(ctx, cfg.kv_dim, dtype=torch.float16, device="cuda")
        vv = torch.empty_like(kv)
        for l in range(2):
            m.debug_read_kv(seq, l, kv, vv)
            assert_close(host(kv, stream), oseq.keys(l)[:ctx].reshape(ctx, -1), f"K cache layer {l}")
            assert_close(host(vv, stream), oseq.values(l)[:ctx].reshape(ctx, -1), f"V cache layer {l}")
        for i in range(D):
            m.decode_step(seq, int(toks[i]), ctx + i, lg)
            g = host(lg, stream)
            assert_close(g, ref_logits[i], f"2-layer model, decode step {i} logits")
            check_greedy(g, ref_logits[i], f"2-layer model, decode step {i}")
    finally:
        release(m)


def teacher_forced_layers(cfg, w, m, stream, seq, steps, layers, what):
    """The layer-sliced check: for each decode step (token, position, the
    GPU's captured residual after every layer) and each layer in `layers`,
    the oracle runs that layer alone from the GPU's input to it (the
    embedding row for layer 0) and the GPU's K/V cache of the positions
    before the step, and its output and the K/V it appends at the step's
    position are compared with the GPU's.  One oracle per layer holds that
    layer's dequantised matrices for all steps."""
    torch = _torch()
    n = m.seq_length(seq)
    kv = torch.empty(n, cfg.kv_dim, dtype=torch.float16, device="cuda")
    vv = torch.empty_like(kv)
    shape = (n, cfg.n_kv_heads, cfg.head_dim)
    for l in layers:
        m.debug_read_kv(seq, l, kv, vv)
        K = host(kv, stream).reshape(shape)
        V = host(vv, stream).reshape(shape)
        orc = OracleModel(cfg, w, cache_bytes=4 * GB)
        for i, (tok, pos, got) in enumerate(steps):
            x_in = orc.embed(tok) if l == 0 else got[l - 1]
            oseq = orc.new_seq(capacity=pos + 1)
            oseq.set_layer(l, K[:pos], V[:pos])
            out = orc.layer_forward(l, x_in, pos, oseq)
            assert_close(got[l], out, f"{what}, step {i}, layer {l}")
            assert_close(K[pos], oseq.keys(l)[pos], f"{what}, step {i}, layer {l}, K appended")
            assert_close(V[pos], oseq.values(l)[pos], f"{what}, step {i}, layer {l}, V appended")
        del orc


@pytest.mark.slow
@pytest.mark.parametrize("ctx", [2048, 8192])
def test_8b_every_layer_teacher_forced(gpu_lib, w8b, ctx):
    """All 32 layers of the full 8B Q8_0 model, for two decode steps at KV
    context 2048 and 8192 on the benchmark's path (the persistent step
    kernel, which writes each layer's residual when the capture is armed):
    every layer's output and appended K/V against the oracle run from the
    GPU's input to that layer and the GPU's cache (layer-sliced; the
    independent full-model check is the 2-layer one above)."""
    cfg, w = w8b
    D = 2
    prompt = synth.prompt_tokens(cfg, ctx, seed=1)
    toks = [int(t) for t in synth.prompt_tokens(cfg, D, seed=6)]
    m, stream = gpu_model(cfg, w, max_seqs=1, max_ctx=ctx + D + 8)
    try:
        used, why = m.step_kernel_in_use()
        assert used, why
        seq = m.seq_create()
        m.prefill(seq, prompt)
        steps = []
        for i in range(D):
            got = captured(m, stream, cfg, lambda: m.decode_step(seq, toks[i], ctx + i))
            steps.append((toks[i], ctx + i, got))
        teacher_forced_layers(cfg, w, m, stream, seq, steps, range(cfg.n_layers), f"8B ctx {ctx}")
    finally:
        release(m)


def test_8b_layer_skip_and_speculative_at_full_size(gpu_lib, w8b):
    """The 8B Q8_0 model at ctx 2048, as the skip and spec workloads run it:
    the calibration's cosines are finite and in [-1, 1]; self-speculative
    greedy generation (the calibrated layers as the draft's skips, draft
    lengths 1, 3 and 9, so both verify forms) gives the library's own plain
    greedy tokens up to the first step whose top-2 logit gap is within 1e-3
    (a property that holds at any size; the tiny tests pin both to the
    oracle); with every layer skipped, a decode step's logits are the LM
    head of the embedding row (checked against the oracle on sampled vocab
    rows)."""
    torch = _torch()
    cfg, w = w8b
    P, N = 2048, 24
    prompt = synth.prompt_tokens(cfg, P, seed=1)
    m, stream = gpu_model(cfg, w, max_seqs=3, max_ctx=P + N + 32)
    try:
        base, a, b = m.seq_create(), m.seq_create(), m.seq_create()
        lg = torch.empty(cfg.vocab, device="cuda")
        m.prefill(base, prompt, lg)
        tok = int(torch.argmax(lg).item())
        m.kv_fork(base, [a])
        cos = m.layer_cosines(a, tok, P)
        assert np.all(np.isfinite(cos)) and np.all(np.abs(cos) <= 1.0 + 1e-5)
        mask = cos > 0.98
        # plain greedy with per-step logits (gaps)
        m.kv_fork(base, [a])
        plain, gaps, t = [], [], tok
        for i in range(N):
            m.decode_step(a, t, P + i, lg)
            g = host(lg, stream)
            top = np.sort(g)[-2:]
            gaps.append(top[1] - top[0])
            t = int(np.argmax(g))
            plain.append(t)
        agree = next((i for i in range(N) if gaps[i] <= 1e-3), N)
        for k in (1, 3, 9):
            m.kv_fork(base, [b])
            toks, st = m.generate_speculative(b, tok, N, mask, k)
            assert st["rounds"] + st["accepted"] == N
            assert list(toks[:agree]) == plain[:agree], f"k={k}"
            assert m.seq_length(b) == P + N
        # every layer skipped: embedding -> final norm -> LM head
        m.kv_fork(base, [a])
        m.set_layer_skip([True] * cfg.n_layers)
        m.decode_step(a, tok, P, lg)
        got = host(lg, stream)
        m.set_layer_skip(None)
        orc = OracleModel(cfg, w, cache_bytes=0)
        rows = np.unique(np.concatenate([[int(np.argmax(got))], np.random.default_rng(3).integers(0, cfg.vocab, 64)]))
        ref = orc.final_logits(orc.embed(tok), rows=rows)
        assert_close(got[rows], ref, "all layers skipped: LM head of the embedding")
    finally:
        release(m)


def test_fork_8b_q4_0_prefix_4096_eight_branches(gpu_lib):
    """8B shape, Q4_0: one prefill of a 4096-token seeded prefix, a KV fork
    into 8 branch slots, then batch-8 greedy decode of 128 tokens from each
    branch's own seeded start token.  Full model: the fork copies every
    layer's K/V bit for bit, and the forked branches decode exactly like 8
    independent prefills of the prefix.  Model cut to 2 layers: the branches'
    batch-8 logits against the oracle's forked branches (teacher-forced)."""
    torch = _torch()
    cfg = synth.get_config("fork8b")
    P, B, D = cfg.workload["prefix"], cfg.workload["branches"], cfg.workload["decode"]
    w = synth.model_weights(cfg)
    prefix = synth.prompt_tokens(cfg, P, seed=1)
    start = [100 + b for b in range(B)]
    m, stream = gpu_model(cfg, w, max_seqs=2 * B + 1, max_ctx=P + D + 8, max_batch=B)
    try:
        src = m.seq_create()
        m.prefill(src, prefix)
        dsts = [m.seq_create() for _ in range(B)]
        m.kv_fork(src, dsts)
        ks = torch.empty(P, cfg.kv_dim, dtype=torch.float16, device="cuda")
        vs, kd, vd = torch.empty_like(ks), torch.empty_like(ks), torch.empty_like(ks)
        for l in range(cfg.n_layers):
            m.debug_read_kv(src, l, ks, vs)
            for d in dsts:
                assert m.seq_length(d) == P
                m.debug_read_kv(d, l, kd, vd)
                stream.synchronize()
                assert torch.equal(kd.view(torch.int16), ks.view(torch.int16)), f"K layer {l}"
                assert torch.equal(vd.view(torch.int16), vs.view(torch.int16)), f"V layer {l}"
        last_f = torch.empty(B, cfg.vocab, device="cuda")
        toks_f = m.generate(dsts, start, D, last_f)
        indep = []
        for _ in range(B):
            s = m.seq_create()
            m.prefill(s, prefix)
            indep.append(s)
        last_i = torch.empty_like(last_f)
        toks_i = m.generate(indep, start, D, last_i)
        stream.synchronize()
        assert np.array_equal(toks_f, toks_i)
        assert torch.equal(last_f, last_i)
        for s in dsts + indep:
            assert m.seq_length(s) == P + D
        # the shared-prefix fork (pages by reference): its batched steps run
        # the cascade attention (the prefix read once for all 8 branches),
        # which changes only the fp32 summation order of attention; checked
        # step by step against the copying fork's branches, teacher-forced
        # with the copying fork's greedy tokens
        for s in indep:
            m.seq_free(s)
        shared = [m.seq_create() for _ in range(B)]
        free_before = m.kv_free_pages()
        m.kv_fork(src, shared, shared=True)
        assert m.kv_free_pages() == free_before                # 4096 = 64 full pages: nothing copied
        for s in dsts:
            m.seq_free(s)
        copies = [m.seq_create() for _ in range(B)]
        m.kv_fork(src, copies)
        out_s = torch.empty(B, cfg.vocab, device="cuda")
        out_c = torch.empty_like(out_s)
        toks = list(start)
        for i in range(8):
            m.decode_batch(shared, toks, [P + i] * B, out_s)
            m.decode_batch(copies, toks, [P + i] * B, out_c)
            gs, gc = host(out_s, stream), host(out_c, stream)
            for b in range(B):
                assert_close(gs[b], gc[b], f"shared fork (cascade) vs copied fork, branch {b} step {i}", tol=1e-4)
                toks[b] = check_greedy(gs[b], gc[b], f"shared fork branch {b} step {i}")
    finally:
        release(m)

    c2 = cut(cfg, 2)
    w2 = dict(w, layers=w["layers"][:2])
    del w
    Do = 3
    orc = OracleModel(c2, w2, cache_bytes=12 * GB)
    oseq = orc.new_seq(capacity=P + Do)
    orc.prefill(oseq, prefix)
    branches = [oseq.fork() for _ in range(B)]
    m, stream = gpu_model(c2, w2, max_seqs=B + 1, max_ctx=P + Do + 8, max_batch=B)
    try:
        src = m.seq_create()
        m.prefill(src, prefix)
        dsts = [m.seq_create() for _ in range(B)]
        m.kv_fork(src, dsts)
        toks = list(start)
        out = torch.empty(B, cfg.vocab, device="cuda")
        for i in range(Do):
            m.decode_batch(dsts, toks, [P + i] * B, out)
            got = host(out, stream)
            for b in range(B):
                ref = orc.decode_step(branches[b], toks[b], P + i)
                assert_close(got[b], ref, f"branch {b} step {i}")
                toks[b] = check_greedy(got[b], ref, f"branch {b} step {i}")
    finally:
        release(m)


def test_70b_q4_0_resident_and_streamed(gpu_lib):
    """70B shape, Q4_0, batch-1 decode at context 4096.  Full 80-layer model:
    a 24 GB device budget keeps the first layers resident and streams the
    rest through the two staging buffers; its greedy tokens and logits equal
    the fully resident model's.  Model cut to 1 layer (full width, 64/8 heads,
    FFN 28672): resident and streamed runs against the oracle."""
    torch = _torch()
    cfg = synth.get_config("70b")
    ctx = cfg.workload["ctx"]
    D = 4
    prompt = synth.prompt_tokens(cfg, ctx, seed=1)

    c1 = cut(cfg, 1)
    w1 = synth.model_weights(c1)
    orc = OracleModel(c1, w1, cache_bytes=16 * GB)
    oseq = orc.new_seq(capacity=ctx + D)
    ref_pre = orc.prefill(oseq, prompt)
    toks = [int(np.argmax(ref_pre))]
    ref_logits = []
    for i in range(D):
        ref_logits.append(orc.decode_step(oseq, toks[-1], ctx + i))
        toks.append(ops.greedy(ref_logits[-1]))
    del orc
    m, stream = gpu_model(c1, w1, max_seqs=1, max_ctx=ctx + D + 8)
    try:
        for n_res in (1, 0):
            m.set_resident_layers(n_res)
            assert m.resident_layers() == n_res
            seq = m.seq_create()
            lg = torch.empty(cfg.vocab, device="cuda")
            m.prefill(seq, prompt, lg)
            assert_close(host(lg, stream), ref_pre, f"resident={n_res} prefill logits")
            for i in range(D):
                m.decode_step(seq, toks[i], ctx + i, lg)
                g = host(lg, stream)
                assert_close(g, ref_logits[i], f"resident={n_res} decode step {i}")
                check_greedy(g, ref_logits[i], f"resident={n_res} decode step {i}")
            m.seq_free(seq)
    finally:
        release(m)
    del w1

    w = synth.model_weights(cfg)
    runs = {}
    for label, budget in (("resident", 0), ("budget", cfg.workload["budget_bytes"])):
        m, stream = gpu_model(cfg, w, max_seqs=1, max_ctx=ctx + D + 8, device_budget_bytes=budget)
        try:
            if budget:
                assert 0 < m.resident_layers() < cfg.n_layers
                assert m.device_bytes() <= budget
            seq = m.seq_create()
            lg = torch.empty(cfg.vocab, device="cuda")
            m.prefill(seq, prompt, lg)
            t0 = int(np.argmax(host(lg, stream)))
            last = torch.empty(1, cfg.vocab, device="cuda")
            gen = m.generate([seq], [t0], D, last)
            runs[label] = (t0, np.asarray(gen)[:, 0].copy(), host(last, stream)[0])
            if budget:
                # one more step with the capture armed; sampled resident and
                # streamed layers, layer-sliced against the oracle
                n_res = m.resident_layers()
                tok, pos = int(np.asarray(gen)[-1, 0]), ctx + D
                got = captured(m, stream, cfg, lambda: m.decode_step(seq, tok, pos))
                sample = sorted({0, n_res - 1, n_res, (n_res + cfg.n_layers) // 2, cfg.n_layers - 1})
                teacher_forced_layers(cfg, w, m, stream, seq, [(tok, pos, got)], sample,
                                      f"70B, 24 GB budget ({n_res} resident)")
        finally:
            release(m)
    assert runs["resident"][0] == runs["budget"][0]
    assert np.array_equal(runs["resident"][1], runs["budget"][1])
    # the fully resident model decodes through the persistent step kernel,
    # the budgeted one through the separate kernels (its layers stream):
    # the same arithmetic in other fp32 reduction orders, over 80 layers;
    # each path is held to the oracle's 2e-3 above and layer by layer
    assert_close(runs["budget"][2], runs["resident"][2], "streamed vs resident logits", tol=1e-3)
