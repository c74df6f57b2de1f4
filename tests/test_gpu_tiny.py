"""GPU parity on the tiny configuration (2 layers, hidden 256, 4/2 heads,
head_dim 64, FFN 688, vocab 1024, Q8_0) and a Q4_0 twin, through the C ABI.
"""
import numpy as np
import pytest

import synth
from oracle import OracleModel, ops, quant
from synth.configs import ModelConfig

from parity import assert_close, check_greedy

pytestmark = pytest.mark.gpu

TINY = synth.get_config("tiny")
TINY_Q4 = ModelConfig("tinyq4", 2, 256, 4, 2, 64, 688, 1024, 10000.0, 4, 0.02)


def _torch():
    import torch
    return torch


@pytest.fixture(scope="module", params=[(TINY, "1"), (TINY_Q4, "1"), (TINY, "0")],
                ids=["q8_0-persistent", "q4_0-persistent", "q8_0-separate"])
def setup(request, gpu_lib):
    """The tiny model, decoding with the persistent step kernel or with the
    separate kernels (DLS_STEP_KERNEL is read when the model is created)."""
    import os
    torch = _torch()
    from decode_llama_step_gb300 import dls
    cfg, step_kernel = request.param
    w = synth.model_weights(cfg)
    stream = torch.cuda.Stream()
    old = os.environ.get("DLS_STEP_KERNEL")
    os.environ["DLS_STEP_KERNEL"] = step_kernel
    try:
        m = dls.Model(cfg, w, max_seqs=6, max_ctx=160, max_batch=4, page_tokens=32, stream=stream)
        m.step_kernel = step_kernel
        used, why = m.step_kernel_in_use()
        assert used == (step_kernel == "1"), why
    finally:
        if old is None:
            del os.environ["DLS_STEP_KERNEL"]
        else:
            os.environ["DLS_STEP_KERNEL"] = old
    orc = OracleModel(cfg, w)
    yield cfg, w, m, orc, stream
    m.close()


def test_dequant_bit_exact(setup):
    torch = _torch()
    cfg, w, m, orc, stream = setup
    shapes = synth.matrix_shapes(cfg)
    for l in range(cfg.n_layers):
        for name in synth.LAYER_MATRICES:
            rows, cols = shapes[name]
            out = torch.empty(rows, cols, device="cuda")
            m.debug_dequant(l, name, out)
            stream.synchronize()
            ref = quant.matrix(w["layers"][l][name], rows, cols, cfg.wtype)
            got = out.cpu().numpy().astype(np.float64)
            assert np.array_equal(got, ref), f"layer {l} {name}"
    for name in ("tok_embd", "output"):
        out = torch.empty(cfg.vocab, cfg.hidden, device="cuda")
        m.debug_dequant(0, name, out)
        stream.synchronize()
        ref = quant.matrix(w[name], cfg.vocab, cfg.hidden, cfg.wtype)
        assert np.array_equal(out.cpu().numpy().astype(np.float64), ref), name


def test_gemv_every_matrix(setup):
    torch = _torch()
    cfg, w, m, orc, stream = setup
    shapes = synth.matrix_shapes(cfg)
    shapes["output"] = (cfg.vocab, cfg.hidden)
    for name, (rows, cols) in shapes.items():
        x = synth.normal(synth.stream_key("gemv-x", name), cols, 1.0).astype(np.float32)
        xd = torch.from_numpy(x).cuda()
        y = torch.empty(rows, device="cuda")
        m.debug_gemv(1, name, xd, y)
        stream.synchronize()
        ref = orc.matmul(1 if name != "output" else None, name, x.astype(np.float64))
        # The kernel quantises each lane's 16/32-element activation slice to
        # int16 (step = slice max / 32767) and accumulates code x activation
        # products exactly in int32: relative error ~1e-5, far inside the
        # layer tolerance of 2e-3
        assert_close(y.cpu().numpy(), ref, f"gemv {name}", tol=1e-4)


def _run_against_oracle(cfg, m, orc, n_prompt, n_decode, seed=1):
    torch = _torch()
    prompt = synth.prompt_tokens(cfg, n_prompt, seed=seed)
    seq = m.seq_create()
    try:
        logits = torch.empty(cfg.vocab, device="cuda")
        cap = torch.empty(cfg.n_layers, cfg.hidden, device="cuda")
        m.prefill(seq, prompt, logits)
        oseq = orc.new_seq()
        ref = orc.prefill(oseq, prompt)
        assert_close(logits.cpu().numpy(), ref, "prefill logits")
        tok = check_greedy(logits.cpu().numpy(), ref, "prefill")
        for i in range(n_decode):
            pos = n_prompt + i
            m.debug_capture(cap)
            m.decode_step(seq, tok, pos, logits)
            ocap = []
            ref = orc.decode_step(oseq, tok, pos, capture=ocap)
            got_cap = cap.cpu().numpy()
            for l in range(cfg.n_layers):
                assert_close(got_cap[l], ocap[l], f"step {i} layer {l} residual")
            assert_close(logits.cpu().numpy(), ref, f"step {i} logits")
            tok = check_greedy(logits.cpu().numpy(), ref, f"step {i}")
        assert m.seq_length(seq) == n_prompt + n_decode
    finally:
        m.seq_free(seq)


def test_prefill_and_greedy_decode_parity(setup):
    cfg, w, m, orc, stream = setup
    _run_against_oracle(cfg, m, orc, 16, 32)


def test_decode_across_page_boundaries(setup):
    # 32-token pages: positions 31/32/33 and 63/64/65 cross pages
    cfg, w, m, orc, stream = setup
    _run_against_oracle(cfg, m, orc, 30, 37, seed=5)


def test_graph_replay_matches_eager(setup):
    # decode without capture replays a captured graph; with capture armed
    # the same kernels (the persistent step kernel where the shape has one)
    # launch eagerly and also write the per-layer residuals, which must not
    # change the logits.
    torch = _torch()
    cfg, w, m, orc, stream = setup
    prompt = synth.prompt_tokens(cfg, 9, seed=3)
    a, b = m.seq_create(), m.seq_create()
    try:
        la = torch.empty(cfg.vocab, device="cuda")
        lb = torch.empty(cfg.vocab, device="cuda")
        m.prefill(a, prompt)
        m.prefill(b, prompt)
        cap = torch.empty(cfg.n_layers, cfg.hidden, device="cuda")
        m.decode_step(a, 7, 9, la)
        m.debug_capture(cap)
        m.decode_step(b, 7, 9, lb)
        stream.synchronize()
        assert_close(la.cpu().numpy(), lb.cpu().numpy(), "graph vs eager", tol=1e-4)
        # replaying again gives the same bits (the step is deterministic)
        lc = torch.empty(cfg.vocab, device="cuda")
        c = m.seq_create()
        m.prefill(c, prompt)
        m.decode_step(c, 7, 9, lc)
        stream.synchronize()
        assert torch.equal(la, lc)
        m.seq_free(c)
    finally:
        m.seq_free(a)
        m.seq_free(b)


def test_persistent_step_matches_separate_kernels(setup, monkeypatch):
    torch = _torch()
    from decode_llama_step_gb300 import dls
    cfg, w, m, orc, stream = setup
    other = "0" if m.step_kernel == "1" else "1"   # the other decode path
    monkeypatch.setenv("DLS_STEP_KERNEL", other)
    m2 = dls.Model(cfg, w, max_seqs=2, max_ctx=160, page_tokens=32, stream=stream)
    monkeypatch.delenv("DLS_STEP_KERNEL")
    try:
        prompt = synth.prompt_tokens(cfg, 40, seed=4)
        outs = []
        for mm in (m, m2):
            s = mm.seq_create()
            lg = torch.empty(cfg.vocab, device="cuda")
            mm.prefill(s, prompt, lg)
            toks = mm.generate([s], [int(torch.argmax(lg))], 6)
            mm.decode_step(s, 3, 46, lg)
            stream.synchronize()
            outs.append((lg.cpu().numpy(), toks))
            mm.seq_free(s)
        assert_close(outs[0][0], outs[1][0], "persistent vs separate kernels", tol=1e-4)
        # greedy tokens agree where the pick is not a near tie
        assert np.mean(outs[0][1] == outs[1][1]) >= 0.5
    finally:
        m2.close()


def test_generate_matches_oracle_greedy(setup):
    cfg, w, m, orc, stream = setup
    prompt = synth.prompt_tokens(cfg, 16)
    seq = m.seq_create()
    try:
        m.prefill(seq, prompt)
        oseq = orc.new_seq()
        ref = orc.prefill(oseq, prompt)
        tok0 = int(np.argmax(ref))
        toks = m.generate([seq], [tok0], 12)[:, 0]
        otoks, ologits = orc.greedy_decode(oseq, tok0, 12)
        for i in range(12):
            gap = ops.top2_gap(ologits[i])
            if gap <= 1e-2:
                break  # beyond here the runs may legitimately diverge
            assert toks[i] == otoks[i], f"step {i}"
        assert m.seq_length(seq) == 16 + 12
    finally:
        m.seq_free(seq)


def test_decode_batch_equals_single_steps(setup):
    torch = _torch()
    cfg, w, m, orc, stream = setup
    seqs = [m.seq_create() for _ in range(3)]
    try:
        for i, s in enumerate(seqs):
            m.prefill(s, synth.prompt_tokens(cfg, 5 + 3 * i, seed=10 + i))
        pos = [m.seq_length(s) for s in seqs]
        toks = [3, 500, 1023]
        out = torch.empty(3, cfg.vocab, device="cuda")
        m.decode_batch(seqs, toks, pos, out)
        ref_logits = []
        for i, s in enumerate(seqs):
            oseq = orc.new_seq()
            orc.prefill(oseq, synth.prompt_tokens(cfg, 5 + 3 * i, seed=10 + i))
            ref_logits.append(orc.decode_step(oseq, toks[i], pos[i]))
        for i in range(3):
            assert_close(out[i].cpu().numpy(), ref_logits[i], f"batch row {i}")
    finally:
        for s in seqs:
            m.seq_free(s)


@pytest.mark.parametrize("mode", ["rg", "tc"])
@pytest.mark.parametrize("cfg", [TINY, TINY_Q4], ids=["q8_0", "q4_0"])
def test_batch_paths_match_oracle(gpu_lib, mode, cfg):
    """Both batched-step paths (the multi-row CUDA-core GEMV and the
    small-batch tensor-core GEMM, DLS_BATCH_GEMM, read at model creation) at
    every batch size 2..8 against the oracle, rows at different lengths."""
    import os
    torch = _torch()
    from decode_llama_step_gb300 import dls
    w = synth.model_weights(cfg)
    stream = torch.cuda.Stream()
    old = os.environ.get("DLS_BATCH_GEMM")
    os.environ["DLS_BATCH_GEMM"] = mode
    try:
        m = dls.Model(cfg, w, max_seqs=8, max_ctx=96, max_batch=8, page_tokens=32, stream=stream)
    finally:
        if old is None:
            del os.environ["DLS_BATCH_GEMM"]
        else:
            os.environ["DLS_BATCH_GEMM"] = old
    orc = OracleModel(cfg, w)
    try:
        prompts = [synth.prompt_tokens(cfg, 4 + 5 * i, seed=60 + i) for i in range(8)]
        refs = []
        for p in prompts:
            o = orc.new_seq()
            orc.prefill(o, p)
            refs.append(o)
        for n in (2, 3, 4, 5, 8):
            seqs = [m.seq_create() for _ in range(n)]
            try:
                for s, p in zip(seqs, prompts):
                    m.prefill(s, p)
                toks = [(37 * i + n) % cfg.vocab for i in range(n)]
                pos = [m.seq_length(s) for s in seqs]
                out = torch.empty(n, cfg.vocab, device="cuda")
                m.decode_batch(seqs, toks, pos, out)
                stream.synchronize()
                for i in range(n):
                    ref = orc.decode_step(refs[i].fork(), toks[i], pos[i])
                    assert_close(out[i].cpu().numpy(), ref, f"{mode} n={n} row {i}")
            finally:
                for s in seqs:
                    m.seq_free(s)
    finally:
        m.close()


def test_generate_batch_matches_oracle(setup):
    # three sequences of different lengths decode together on the tensor-core
    # path; every step's token is the oracle's greedy token while the
    # oracle's top-2 gap exceeds 1e-2
    torch = _torch()
    cfg, w, m, orc, stream = setup
    lens = (9, 33, 20)
    seqs = [m.seq_create() for _ in lens]
    try:
        oseqs, toks0 = [], []
        for i, (s, n) in enumerate(zip(seqs, lens)):
            prompt = synth.prompt_tokens(cfg, n, seed=40 + i)
            m.prefill(s, prompt)
            oseq = orc.new_seq()
            toks0.append(int(np.argmax(orc.prefill(oseq, prompt))))
            oseqs.append(oseq)
        last = torch.empty(len(lens), cfg.vocab, device="cuda")
        toks = m.generate(seqs, toks0, 10, last)
        for i, oseq in enumerate(oseqs):
            otoks, ologits = orc.greedy_decode(oseq, toks0[i], 10)
            for t in range(10):
                if ops.top2_gap(ologits[t]) <= 1e-2:
                    break
                assert toks[t, i] == otoks[t], f"row {i} step {t}"
            else:
                assert_close(last[i].cpu().numpy(), ologits[-1], f"row {i} final logits")
        for s, n in zip(seqs, lens):
            assert m.seq_length(s) == n + 10
    finally:
        for s in seqs:
            m.seq_free(s)


def test_kv_fork_bit_exact_and_continues(setup):
    torch = _torch()
    cfg, w, m, orc, stream = setup
    prefix = synth.prompt_tokens(cfg, 45, seed=7)   # partial last page (45 = 32 + 13)
    src = m.seq_create()
    dsts = [m.seq_create(), m.seq_create()]
    indep = m.seq_create()
    try:
        m.prefill(src, prefix)
        m.prefill(dsts[0], synth.prompt_tokens(cfg, 70, seed=8))  # old contents dropped by the fork
        m.kv_fork(src, dsts)
        n, kvd = 45, cfg.n_kv_heads * cfg.head_dim
        for l in range(cfg.n_layers):
            ks = torch.empty(n, kvd, dtype=torch.float16, device="cuda")
            vs = torch.empty_like(ks)
            m.debug_read_kv(src, l, ks, vs)
            for d in dsts:
                assert m.seq_length(d) == n
                kd = torch.empty_like(ks)
                vd = torch.empty_like(ks)
                m.debug_read_kv(d, l, kd, vd)
                stream.synchronize()
                assert torch.equal(kd.view(torch.int16), ks.view(torch.int16))
                assert torch.equal(vd.view(torch.int16), vs.view(torch.int16))
        # a branch continues RoPE at the prefix length and matches an independent prefill
        m.prefill(indep, prefix)
        lf = torch.empty(cfg.vocab, device="cuda")
        li = torch.empty(cfg.vocab, device="cuda")
        m.decode_step(dsts[1], 11, n, lf)
        m.decode_step(indep, 11, n, li)
        stream.synchronize()
        assert torch.equal(lf, li)
        from decode_llama_step_gb300 import dls
        with pytest.raises(dls.DlsError) as e:
            m.decode_step(dsts[0], 11, 0, lf)   # restarting at position 0 is refused
        assert e.value.code == dls.DLS_ERR_STATE
    finally:
        for s in [src, *dsts, indep]:
            m.seq_free(s)


def test_kv_fork_shared_pages(setup):
    """The shared-prefix fork: branches hold the source's full pages by
    reference and a private copy of the partly filled page; they read the
    source's K/V bytes exactly, decode exactly like a copied branch, never
    disturb each other or the source, and outlive it; every page comes back
    to the pool when all holders are freed."""
    torch = _torch()
    cfg, w, m, orc, stream = setup
    free0 = m.kv_free_pages()
    n = 45                                        # one full 32-token page + 13 positions of the next
    prefix = synth.prompt_tokens(cfg, n, seed=7)
    src, a, b, cpy = (m.seq_create() for _ in range(4))
    live = [src, a, b, cpy]
    try:
        m.prefill(src, prefix)
        held = free0 - m.kv_free_pages()
        assert held == 2
        m.kv_fork(src, [a, b], shared=True)
        assert free0 - m.kv_free_pages() == held + 2          # one fresh page per branch
        m.kv_fork(src, [cpy])                                  # the copy form, for comparison
        kvd = cfg.n_kv_heads * cfg.head_dim

        def kv(seq, l):
            k = torch.empty(n, kvd, dtype=torch.float16, device="cuda")
            v = torch.empty_like(k)
            m.debug_read_kv(seq, l, k, v)
            stream.synchronize()
            return k.view(torch.int16).clone(), v.view(torch.int16).clone()

        src_kv = [kv(src, l) for l in range(cfg.n_layers)]
        for d in (a, b):
            assert m.seq_length(d) == n
            for l in range(cfg.n_layers):
                kd, vd = kv(d, l)
                assert torch.equal(kd, src_kv[l][0]) and torch.equal(vd, src_kv[l][1])
        la, lb, lc = (torch.empty(cfg.vocab, device="cuda") for _ in range(3))
        m.decode_step(a, 11, n, la)
        m.decode_step(cpy, 11, n, lc)
        m.decode_step(b, 500, n, lb)                           # a different token into b's own page
        stream.synchronize()
        assert torch.equal(la, lc)
        for l in range(cfg.n_layers):                          # the source is untouched
            ks, vs = kv(src, l)
            assert torch.equal(ks, src_kv[l][0]) and torch.equal(vs, src_kv[l][1])
        m.seq_free(src)                                        # the branches keep the shared page
        live.remove(src)
        m.decode_step(a, 12, n + 1, la)
        m.decode_step(cpy, 12, n + 1, lc)
        stream.synchronize()
        assert torch.equal(la, lc)
        ref = orc.new_seq()
        orc.prefill(ref, prefix)
        orc.decode_step(ref, 11, n)
        assert_close(la.cpu().numpy(), orc.decode_step(ref, 12, n + 1), "branch after a shared fork")
    finally:
        for q in live:
            m.seq_free(q)
    assert m.kv_free_pages() == free0


@pytest.mark.parametrize("skipped", [0, 1])
def test_layer_skip_calibration_and_decode(setup, skipped):
    """Layer skip (engine page, sections 2.5, 3.5, 4.5): the per-layer cosine
    calibration matches the oracle's, and decode steps with a layer skipped
    match the oracle with the same layer skipped, one step at a time and
    through greedy generation."""
    torch = _torch()
    cfg, w, m, orc, stream = setup
    prompt = synth.prompt_tokens(cfg, 20, seed=21)
    seq = m.seq_create()
    try:
        m.prefill(seq, prompt)
        oseq = orc.new_seq()
        orc.prefill(oseq, prompt)
        cos = m.layer_cosines(seq, 17, 20)
        ocos = orc.layer_cosines(oseq, 17, 20)
        np.testing.assert_allclose(cos, ocos, atol=2e-4)
        mask = [l == skipped for l in range(cfg.n_layers)]
        m.set_layer_skip(mask)
        lg = torch.empty(cfg.vocab, device="cuda")
        tok = 5
        for i in range(4):
            m.decode_step(seq, tok, 21 + i, lg)
            stream.synchronize()
            ref = orc.decode_step(oseq, tok, 21 + i, skip={skipped})
            got = lg.cpu().numpy()
            assert_close(got, ref, f"skip {skipped} step {i}")
            tok = check_greedy(got, ref, f"skip {skipped} step {i}")
        toks = m.generate([seq], [tok], 6)[:, 0]
        otoks, ologits = orc.greedy_decode(oseq, tok, 6, skip={skipped})
        for i in range(6):
            if ops.top2_gap(ologits[i]) <= 1e-2:
                break
            assert toks[i] == otoks[i], f"skip {skipped} generate step {i}"
    finally:
        m.set_layer_skip(None)
        m.seq_free(seq)


def test_verify_scores_every_position(setup):
    """dls_verify: n tokens through every layer at once, every row's logits
    and greedy pick against the oracle's all-row prefill."""
    torch = _torch()
    cfg, w, m, orc, stream = setup
    prompt = synth.prompt_tokens(cfg, 30, seed=31)
    seq = m.seq_create()
    try:
        m.prefill(seq, prompt[:25])
        oseq = orc.new_seq()
        orc.prefill(oseq, prompt[:25])
        lg = torch.empty(5, cfg.vocab, device="cuda")
        picks = m.verify(seq, prompt[25:], lg)
        stream.synchronize()
        ref = orc.prefill(oseq, prompt[25:], all_logits=True)
        got = lg.cpu().numpy()
        for i in range(5):
            assert_close(got[i], ref[i], f"verify row {i}")
            check_greedy(got[i], ref[i], f"verify row {i}")
            assert picks[i] == int(np.argmax(got[i]))
        assert m.seq_length(seq) == 30
        # the cache it filled serves the next decode step
        m.decode_step(seq, 7, 30, lg[0])
        stream.synchronize()
        assert_close(lg[0].cpu().numpy(), orc.decode_step(oseq, 7, 30), "decode after verify")
    finally:
        m.seq_free(seq)


def test_seq_truncate(setup):
    """Truncation: decoding after a cut equals decoding a sequence that never
    went further; cutting back into a page shared by a fork gives the
    sequence a private copy and leaves the other holder's K/V untouched."""
    torch = _torch()
    from decode_llama_step_gb300 import dls
    cfg, w, m, orc, stream = setup
    free0 = m.kv_free_pages()
    prompt = synth.prompt_tokens(cfg, 70, seed=41)
    a, b, c = (m.seq_create() for _ in range(3))
    try:
        m.prefill(a, prompt[:40])
        m.prefill(b, prompt[:40])
        m.prefill(a, prompt[40:70])                  # a: 70 positions = 3 pages of 32
        assert free0 - m.kv_free_pages() == 3 + 2
        m.seq_truncate(a, 40)
        assert m.seq_length(a) == 40 and free0 - m.kv_free_pages() == 2 + 2
        la, lb = torch.empty(cfg.vocab, device="cuda"), torch.empty(cfg.vocab, device="cuda")
        m.decode_step(a, 9, 40, la)
        m.decode_step(b, 9, 40, lb)
        stream.synchronize()
        assert torch.equal(la, lb)
        with pytest.raises(dls.DlsError) as e:
            m.seq_truncate(a, 42)
        assert e.value.code == dls.DLS_ERR_ARG
        # shared pages: c holds a's first page (positions 0..31) by reference
        m.kv_fork(a, [c], shared=True)
        kvd = cfg.n_kv_heads * cfg.head_dim

        def kv(seq, n):
            k = torch.empty(n, kvd, dtype=torch.float16, device="cuda")
            v = torch.empty_like(k)
            m.debug_read_kv(seq, 1, k, v)
            stream.synchronize()
            return k.clone(), v.clone()

        before = kv(a, 41)
        used = free0 - m.kv_free_pages()
        m.seq_truncate(c, 20)                         # into the shared page: c gets its own copy
        assert free0 - m.kv_free_pages() == used + 1 - 1   # c's private tail page freed, one copy taken
        assert torch.equal(kv(c, 20)[0], before[0][:20])
        m.decode_step(c, 3, 20)                       # writes position 20 of c's copy only
        after = kv(a, 41)
        assert torch.equal(after[0], before[0]) and torch.equal(after[1], before[1])
        oc = orc.new_seq()
        orc.prefill(oc, prompt[:20])
        orc.decode_step(oc, 3, 20)
        m.decode_step(c, 4, 21, lb)
        stream.synchronize()
        assert_close(lb.cpu().numpy(), orc.decode_step(oc, 4, 21), "decode after a copy-on-write cut")
    finally:
        for q in (a, b, c):
            m.seq_free(q)
    assert m.kv_free_pages() == free0


def _oracle_seq(orc, prompt):
    s = orc.new_seq()
    orc.prefill(s, prompt)
    return s


def _check_speculative(cfg, m, orc, seq, prompt, tok, n, mask, k, what):
    """Speculative generation through the library against the oracle: the
    tokens are the oracle's full greedy run up to its first near-tie, and
    when no greedy pick of the oracle's speculative run (draft or full) is
    near a tie, the rounds and acceptance counts are the oracle's too."""
    toks, st = m.generate_speculative(seq, tok, n, mask, k)
    assert st["rounds"] + st["accepted"] == n and st["accepted"] <= st["drafted"], f"{what}: {st}"
    otoks, ologits = orc.greedy_decode(_oracle_seq(orc, prompt), tok, n)
    for i in range(n):
        if ops.top2_gap(ologits[i]) <= 1e-2:
            break  # beyond here the runs may legitimately diverge
        assert toks[i] == otoks[i], f"{what}: step {i}"
    skip = {l for l in range(cfg.n_layers) if mask[l]}
    stoks, ost = orc.speculative_decode(_oracle_seq(orc, prompt), tok, n, skip, k)
    assert stoks == otoks
    if ost["min_gap"] > 1e-3:
        assert list(toks) == otoks, f"{what}: tokens"
        assert (st["rounds"], st["drafted"], st["accepted"]) == \
            (ost["rounds"], ost["drafted"], ost["accepted"]), f"{what}: {st} vs {ost}"
    return toks, st


@pytest.mark.parametrize("k", [1, 3, 9])  # 9: a verify pass of 10 positions (the prefill-chunk form)
@pytest.mark.parametrize("draft", ["skip-last", "skip-first", "skip-all", "full"])
def test_speculative_decode_matches_oracle(setup, draft, k):
    """Self-speculative greedy decoding (engine page, sections 3.5 and 5.3):
    the tokens, the rounds and the acceptance counts equal the oracle's, the
    tokens are the full model's greedy run (the library's own plain greedy
    generation too), and the sequence ends where plain generation would."""
    cfg, w, m, orc, stream = setup
    L = cfg.n_layers
    mask = {"skip-last": [l == L - 1 for l in range(L)], "skip-first": [l == 0 for l in range(L)],
            "skip-all": [True] * L, "full": [False] * L}[draft]
    prompt = synth.prompt_tokens(cfg, 24, seed=51)
    seq, ref = m.seq_create(), m.seq_create()
    try:
        m.prefill(seq, prompt)
        m.prefill(ref, prompt)
        tok = int(np.argmax(orc.prefill(orc.new_seq(), prompt)))
        n = 13
        toks, st = _check_speculative(cfg, m, orc, seq, prompt, tok, n, mask, k, f"{draft} k={k}")
        if draft == "full":
            assert st["accepted"] == st["drafted"]
        assert m.seq_length(seq) == 24 + n
        plain = m.generate([ref], [tok], n)[:, 0]
        _, ologits = orc.greedy_decode(_oracle_seq(orc, prompt), tok, n)
        for i in range(n):
            if ops.top2_gap(ologits[i]) <= 1e-2:
                break
            assert toks[i] == plain[i], f"step {i}"
        # one token: a round with no draft
        one, st1 = m.generate_speculative(seq, int(toks[-1]), 1, mask, k)
        assert st1 == {"rounds": 1, "drafted": 0, "accepted": 0}
        assert m.seq_length(seq) == 24 + n + 1
    finally:
        m.seq_free(seq)
        m.seq_free(ref)


def test_speculative_decode_with_streamed_layers(setup):
    """The pages' configuration: resident layers draft, the streamed rest
    only joins the verify pass (draft steps copy nothing in)."""
    cfg, w, m, orc, stream = setup
    L = cfg.n_layers
    prompt = synth.prompt_tokens(cfg, 24, seed=52)
    m.set_resident_layers(1)
    seq = m.seq_create()
    try:
        m.prefill(seq, prompt)
        tok = int(np.argmax(orc.prefill(orc.new_seq(), prompt)))
        mask = [l >= 1 for l in range(L)]
        _check_speculative(cfg, m, orc, seq, prompt, tok, 11, mask, 3, "streamed")
        assert m.seq_length(seq) == 24 + 11
    finally:
        m.seq_free(seq)
        m.set_resident_layers(L)


def test_streamed_layers_match_resident(setup):
    torch = _torch()
    cfg, w, m, orc, stream = setup
    prompt = synth.prompt_tokens(cfg, 12, seed=9)
    outs = []
    for n_res in (cfg.n_layers, 0, 1):
        m.set_resident_layers(n_res)
        assert m.resident_layers() == n_res
        s = m.seq_create()
        lg = torch.empty(cfg.vocab, device="cuda")
        m.prefill(s, prompt)
        m.decode_step(s, 5, 12, lg)
        stream.synchronize()
        outs.append(lg.clone())
        m.seq_free(s)
    m.set_resident_layers(cfg.n_layers)
    # streamed layers run the separate-kernel step over the staging buffers:
    # identical for any resident count, and equal to the resident step to
    # fp32 rounding
    assert torch.equal(outs[1], outs[2])
    assert_close(outs[0].cpu().numpy(), outs[1].cpu().numpy(), "resident vs streamed", tol=1e-4)


def test_error_paths(setup):
    torch = _torch()
    from decode_llama_step_gb300 import dls
    cfg, w, m, orc, stream = setup
    s = m.seq_create()
    try:
        with pytest.raises(dls.DlsError) as e:
            m.decode_step(s, cfg.vocab, 0)
        assert e.value.code == dls.DLS_ERR_ARG
        with pytest.raises(dls.DlsError) as e:
            m.decode_step(s, 1, 3)
        assert e.value.code == dls.DLS_ERR_STATE
        with pytest.raises(dls.DlsError) as e:
            m.prefill(s, np.zeros(161, dtype=np.int32))
        assert e.value.code == dls.DLS_ERR_CAPACITY
        assert m.seq_length(s) == 0
        with pytest.raises(dls.DlsError):
            m.kv_fork(s, [s])
    finally:
        m.seq_free(s)


def test_attention_op_against_oracle(gpu_lib):
    torch = _torch()
    from decode_llama_step_gb300 import dls
    rng = np.random.default_rng(3)
    for nh, nkv, hd in [(4, 2, 64), (32, 8, 128), (8, 8, 32), (64, 8, 128)]:
        pt, maxp = 32, 12
        lengths = np.array([1, 2, 31, 32, 33, 65, 200, 384][: 4 if nh == 64 else 8], dtype=np.int32)
        nb = len(lengths)
        npages = nb * maxp
        kp = rng.standard_normal((npages, nkv, pt, hd)).astype(np.float16)
        vp = rng.standard_normal((npages, nkv, pt, hd)).astype(np.float16)
        table = rng.permutation(npages).astype(np.int32).reshape(nb, maxp)
        q = rng.standard_normal((nb, nh, hd)).astype(np.float32) * 2
        tk, tv = torch.from_numpy(kp).cuda(), torch.from_numpy(vp).cuda()
        tt, tl = torch.from_numpy(table).cuda(), torch.from_numpy(lengths).cuda()
        tq = torch.from_numpy(q).cuda()
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        for splits in (1, 3, 7, 0):
            # splits = 0: the call chooses; a workspace sized for the most
            # splits (128) serves any choice
            wsb = dls.attention_workspace_bytes(nb, nh, nkv, hd, splits or 128)
            ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
            o = torch.empty(nb, nh, hd, device="cuda")
            dls.attention_decode(tq, tk, tv, tt, tl, o, ws, wsb, nb, nh, nkv, hd, pt, maxp, splits, status=status)
            dls.attention_status(status)
            got = o.cpu().numpy()
            for b in range(nb):
                n = lengths[b]
                pos = np.arange(n)
                pages = table[b][pos // pt]
                K = kp[pages, :, pos % pt, :].astype(np.float64)   # [n, nkv, hd]
                V = vp[pages, :, pos % pt, :].astype(np.float64)
                ref = ops.attention(q[b].astype(np.float64), K, V)
                assert_close(got[b], ref, f"attn nh={nh} nkv={nkv} hd={hd} n={n} splits={splits}", tol=1e-5)
            # the call leaves its arrival counters at zero for the next call
            assert int(ws[: nb * nkv * 4].view(torch.int32).abs().sum()) == 0


def test_attention_op_reports_bad_pages_and_lengths(gpu_lib):
    # a negative page-table entry and a length outside 1..page_tokens*max_pages
    # are reported through the status word (the kernel skips the missing
    # page and clamps the length; nothing is read out of bounds)
    torch = _torch()
    from decode_llama_step_gb300 import dls
    rng = np.random.default_rng(4)
    nb, nh, nkv, hd, pt, maxp = 2, 4, 2, 64, 32, 4
    kp = torch.from_numpy(rng.standard_normal((nb * maxp, nkv, pt, hd)).astype(np.float16)).cuda()
    vp = torch.from_numpy(rng.standard_normal((nb * maxp, nkv, pt, hd)).astype(np.float16)).cuda()
    q = torch.from_numpy(rng.standard_normal((nb, nh, hd)).astype(np.float32)).cuda()
    o = torch.empty(nb, nh, hd, device="cuda")
    wsb = dls.attention_workspace_bytes(nb, nh, nkv, hd, 2)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    good = np.arange(nb * maxp, dtype=np.int32).reshape(nb, maxp)
    cases = [(good, [100, 128], None),
             (np.where(good == 5, -1, good), [100, 128], dls.DLS_ERR_STATE),   # row 1's page 1 missing
             (good, [0, 128], dls.DLS_ERR_STATE),                              # empty row
             (good, [100, 129], dls.DLS_ERR_STATE)]                            # past the table
    for table, lens, want in cases:
        tt = torch.from_numpy(np.ascontiguousarray(table, dtype=np.int32)).cuda()
        tl = torch.from_numpy(np.array(lens, dtype=np.int32)).cuda()
        dls.attention_decode(q, kp, vp, tt, tl, o, ws, wsb, nb, nh, nkv, hd, pt, maxp, 2, status=status)
        if want is None:
            dls.attention_status(status)
        else:
            with pytest.raises(dls.DlsError) as e:
                dls.attention_status(status)
            assert e.value.code == want
        for fn in ("noalloc",):
            dls.attention_decode_noalloc(q, kp, vp, tt, tl, o, nb, nh, nkv, hd, pt, maxp, 2, status=status)
            if want is None:
                dls.attention_status(status)
            else:
                with pytest.raises(dls.DlsError) as e:
                    dls.attention_status(status)
                assert e.value.code == want, fn
