"""Cascade attention for batched steps over a shared prefix (the SwarmKV
page, section 3: paged sharing of a prefix; section 10: device-side
materialisation): branches forked with shared pages hold the prefix's KV
pages by reference, and each batched step reads those pages once for all
branches (one partial per KV head and split), then merges them with each
branch's own suffix.  Checked against the oracle's forked branches (full
attention over prefix + suffix, fp64) and against the same steps with the
cascade switched off (DLS_CASCADE=0, read at model creation).
"""
import os

import numpy as np
import pytest

import synth
from oracle import OracleModel, ops
from synth.configs import ModelConfig

from parity import assert_close, check_greedy

pytestmark = pytest.mark.gpu

TINY = synth.get_config("tiny")
# a group of 8 query heads per KV head: 8 branches fill 64 rows of the
# tensor-core kernel's tile; head_dim 64 and 128
G8 = ModelConfig("g8", 2, 512, 8, 1, 64, 1024, 1024, 10000.0, 8, 0.02)
G8H128 = ModelConfig("g8h128", 1, 1024, 8, 1, 128, 1024, 1024, 10000.0, 8, 0.02)


def _model(cfg, w, cascade: bool, tc: str, max_batch=8):
    import torch
    from decode_llama_step_gb300 import dls
    env = {"DLS_CASCADE": "1" if cascade else "0", "DLS_CASCADE_TC": tc}
    old = {k: os.environ.get(k) for k in env}
    os.environ.update(env)
    try:
        stream = torch.cuda.Stream()
        return dls.Model(cfg, w, max_seqs=2 * max_batch + 2, max_ctx=320, max_batch=max_batch, page_tokens=32,
                         stream=stream), stream
    finally:
        for k, v in old.items():
            if v is None:
                del os.environ[k]
            else:
                os.environ[k] = v


@pytest.fixture(scope="module", params=[(TINY, "1"), (TINY, "0"), (G8, "1"), (G8H128, "1")],
                ids=["tiny-tensor-cores", "tiny-cuda-cores", "g8-tensor-cores", "g8-hd128-tensor-cores"])
def models(request, gpu_lib):
    """The shared-prefix pass on the tensor cores (casc_tc.cu) or on the
    CUDA cores (DLS_CASCADE_TC=0), beside the same model without cascade
    attention."""
    cfg, tc = request.param
    w = synth.model_weights(cfg)
    on, s_on = _model(cfg, w, True, tc)
    off, s_off = _model(cfg, w, False, tc)
    yield cfg, on, s_on, off, s_off, OracleModel(cfg, w)
    on.close()
    off.close()


@pytest.mark.parametrize("prefix,branches", [(128, 4), (150, 8), (200, 3), (256, 8)])
def test_cascade_batch_matches_oracle_and_plain_attention(models, prefix, branches):
    """Prefix on a page boundary (128, 256: every prefix page shared) and off
    it (150, 200: the partly filled page is copied per branch); branches
    continue from their own tokens; three teacher-forced batched steps."""
    import torch
    cfg, on, s_on, off, s_off, orc = models
    prompt = synth.prompt_tokens(cfg, prefix, seed=prefix)
    oseq = orc.new_seq(capacity=prefix + 8)
    orc.prefill(oseq, prompt)
    obr = [oseq.fork() for _ in range(branches)]
    runs = []
    for m, stream in ((on, s_on), (off, s_off)):
        src = m.seq_create()
        m.prefill(src, prompt)
        dst = [m.seq_create() for _ in range(branches)]
        m.kv_fork(src, dst, shared=True)
        runs.append((m, stream, src, dst))
    toks = [int(t) for t in synth.prompt_tokens(cfg, branches, seed=7)]
    try:
        for i in range(3):
            outs = []
            for m, stream, src, dst in runs:
                out = torch.empty(branches, cfg.vocab, device="cuda")
                m.decode_batch(dst, toks, [prefix + i] * branches, out)
                stream.synchronize()
                outs.append(out.cpu().numpy())
            assert on.launches_per_step() == off.launches_per_step() + cfg.n_layers   # the cascade kernel ran
            for b in range(branches):
                ref = orc.decode_step(obr[b], toks[b], prefix + i)
                assert_close(outs[0][b], ref, f"cascade prefix {prefix} branch {b} step {i}")
                assert_close(outs[0][b], outs[1][b], f"cascade vs plain, branch {b} step {i}", tol=1e-4)
                toks[b] = check_greedy(outs[0][b], ref, f"branch {b} step {i}")
    finally:
        for m, stream, src, dst in runs:
            for q in [src] + dst:
                m.seq_free(q)


def test_cascade_generate_and_mixed_batches(models):
    """Greedy generation on the device (graph replay) over a shared prefix
    agrees with the plain attention path; a batch whose rows share nothing
    runs without the cascade kernel."""
    import torch
    cfg, on, s_on, off, s_off, orc = models
    prefix, B, D = 160, 6, 12
    prompt = synth.prompt_tokens(cfg, prefix, seed=3)
    res = []
    for m, stream in ((on, s_on), (off, s_off)):
        src = m.seq_create()
        m.prefill(src, prompt)
        dst = [m.seq_create() for _ in range(B)]
        m.kv_fork(src, dst, shared=True)
        last = torch.empty(B, cfg.vocab, device="cuda")
        toks = m.generate(dst, list(range(20, 20 + B)), D, last)
        stream.synchronize()
        res.append((toks, last.cpu().numpy()))
        for q in [src] + dst:
            m.seq_free(q)
    assert np.array_equal(res[0][0], res[1][0])
    assert_close(res[0][1], res[1][1], "generate: cascade vs plain", tol=1e-4)
    # independent sequences: no shared pages, no cascade kernel
    seqs = []
    for r in range(3):
        s = on.seq_create()
        on.prefill(s, synth.prompt_tokens(cfg, 140 + r, seed=30 + r))
        seqs.append(s)
    on.decode_batch(seqs, [1, 2, 3], [140, 141, 142])
    s_on.synchronize()
    base = on.launches_per_step()
    a, b = on.seq_create(), on.seq_create()
    on.kv_fork(seqs[0], [a, b], shared=True)
    on.decode_batch([a, b], [4, 5], [141, 141])
    s_on.synchronize()
    assert on.launches_per_step() == base + cfg.n_layers
    for q in seqs + [a, b]:
        on.seq_free(q)


def test_cascade_partials_merge_like_the_oracle():
    """The split-softmax algebra the cascade relies on, at the shapes of the
    tiny model: prefix and suffix partials merge to full attention (CPU)."""
    rng = np.random.default_rng(9)
    q = rng.standard_normal((4, 64))
    K = ops.round_f16(rng.standard_normal((300, 2, 64)))
    V = ops.round_f16(rng.standard_normal((300, 2, 64)))
    full = ops.attention(q, K, V)
    parts = [ops.attention_partial(q, K[:256], V[:256]), ops.attention_partial(q, K[256:], V[256:])]
    np.testing.assert_allclose(ops.merge_partials(parts), full, rtol=1e-12, atol=1e-12)
