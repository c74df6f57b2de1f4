"""Failure paths of the C ABI on a GPU, every failure made on the host (an
allocator callback that returns NULL, a budget or KV pool too small, a
bounded device wait on a barrier nothing arrives at): no GPU fault is
involved.  The LayerStreamer page's admission ledger is the model: reserve,
commit on success, roll back on failure, so a failed call leaves no trace.
Each case checks the error code, that nothing leaked (the allocator's live
set, the ledger's byte count, the free KV pages) and that the model still
decodes exactly as before the failure.
"""
import numpy as np
import pytest

import synth
from oracle import OracleModel
from synth.configs import ModelConfig

from parity import assert_close

pytestmark = pytest.mark.gpu

# four layers, so that a budget can hold some layers plus the two staging
# buffers of the streamed ones
TINY4 = ModelConfig("tiny4", 4, 256, 4, 2, 64, 688, 1024, 10000.0, 8, 0.02)


@pytest.fixture(scope="module")
def env(gpu_lib):
    import torch
    from decode_llama_step_gb300 import dls
    w = synth.model_weights(TINY4)
    return torch, dls, w, OracleModel(TINY4, w)


def _decode(torch, m, cfg, prompt, tok):
    """Prefill `prompt` on a fresh sequence, decode `tok`; the step's logits."""
    s = m.seq_create()
    try:
        lg = torch.empty(cfg.vocab, device="cuda")
        m.prefill(s, prompt)
        m.decode_step(s, tok, len(prompt), lg)
        m.stream.synchronize()
        return lg.cpu().numpy().astype(np.float64)
    finally:
        m.seq_free(s)


def _oracle_decode(orc, prompt, tok):
    s = orc.new_seq()
    orc.prefill(s, prompt)
    return orc.decode_step(s, tok, len(prompt))


def test_create_rolls_back_when_any_allocation_fails(env):
    torch, dls, w, orc = env
    dev = torch.cuda.current_device()
    stream = torch.cuda.Stream()
    probe = dls.TorchAllocator(dev)
    m = dls.Model(TINY4, w, max_seqs=2, max_ctx=96, stream=stream, allocator=probe)
    n = probe.calls
    m.close()
    assert n >= 10 and not probe.live
    for k in sorted({1, 2, 3, n // 3, n // 2, n - 1, n}):
        a = dls.TorchAllocator(dev, fail_at=k)
        with pytest.raises(dls.DlsError) as e:
            dls.Model(TINY4, w, max_seqs=2, max_ctx=96, stream=stream, allocator=a)
        assert e.value.code == dls.DLS_ERR_CUDA, k
        assert "allocation failed" in str(e.value), str(e.value)
        assert a.calls == k and not a.live, f"allocation {k} of {n} failed: {len(a.live)} buffers leaked"


def test_residency_change_rolls_back_when_an_allocation_fails(env):
    torch, dls, w, orc = env
    dev = torch.cuda.current_device()
    stream = torch.cuda.Stream()
    prompt = synth.prompt_tokens(TINY4, 12, seed=7)
    ref = _oracle_decode(orc, prompt, 9)
    alloc = dls.TorchAllocator(dev)
    m = dls.Model(TINY4, w, max_seqs=2, max_ctx=96, stream=stream, allocator=alloc)
    try:
        base = _decode(torch, m, TINY4, prompt, 9)
        assert_close(base, ref, "resident model")
        # resident -> 1 layer needs the two staging buffers: fail the first
        # and the second of them
        for k in (1, 2):
            before = (m.resident_layers(), m.device_bytes(), dict(alloc.live))
            alloc.fail_at = k
            with pytest.raises(dls.DlsError) as e:
                m.set_resident_layers(1)
            assert e.value.code == dls.DLS_ERR_CUDA
            alloc.fail_at = None
            assert (m.resident_layers(), m.device_bytes(), dict(alloc.live)) == before
            assert np.array_equal(_decode(torch, m, TINY4, prompt, 9), base)
        m.set_resident_layers(1)
        streamed = _decode(torch, m, TINY4, prompt, 9)
        assert_close(streamed, ref, "one resident layer")
        # 1 -> 4 resident layers loads three layers (and the persistent
        # kernel's scratch, made once): fail each of the loads
        for k in (1, 2, 3):
            before = (m.resident_layers(), m.device_bytes(), dict(alloc.live))
            alloc.fail_at = k
            with pytest.raises(dls.DlsError) as e:
                m.set_resident_layers(4)
            assert e.value.code == dls.DLS_ERR_CUDA
            alloc.fail_at = None
            assert (m.resident_layers(), m.device_bytes(), dict(alloc.live)) == before
            assert np.array_equal(_decode(torch, m, TINY4, prompt, 9), streamed)
        m.set_resident_layers(4)
        assert m.resident_layers() == 4
        assert_close(_decode(torch, m, TINY4, prompt, 9), ref, "resident again")
    finally:
        m.close()
    assert not alloc.live


def test_residency_over_budget_fails_and_changes_nothing(env):
    torch, dls, w, orc = env
    stream = torch.cuda.Stream()
    prompt = synth.prompt_tokens(TINY4, 12, seed=8)
    ref = _oracle_decode(orc, prompt, 3)
    full = dls.Model(TINY4, w, max_seqs=2, max_ctx=96, stream=stream)
    resident_bytes = full.device_bytes()      # every layer resident, nothing staged
    lb = full.layer_bytes()
    full.close()
    # half a layer of headroom: all four layers fit, but three resident
    # layers plus the two staging buffers of the streamed one (five layers'
    # worth) do not; two resident plus staging (four) do
    m = dls.Model(TINY4, w, max_seqs=2, max_ctx=96, stream=stream, device_budget_bytes=resident_bytes + lb // 2)
    try:
        assert m.resident_layers() == 4
        base = _decode(torch, m, TINY4, prompt, 3)
        assert_close(base, ref, "resident under the budget")
        for start in (4, 2):
            if start == 2:
                m.set_resident_layers(2)
                base = _decode(torch, m, TINY4, prompt, 3)
                assert_close(base, ref, "two resident layers")
            used = m.device_bytes()
            with pytest.raises(dls.DlsError) as e:
                m.set_resident_layers(3)
            assert e.value.code == dls.DLS_ERR_BUDGET
            assert "budget" in str(e.value)
            assert m.resident_layers() == start and m.device_bytes() == used
            assert np.array_equal(_decode(torch, m, TINY4, prompt, 3), base)
        m.set_resident_layers(4)
        assert_close(_decode(torch, m, TINY4, prompt, 3), ref, "resident again")
    finally:
        m.close()


def test_kv_pool_exhaustion_fails_and_changes_nothing(env):
    torch, dls, w, orc = env
    stream = torch.cuda.Stream()
    # 4 sequences of up to 128 tokens (4 pages of 32) share a pool of 6 pages
    m = dls.Model(TINY4, w, max_seqs=4, max_ctx=128, page_tokens=32, stream=stream, kv_pool_pages=6)
    try:
        src = m.seq_create()
        dst = [m.seq_create() for _ in range(3)]
        prompt = synth.prompt_tokens(TINY4, 64, seed=9)
        m.prefill(src, prompt)                      # 2 pages
        assert m.kv_free_pages() == 4
        with pytest.raises(dls.DlsError) as e:      # 3 copies of 2 pages > 4 free
            m.kv_fork(src, dst)
        assert e.value.code == dls.DLS_ERR_CAPACITY
        assert m.kv_free_pages() == 4 and [m.seq_length(s) for s in dst] == [0, 0, 0]
        m.kv_fork(src, dst[:2])                     # 4 pages: fits exactly
        assert m.kv_free_pages() == 0
        with pytest.raises(dls.DlsError) as e:      # no page left for a prompt
            m.prefill(dst[2], synth.prompt_tokens(TINY4, 10, seed=10))
        assert e.value.code == dls.DLS_ERR_CAPACITY
        assert m.kv_free_pages() == 0 and m.seq_length(dst[2]) == 0
        with pytest.raises(dls.DlsError) as e:      # position 64 needs a third page
            m.decode_step(dst[0], 5, 64)
        assert e.value.code == dls.DLS_ERR_CAPACITY
        assert m.seq_length(dst[0]) == 64
        # once a branch returns its pages the other decodes like the
        # oracle's fork
        m.seq_free(dst[1])
        assert m.kv_free_pages() == 2
        lg = torch.empty(TINY4.vocab, device="cuda")
        m.decode_step(dst[0], 5, 64, lg)
        stream.synchronize()
        s = orc.new_seq()
        orc.prefill(s, prompt)
        assert_close(lg.cpu().numpy(), orc.decode_step(s.fork(), 5, 64), "forked branch after the failures")
    finally:
        m.close()


def test_bounded_device_wait_reports_timeout_and_model_stays_usable(env):
    torch, dls, w, orc = env
    stream = torch.cuda.Stream()
    prompt = synth.prompt_tokens(TINY4, 12, seed=11)
    ref = _oracle_decode(orc, prompt, 4)
    m = dls.Model(TINY4, w, max_seqs=2, max_ctx=96, stream=stream)
    try:
        base = _decode(torch, m, TINY4, prompt, 4)
        for limit_ns in (2_000, 50_000_000):
            with pytest.raises(dls.DlsError) as e:
                m.debug_bounded_wait(limit_ns)
            assert e.value.code == dls.DLS_ERR_TIMEOUT
            assert "bounded device wait" in str(e.value)
            # the status word was cleared: the next calls succeed and agree
            assert np.array_equal(_decode(torch, m, TINY4, prompt, 4), base)
        with pytest.raises(dls.DlsError) as e:
            m.debug_bounded_wait(10)
        assert e.value.code == dls.DLS_ERR_ARG
        assert_close(base, ref, "after the timeouts")
    finally:
        m.close()
