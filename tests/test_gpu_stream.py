"""Host-to-device paths of layer streaming: the SM-driven copy kernel
(dls_h2d_copy_sm) copies pinned host memory bit for bit and refuses any
other pointer kind before launching; a model whose streamed layers arrive
through it decodes exactly like one using the copy engines (the engine
page, sections 3.3 and 4.2: double-buffered layer streaming from pinned host
memory)."""
import os

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


def test_sm_copy_is_bit_exact_and_checks_pointers(gpu_lib):
    import torch
    from decode_llama_step_gb300 import dls
    rng = np.random.default_rng(0)
    for nbytes, ctas in [(16, 1), (4096, 3), (3 << 20, 64), ((40 << 20) + 48, 152)]:
        src = torch.from_numpy(rng.integers(0, 256, nbytes, dtype=np.uint8)).pin_memory()
        dst = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
        dls.h2d_copy_sm(dst, src, nbytes, ctas)
        torch.cuda.synchronize()
        assert torch.equal(dst.cpu(), src), (nbytes, ctas)
    pageable = np.zeros(4096, dtype=np.uint8)
    dev = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    pinned = torch.zeros(4096, dtype=torch.uint8).pin_memory()
    for args in [(dev, pageable, 4096, 8), (dev, dev, 4096, 8), (pinned, pinned, 4096, 8), (dev, pinned, 4008, 8),
                 (dev, pinned, 4096, 0)]:
        with pytest.raises(dls.DlsError) as e:
            dls.h2d_copy_sm(*args)
        assert e.value.code == dls.DLS_ERR_ARG


def test_sm_copy_streamer_matches_copy_engines(gpu_lib, monkeypatch):
    import torch
    from decode_llama_step_gb300 import dls
    cfg = synth.get_config("tiny")
    w = synth.model_weights(cfg)
    prompt = synth.prompt_tokens(cfg, 24, seed=12)
    outs = []
    for mode in (None, "sm:4"):
        if mode:
            monkeypatch.setenv("DLS_STREAM_COPY", mode)
        stream = torch.cuda.Stream()
        m = dls.Model(cfg, w, max_seqs=1, max_ctx=64, stream=stream)
        monkeypatch.delenv("DLS_STREAM_COPY", raising=False)
        try:
            m.set_resident_layers(0)          # both layers stream every step
            s = m.seq_create()
            m.prefill(s, prompt)
            last = torch.empty(1, cfg.vocab, device="cuda")
            toks = m.generate([s], [3], 6, last)
            stream.synchronize()
            outs.append((toks.copy(), last.cpu()))
        finally:
            m.close()
    assert np.array_equal(outs[0][0], outs[1][0])
    assert torch.equal(outs[0][1], outs[1][1])
