"""GPU parity of the K-quant dequant-GEMV (Q4_K, Q5_K, Q6_K) against the oracle,
through the C ABI: the device layout byte for byte, y = W x on small and
ragged shapes in full, and on the 70B projection shapes on sampled rows."""
import numpy as np
import pytest

import synth
from oracle import kquant as kq

pytestmark = pytest.mark.gpu


def _torch():
    import torch
    return torch


def _setup(fmt, rows, cols, seed=0):
    torch = _torch()
    from decode_llama_step_gb300 import dls
    blocks = synth.kquant_matrix(synth.stream_key("kq-gpu", fmt, rows, cols, seed), rows, cols, fmt)
    x = synth.normal(synth.stream_key("kq-gpu-x", cols, seed), cols, 1.0).astype(np.float32)
    x[:: 97] *= 30.0                                  # a few large activations
    stream = torch.cuda.Stream()
    dev_blocks = torch.from_numpy(blocks).cuda()
    packed = torch.zeros(dls.kquant_packed_bytes(fmt, rows, cols), dtype=torch.uint8, device="cuda")
    dls.kquant_pack(fmt, dev_blocks, rows, cols, packed, stream=stream)
    xd = torch.from_numpy(x).cuda()
    y = torch.full((rows,), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dls.kquant_gemv(fmt, packed, rows, cols, xd, y, status=status, stream=stream)
    stream.synchronize()
    assert int(status.item()) == 0
    return blocks, x, packed.cpu().numpy(), y.cpu().numpy().astype(np.float64)


def _bound(w, x):
    """Worst case of the int16 activation slices (at most half a step of
    max|x| / 32767 per element) plus fp32 accumulation."""
    step = float(np.max(np.abs(x))) / 32767.0
    return 0.5 * step * np.abs(w).sum(axis=-1) * 1.001 + 2e-6 * np.abs(w * x).sum(axis=-1) + 1e-6


@pytest.mark.parametrize("fmt", ["q4_k", "q5_k", "q6_k"])
@pytest.mark.parametrize("rows,cols", [(1, 256), (37, 512), (300, 2048), (129, 4352), (1000, 8192),
                                       (5, 28672)])
def test_kquant_gemv_matches_oracle(fmt, rows, cols):
    blocks, x, packed, y = _setup(fmt, rows, cols)
    w = kq.matrix_rows(blocks, cols, fmt, 0, rows)
    ref = w @ x.astype(np.float64)
    err = np.abs(y - ref)
    assert np.all(err <= _bound(w, x.astype(np.float64))), f"max err {err.max():.3e}"


@pytest.mark.parametrize("fmt", ["q4_k", "q5_k", "q6_k"])
def test_kquant_packed_layout_bytes(fmt):
    rows, cols = 9, 4352                             # 17 super-blocks: the Q6_K scale rows are padded
    blocks, _, packed, _ = _setup(fmt, rows, cols)
    nsb = cols // 256
    raw = blocks.reshape(rows * nsb, kq.BLOCK_BYTES[fmt])
    if fmt in ("q4_k", "q5_k"):
        assert np.array_equal(packed, blocks)
        return
    main = packed[: rows * nsb * 208].reshape(rows * nsb, 208)
    assert np.array_equal(main, raw[:, :208])
    off = (rows * nsb * 208 + 255) // 256 * 256
    pad = (nsb + 7) // 8 * 8
    d = packed[off: off + rows * pad * 2].reshape(rows, pad, 2)
    assert np.array_equal(d[:, :nsb, :].reshape(rows * nsb, 2), raw[:, 208:210])
    assert not d[:, nsb:, :].any()


@pytest.mark.parametrize("fmt", ["q4_k", "q5_k", "q6_k"])
@pytest.mark.parametrize("rows,cols", [(8192, 8192), (28672, 8192), (8192, 28672)])
def test_kquant_gemv_70b_shapes_sampled_rows(fmt, rows, cols):
    blocks, x, _, y = _setup(fmt, rows, cols, seed=1)
    rng = np.random.default_rng(rows + cols)
    sample = np.unique(np.concatenate([[0, rows - 1], rng.integers(0, rows, 48)]))
    for r in sample:
        w = kq.matrix_rows(blocks, cols, fmt, int(r), int(r) + 1)[0]
        ref = float(w @ x.astype(np.float64))
        assert abs(y[r] - ref) <= _bound(w, x.astype(np.float64)), f"row {r}: {y[r]} vs {ref}"


def test_kquant_rejects_bad_arguments():
    torch = _torch()
    from decode_llama_step_gb300 import dls
    buf = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    x = torch.zeros(300, device="cuda")
    y = torch.zeros(4, device="cuda")
    assert dls.kquant_packed_bytes("q4_k", 4, 300) == 0
    with pytest.raises(dls.DlsError):
        dls.kquant_gemv("q4_k", buf, 4, 300, x, y)          # cols not a multiple of 256
    with pytest.raises(dls.DlsError):
        dls.kquant_gemv("q6_k", buf, 4, 256 * 129, x, y)    # wider than the kernel takes
    with pytest.raises(dls.DlsError):
        dls.kquant_gemv("q4_k", buf[1:], 1, 256, x, y)       # misaligned matrix
