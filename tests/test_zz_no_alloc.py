"""The allocation-free attention entry point, for callers that may not
allocate device memory (a fixed device-memory plan, or a path where an
allocator call could block or synchronise).  It must give the same result as
the workspace-taking entry point, call after call, with its scratch kept
inside the library.  This file sorts last so a run that stops at the first
failure has run every other test before it."""
import numpy as np
import pytest

from parity import assert_close

pytestmark = pytest.mark.gpu


def _case(torch, rng, nb, nh, nkv, hd, pt, maxp):
    lengths = rng.integers(1, pt * maxp + 1, size=nb).astype(np.int32)
    lengths[0] = pt * maxp            # a full row
    npages = nb * maxp
    kp = torch.from_numpy(rng.standard_normal((npages, nkv, pt, hd)).astype(np.float16)).cuda()
    vp = torch.from_numpy(rng.standard_normal((npages, nkv, pt, hd)).astype(np.float16)).cuda()
    table = torch.from_numpy(rng.permutation(npages).astype(np.int32).reshape(nb, maxp)).cuda()
    q = torch.from_numpy(rng.standard_normal((nb, nh, hd)).astype(np.float32)).cuda()
    return q, kp, vp, table, torch.from_numpy(lengths).cuda()


@pytest.mark.parametrize("nb,nh,nkv,hd,pt,maxp,splits", [
    (1, 32, 8, 128, 64, 36, 19),   # the 8B decode shape at ~2300 positions
    (3, 4, 2, 64, 32, 5, 0),       # tiny shape, the call picks the split count
    (2, 64, 8, 128, 64, 8, 7),     # 70B grouping (8 query heads per KV head)
    (8, 32, 8, 128, 64, 64, 0),    # 8 branches at ctx 4096: the usual split count needs more than the array
])
def test_noalloc_matches_workspace_entry_point_twice(gpu_lib, nb, nh, nkv, hd, pt, maxp, splits):
    import torch
    from decode_llama_step_gb300 import dls
    rng = np.random.default_rng(11)
    q, kp, vp, table, lens = _case(torch, rng, nb, nh, nkv, hd, pt, maxp)
    # the reference call gets room for any split count it may choose (128 at
    # most); split counts change the result only by fp32 rounding
    wsb = dls.attention_workspace_bytes(nb, nh, nkv, hd, splits or 128)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    ref = torch.empty(nb, nh, hd, device="cuda")
    dls.attention_decode(q, kp, vp, table, lens, ref, ws, wsb, nb, nh, nkv, hd, pt, maxp, splits)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call in range(2):   # the shared scratch keeps the last call's contents
        out = torch.full((nb, nh, hd), float("nan"), device="cuda")
        dls.attention_decode_noalloc(q, kp, vp, table, lens, out, nb, nh, nkv, hd, pt, maxp, splits, status=status)
        dls.attention_status(status)
        assert_close(out.cpu().numpy(), ref.cpu().numpy(), f"noalloc call {call}", tol=1e-5)


def test_noalloc_rejects_shapes_beyond_its_scratch(gpu_lib):
    import torch
    from decode_llama_step_gb300 import dls
    nb, nh, nkv, hd, pt, maxp, ns = 8, 64, 8, 128, 64, 4, 128
    assert dls.attention_workspace_bytes(nb, nh, nkv, hd, ns) > dls.NOALLOC_SCRATCH_BYTES
    rng = np.random.default_rng(12)
    q, kp, vp, table, lens = _case(torch, rng, nb, nh, nkv, hd, pt, maxp)
    out = torch.empty(nb, nh, hd, device="cuda")
    with pytest.raises(dls.DlsError) as e:
        dls.attention_decode_noalloc(q, kp, vp, table, lens, out, nb, nh, nkv, hd, pt, maxp, ns)
    assert e.value.code == dls.DLS_ERR_CAPACITY
    assert "scratch" in str(e.value)
