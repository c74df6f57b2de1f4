"""The C-ABI library on a machine without a GPU: it builds, loads, exports
every entry point the header declares, and rejects bad input on the host
before touching a device."""
import ctypes
import os
import re
import subprocess

import pytest

from decode_llama_step_gb300 import _build, dls

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    text = open(os.path.join(ROOT, "include", "dls.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dls_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return dls.load()


def test_library_exports_every_declared_function(lib):
    names = header_functions()
    assert len(names) >= 25
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (dls_\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    # the binding wraps exactly the declared set
    assert sorted(dls.exported_symbols()) == names


def test_abi_version_and_status_names(lib):
    assert lib.dls_abi_version() == 2
    assert dls.status_name(0) == "OK"
    assert dls.status_name(-2) == "BUDGET"
    assert dls.status_name(-6) == "STATE"


def test_step_kernel_query_without_a_model(lib):
    # no model: not in use, and no reason string is invented
    why = ctypes.c_char_p(b"unset")
    assert lib.dls_step_kernel_in_use(None, ctypes.byref(why)) == 0
    assert why.value is None
    assert lib.dls_step_kernel_in_use(None, None) == 0


def _golden_budget_cases():
    rows = []
    for line in open(os.path.join(ROOT, "tests", "golden", "context_budget.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            a, b, c, d, e = line.split()
            rows.append((int(a), int(b), int(c), int(d), e))
    return rows


@pytest.mark.parametrize("prefix,branch,headroom,n_ctx,expected", _golden_budget_cases())
def test_context_budget_fail_fast(lib, prefix, branch, headroom, n_ctx, expected):
    rc = lib.dls_check_context_budget(prefix, branch, headroom, n_ctx)
    assert dls.status_name(rc) == expected
    if expected != "OK":
        msg = lib.dls_last_error(None).decode()
        assert msg.startswith("ERR CAPACITY") and f"required={prefix + branch + headroom}" in msg


def _desc(**over):
    d = dls.dls_model_desc()
    d.n_layers, d.hidden, d.n_heads, d.n_kv_heads, d.head_dim, d.ffn, d.vocab = 2, 256, 4, 2, 64, 688, 1024
    d.rope_theta, d.rms_eps, d.wtype, d.max_seqs, d.max_ctx = 10000.0, 1e-5, 8, 1, 64
    for k, v in over.items():
        setattr(d, k, v)
    return d


@pytest.mark.parametrize("over,frag", [
    ({"n_layers": 0}, "shape"),
    ({"hidden": 250}, "hidden=250"),
    ({"n_heads": 5}, "n_heads=5"),
    ({"head_dim": 96}, "head_dim=96"),
    ({"wtype": 5}, "wtype=5"),
    ({"page_tokens": 48}, "page_tokens=48"),
    ({"max_ctx": 0}, "max_ctx=0"),
    ({"max_batch": 9}, "max_batch=9"),
    ({}, "missing tensor pointer"),
])
def test_create_rejects_bad_descriptor_before_any_cuda_call(lib, over, frag):
    d = _desc(**over)
    h = ctypes.c_void_p()
    rc = lib.dls_model_create(ctypes.byref(d), None, None, ctypes.byref(h))
    assert rc == dls.DLS_ERR_ARG
    assert h.value is None
    msg = lib.dls_last_error(None).decode()
    assert msg.startswith("ERR ARG") and frag in msg


def test_null_model_calls_fail_cleanly(lib):
    assert lib.dls_decode_step(None, 0, 1, 0, None) == dls.DLS_ERR_ARG
    assert lib.dls_kv_fork(None, 0, None, 1) == dls.DLS_ERR_ARG
    assert lib.dls_set_resident_layers(None, 1) == dls.DLS_ERR_ARG
    assert lib.dls_seq_length(None, 0) == dls.DLS_ERR_ARG
    assert lib.dls_resident_layers(None) == -1


def test_attention_op_rejects_bad_shapes(lib):
    assert lib.dls_attention_workspace_bytes(1, 5, 2, 64, 4) == 0
    rc = lib.dls_attention_decode(1, 1, 1, 1, 1, 1, 1, 1 << 20, 1, 4, 2, 96, 64, 4, 1, None, None)
    assert rc == dls.DLS_ERR_ARG
    rc = lib.dls_attention_decode(None, 1, 1, 1, 1, 1, 1, 1 << 20, 1, 4, 2, 64, 64, 4, 1, None, None)
    assert rc == dls.DLS_ERR_ARG
    rc = lib.dls_attention_decode(1, 1, 1, 1, 1, 1, 1, 1 << 20, 1, 4, 2, 64, 64, 4, 129, None, None)
    assert rc == dls.DLS_ERR_ARG
    assert "attention" in lib.dls_last_error(None).decode()
    rc = lib.dls_attention_decode_noalloc(1, 1, 1, 1, 1, 1, 1, 4, 2, 64, 16, 4, 1, None, None)
    assert rc == dls.DLS_ERR_ARG       # page_tokens below 32
    assert lib.dls_attention_status(None, None) == dls.DLS_ERR_ARG


def test_null_model_calls_of_the_later_entry_points(lib):
    assert lib.dls_seq_truncate(None, 0, 0) == dls.DLS_ERR_ARG
    assert lib.dls_verify(None, 0, None, 1, None, None) == dls.DLS_ERR_ARG
    assert lib.dls_generate_speculative(None, 0, 1, 4, None, 3, None, None) == dls.DLS_ERR_ARG
    assert lib.dls_set_layer_skip(None, None, 0) == dls.DLS_ERR_ARG
    assert lib.dls_layer_cosines(None, 0, 1, 0, None) == dls.DLS_ERR_ARG


def test_kquant_layout_sizes_and_argument_checks(lib):
    # Q4_K: the GGUF super-blocks as they are (144 bytes per 256 weights)
    assert lib.dls_kquant_packed_bytes(dls.DLS_Q4_K, 3, 512) == 3 * 2 * 144
    assert lib.dls_kquant_packed_bytes(dls.DLS_Q5_K, 3, 512) == 3 * 2 * 176
    # Q6_K: 208 bytes per super-block, 256-byte aligned, then fp16 scales
    # with each row padded to 8 super-blocks
    rows, nsb = 5, 17
    main = (rows * nsb * 208 + 255) // 256 * 256
    assert lib.dls_kquant_packed_bytes(dls.DLS_Q6_K, rows, nsb * 256) == main + rows * 24 * 2
    for bad in [(dls.DLS_Q4_K, 3, 300), (dls.DLS_Q4_K, 0, 256), (15, 4, 256), (dls.DLS_Q6_K, 4, 0)]:
        assert lib.dls_kquant_packed_bytes(*bad) == 0
    # rejected before any CUDA call
    assert lib.dls_kquant_gemv(15, 256, 4, 256, 256, 256, None, None) == dls.DLS_ERR_ARG
    assert lib.dls_kquant_gemv(dls.DLS_Q4_K, None, 4, 256, 256, 256, None, None) == dls.DLS_ERR_ARG
    assert lib.dls_kquant_gemv(dls.DLS_Q4_K, 256, 4, 300, 256, 256, None, None) == dls.DLS_ERR_ARG
    assert lib.dls_kquant_gemv(dls.DLS_Q4_K, 256 + 16, 4, 256, 256, 256, None, None) == dls.DLS_ERR_ARG
    assert lib.dls_kquant_pack(dls.DLS_Q6_K, None, 4, 256, 256, None) == dls.DLS_ERR_ARG
    assert "kquant" in lib.dls_last_error(None).decode()
