"""ctypes binding of ``include/dls.h`` (argument marshalling only).

Every step of the decode path runs in the CUDA library; this module only
passes pointers and sizes.  If the library is missing or fails to load it
raises: there is no fallback.  PyTorch supplies device memory (through the
allocator callbacks) and streams.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from . import _build

_lock = threading.Lock()
_lib = None

DLS_OK, DLS_ERR_ARG, DLS_ERR_BUDGET, DLS_ERR_CAPACITY, DLS_ERR_CUDA, DLS_ERR_TIMEOUT, DLS_ERR_STATE = 0, -1, -2, -3, -4, -5, -6
DLS_Q4_0, DLS_Q8_0 = 4, 8
TENSOR_IDS = {"wq": 0, "wk": 1, "wv": 2, "wo": 3, "w_gate": 4, "w_up": 5, "w_down": 6, "tok_embd": 7, "output": 8}

i32, u64, vp, sz = ctypes.c_int32, ctypes.c_uint64, ctypes.c_void_p, ctypes.c_size_t


class DlsError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(msg)
        self.code = code


class dls_allocator(ctypes.Structure):
    _fields_ = [("alloc", ctypes.CFUNCTYPE(vp, vp, sz, vp)),
                ("free", ctypes.CFUNCTYPE(None, vp, vp, vp)),
                ("ctx", vp)]


class dls_layer_desc(ctypes.Structure):
    _fields_ = [(n, vp) for n in ("attn_norm", "ffn_norm", "wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")] + \
               [("types", i32 * 7)]


class dls_model_desc(ctypes.Structure):
    _fields_ = [("n_layers", i32), ("hidden", i32), ("n_heads", i32), ("n_kv_heads", i32), ("head_dim", i32),
                ("ffn", i32), ("vocab", i32), ("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float),
                ("tied_embeddings", i32), ("wtype", i32), ("page_tokens", i32), ("max_seqs", i32),
                ("max_ctx", i32), ("max_batch", i32), ("device_budget_bytes", u64), ("tok_embd", vp),
                ("output", vp), ("output_norm", vp), ("layers", ctypes.POINTER(dls_layer_desc)),
                ("kv_pool_pages", i32), ("tok_embd_type", i32), ("output_type", i32)]


_SIGS = {
    "dls_abi_version": (ctypes.c_int, []),
    "dls_status_name": (ctypes.c_char_p, [ctypes.c_int]),
    "dls_last_error": (ctypes.c_char_p, [vp]),
    "dls_model_create": (ctypes.c_int, [ctypes.POINTER(dls_model_desc), ctypes.POINTER(dls_allocator), vp,
                                        ctypes.POINTER(vp)]),
    "dls_model_destroy": (None, [vp]),
    "dls_device_bytes": (u64, [vp]),
    "dls_device_budget": (u64, [vp]),
    "dls_seq_create": (ctypes.c_int, [vp, ctypes.POINTER(i32)]),
    "dls_seq_free": (ctypes.c_int, [vp, i32]),
    "dls_seq_length": (i32, [vp, i32]),
    "dls_prefill": (ctypes.c_int, [vp, i32, vp, i32, vp]),
    "dls_decode_step": (ctypes.c_int, [vp, i32, i32, i32, vp]),
    "dls_decode_batch": (ctypes.c_int, [vp, i32, vp, vp, vp, vp]),
    "dls_generate": (ctypes.c_int, [vp, i32, vp, vp, i32, vp, vp]),
    "dls_argmax": (ctypes.c_int, [vp, vp, i32, vp]),
    "dls_kv_fork": (ctypes.c_int, [vp, i32, vp, i32]),
    "dls_kv_fork_shared": (ctypes.c_int, [vp, i32, vp, i32]),
    "dls_kv_free_pages": (i32, [vp]),
    "dls_set_layer_skip": (ctypes.c_int, [vp, vp, i32]),
    "dls_layer_cosines": (ctypes.c_int, [vp, i32, i32, i32, vp]),
    "dls_seq_truncate": (ctypes.c_int, [vp, i32, i32]),
    "dls_verify": (ctypes.c_int, [vp, i32, vp, i32, vp, vp]),
    "dls_generate_speculative": (ctypes.c_int, [vp, i32, i32, i32, vp, i32, vp, vp]),
    "dls_check_context_budget": (ctypes.c_int, [i32, i32, i32, i32]),
    "dls_h2d_copy_sm": (ctypes.c_int, [vp, vp, sz, i32, vp]),
    "dls_set_resident_layers": (ctypes.c_int, [vp, i32]),
    "dls_resident_layers": (i32, [vp]),
    "dls_layer_bytes": (u64, [vp]),
    "dls_attention_decode": (ctypes.c_int, [vp, vp, vp, vp, vp, vp, vp, sz, i32, i32, i32, i32, i32, i32, i32, vp, vp]),
    "dls_attention_status": (ctypes.c_int, [vp, vp]),
    "dls_attention_workspace_bytes": (sz, [i32, i32, i32, i32, i32]),
    "dls_attention_decode_noalloc": (ctypes.c_int, [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, vp]),
    "dls_kquant_packed_bytes": (ctypes.c_uint64, [i32, i32, i32]),
    "dls_kquant_pack": (ctypes.c_int, [i32, vp, i32, i32, vp, vp]),
    "dls_kquant_gemv": (ctypes.c_int, [i32, vp, i32, i32, vp, vp, vp, vp]),
    "dls_debug_capture": (ctypes.c_int, [vp, vp]),
    "dls_debug_read_kv": (ctypes.c_int, [vp, i32, i32, vp, vp]),
    "dls_debug_bounded_wait": (ctypes.c_int, [vp, ctypes.c_int64]),
    "dls_debug_dequant": (ctypes.c_int, [vp, i32, i32, vp]),
    "dls_debug_gemv": (ctypes.c_int, [vp, i32, i32, vp, vp]),
    "dls_debug_gemm": (ctypes.c_int, [vp, i32, i32, i32, vp, vp]),
    "dls_debug_launches_per_step": (i32, [vp]),
    "dls_debug_profile_step": (ctypes.c_int, [vp, i32, i32, i32, i32, vp, vp, vp]),
    "dls_debug_step_trace": (ctypes.c_int, [vp, vp, i32, vp]),
    "dls_step_kernel_in_use": (i32, [vp, vp]),
    "dls_debug_profile_batch": (ctypes.c_int, [vp, i32, vp, vp, vp, i32, vp, vp, vp]),
}


def exported_symbols():
    """Names the header declares (the binding's contract)."""
    return sorted(_SIGS)


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load the CUDA library (building it first if needed)."""
    global _lib
    with _lock:
        if _lib is None:
            if build_if_missing and not _build.up_to_date():
                _build.build()
            if not os.path.exists(_build.LIB):
                raise RuntimeError(f"decode-step CUDA library missing: {_build.LIB}")
            lib = ctypes.CDLL(_build.LIB)
            for name, (res, args) in _SIGS.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _ptr(obj):
    """Device or host pointer of a torch tensor / numpy array / int / None."""
    if obj is None:
        return None
    if isinstance(obj, int):
        return obj
    if isinstance(obj, np.ndarray):
        if not obj.flags["C_CONTIGUOUS"]:
            raise ValueError("array must be C-contiguous")
        return obj.ctypes.data
    if hasattr(obj, "data_ptr"):
        if not obj.is_contiguous():
            raise ValueError("tensor must be contiguous")
        return obj.data_ptr()
    raise TypeError(f"cannot pass {type(obj)} as a pointer")


def _check(rc: int, model_handle=None):
    if rc != DLS_OK:
        lib = load(False)
        msg = lib.dls_last_error(model_handle).decode(errors="replace")
        raise DlsError(rc, msg or lib.dls_status_name(rc).decode())


def status_name(code: int) -> str:
    return load().dls_status_name(code).decode()


def h2d_copy_sm(dst, src_host, nbytes: int, ctas: int = 64, stream=None):
    """Copy pinned host memory to the device with an SM-driven kernel."""
    _check(load().dls_h2d_copy_sm(_ptr(dst), _ptr(src_host), int(nbytes), int(ctas), _stream_handle(stream)))


def check_context_budget(prefix_tokens: int, max_branch_tokens: int, headroom: int, n_ctx: int) -> None:
    _check(load().dls_check_context_budget(prefix_tokens, max_branch_tokens, headroom, n_ctx))


def attention_workspace_bytes(n_batch, n_heads, n_kv_heads, head_dim, n_splits) -> int:
    return int(load().dls_attention_workspace_bytes(n_batch, n_heads, n_kv_heads, head_dim, n_splits))


def attention_decode(q, k_pages, v_pages, page_table, lengths, o, workspace, workspace_bytes, n_batch, n_heads,
                     n_kv_heads, head_dim, page_tokens, max_pages, n_splits=0, status=None, stream=None):
    """Split-K GQA decode attention over a paged fp16 cache (device buffers).
    ``status``: optional device int32[1] the kernel reports into; read it
    with attention_status()."""
    _check(load().dls_attention_decode(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table), _ptr(lengths),
                                       _ptr(o), _ptr(workspace), workspace_bytes, n_batch, n_heads, n_kv_heads,
                                       head_dim, page_tokens, max_pages, n_splits, _ptr(status),
                                       _stream_handle(stream)))


def attention_status(status, stream=None):
    """Wait for the stream and raise DlsError (DLS_ERR_STATE or
    DLS_ERR_TIMEOUT) if the attention kernel flagged its status word."""
    _check(load().dls_attention_status(_ptr(status), _stream_handle(stream)))


NOALLOC_SCRATCH_BYTES = 4 << 20  # DLS_ATTENTION_NOALLOC_SCRATCH_BYTES


def attention_decode_noalloc(q, k_pages, v_pages, page_table, lengths, o, n_batch, n_heads, n_kv_heads, head_dim,
                             page_tokens, max_pages, n_splits=0, status=None, stream=None):
    """dls_attention_decode without a workspace: for callers that may not
    allocate device memory; the scratch is a fixed array in the library."""
    _check(load().dls_attention_decode_noalloc(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table),
                                               _ptr(lengths), _ptr(o), n_batch, n_heads, n_kv_heads, head_dim,
                                               page_tokens, max_pages, n_splits, _ptr(status),
                                               _stream_handle(stream)))


DLS_Q4_K = 12
DLS_Q5_K = 13
DLS_Q6_K = 14
KQUANT_TYPES = {"q4_k": DLS_Q4_K, "q5_k": DLS_Q5_K, "q6_k": DLS_Q6_K}


def kquant_packed_bytes(fmt: str, rows: int, cols: int) -> int:
    return int(load().dls_kquant_packed_bytes(KQUANT_TYPES[fmt], rows, cols))


def kquant_pack(fmt: str, blocks, rows: int, cols: int, packed, stream=None):
    """GGUF K-quant super-blocks (device) -> the GEMV's device layout."""
    _check(load().dls_kquant_pack(KQUANT_TYPES[fmt], _ptr(blocks), rows, cols, _ptr(packed), _stream_handle(stream)))


def kquant_gemv(fmt: str, packed, rows: int, cols: int, x, y, status=None, stream=None):
    """y = W x on a packed K-quant matrix (device buffers)."""
    _check(load().dls_kquant_gemv(KQUANT_TYPES[fmt], _ptr(packed), rows, cols, _ptr(x), _ptr(y), _ptr(status),
                                  _stream_handle(stream)))


def _stream_handle(stream):
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class TorchAllocator:
    """Device memory from PyTorch's caching allocator, through the library's
    allocator callbacks.  ``live`` maps the pointers it handed out to their
    sizes.  ``fail_at`` = k makes the k-th allocation call from now on return
    NULL (the library then reports DLS_ERR_CUDA and rolls the call back);
    ``calls`` counts allocation calls."""

    def __init__(self, device: int, fail_at=None):
        import torch

        self.torch = torch
        self.device = device
        self.live = {}
        self.calls = 0
        self.fail_at = fail_at

        def _alloc(ctx, nbytes, stream):
            self.calls += 1
            if self.fail_at is not None:
                self.fail_at -= 1
                if self.fail_at == 0:
                    self.fail_at = None
                    return None
            try:
                p = torch.cuda.caching_allocator_alloc(int(nbytes), self.device, int(stream or 0))
                self.live[p] = nbytes
                return p
            except Exception:  # out of memory -> NULL -> DLS_ERR_CUDA
                return None

        def _free(ctx, ptr, stream):
            try:
                if ptr in self.live:
                    del self.live[ptr]
                    torch.cuda.caching_allocator_delete(ptr)
            except Exception:
                pass

        self._alloc_cb = dls_allocator._fields_[0][1](_alloc)
        self._free_cb = dls_allocator._fields_[1][1](_free)
        self.struct = dls_allocator(self._alloc_cb, self._free_cb, None)


class Model:
    """A model on the GPU: weights, paged KV pool, decode step.

    ``weights`` is the dict the synthetic generator returns (GGUF-style
    block bytes, host numpy arrays).  ``cfg`` supplies the shapes.
    """

    def __init__(self, cfg, weights, *, max_seqs=1, max_ctx=1024, max_batch=1, page_tokens=64,
                 device_budget_bytes=0, stream=None, torch_allocator=True, allocator=None, kv_pool_pages=0):
        self.lib = load()
        self.cfg = cfg
        self.stream = stream
        L = cfg.n_layers
        keep = []

        def host(a, dtype):
            a = np.ascontiguousarray(a, dtype=dtype)
            keep.append(a)
            return a.ctypes.data

        # per-matrix weight types (weights["formats"]: (layer, name) -> "q4_k" / "q5_k" / "q6_k"; others
        # are the config's Q8_0 / Q4_0)
        fmts = weights.get("formats", {})
        names = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")
        layers = (dls_layer_desc * L)()
        for l in range(L):
            lw = weights["layers"][l]
            if lw is None:
                raise ValueError(f"layer {l} weights missing")
            types = (i32 * 7)(*(KQUANT_TYPES.get(fmts.get((l, n)), 0) for n in names))
            layers[l] = dls_layer_desc(host(lw["attn_norm"], np.float32), host(lw["ffn_norm"], np.float32),
                                       *(host(lw[n], np.uint8) for n in names), types)
        out = weights.get("output")
        d = dls_model_desc(L, cfg.hidden, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn, cfg.vocab,
                           float(cfg.rope_theta), float(cfg.rms_eps), int(bool(cfg.tied)), int(cfg.wtype),
                           page_tokens, max_seqs, max_ctx, max_batch, int(device_budget_bytes),
                           host(weights["tok_embd"], np.uint8), None if out is None else host(out, np.uint8),
                           host(weights["output_norm"], np.float32), layers)
        d.kv_pool_pages = int(kv_pool_pages)
        d.tok_embd_type = KQUANT_TYPES.get(fmts.get((None, "tok_embd")), 0)
        d.output_type = KQUANT_TYPES.get(fmts.get((None, "output")), 0)
        self._alloc = None
        alloc_ptr = None
        if allocator is not None:
            self._alloc = allocator
            alloc_ptr = ctypes.pointer(allocator.struct)
        elif torch_allocator:
            import torch

            self._alloc = TorchAllocator(torch.cuda.current_device())
            alloc_ptr = ctypes.pointer(self._alloc.struct)
        h = vp()
        _check(self.lib.dls_model_create(ctypes.byref(d), alloc_ptr, _stream_handle(stream), ctypes.byref(h)))
        self.handle = h.value
        self.max_ctx, self.max_seqs, self.max_batch = max_ctx, max_seqs, max_batch

    def close(self):
        if getattr(self, "handle", None):
            self.lib.dls_model_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _c(self, rc):
        _check(rc, self.handle)

    # --- sequences
    def seq_create(self) -> int:
        s = i32()
        self._c(self.lib.dls_seq_create(self.handle, ctypes.byref(s)))
        return s.value

    def seq_free(self, seq: int):
        self._c(self.lib.dls_seq_free(self.handle, seq))

    def seq_length(self, seq: int) -> int:
        return int(self.lib.dls_seq_length(self.handle, seq))

    # --- hot path
    def prefill(self, seq: int, tokens, logits_out=None):
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        self._c(self.lib.dls_prefill(self.handle, seq, t.ctypes.data, t.size, _ptr(logits_out)))

    def decode_step(self, seq: int, token: int, pos: int, logits_out=None):
        self._c(self.lib.dls_decode_step(self.handle, seq, int(token), int(pos), _ptr(logits_out)))

    def decode_batch(self, seqs, tokens, pos, logits_out=None):
        s = np.ascontiguousarray(seqs, dtype=np.int32)
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        p = np.ascontiguousarray(pos, dtype=np.int32)
        self._c(self.lib.dls_decode_batch(self.handle, s.size, s.ctypes.data, t.ctypes.data, p.ctypes.data,
                                          _ptr(logits_out)))

    def generate(self, seqs, tokens, n_steps: int, last_logits=None) -> np.ndarray:
        s = np.ascontiguousarray(seqs, dtype=np.int32)
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        out = np.empty((n_steps, s.size), dtype=np.int32)
        self._c(self.lib.dls_generate(self.handle, s.size, s.ctypes.data, t.ctypes.data, n_steps, out.ctypes.data,
                                      _ptr(last_logits)))
        return out

    def argmax(self, logits, n_rows: int, out=None):
        res = np.empty(n_rows, dtype=np.int32) if out is None else out
        self._c(self.lib.dls_argmax(self.handle, _ptr(logits), n_rows, _ptr(res)))
        return res

    def kv_fork(self, src_seq: int, dst_seqs, shared: bool = False):
        """Fork src's KV into each destination: a page copy, or (shared=True)
        shared prefix pages plus a private copy of the partly filled page."""
        d = np.ascontiguousarray(dst_seqs, dtype=np.int32)
        fn = self.lib.dls_kv_fork_shared if shared else self.lib.dls_kv_fork
        self._c(fn(self.handle, src_seq, d.ctypes.data, d.size))

    def kv_free_pages(self) -> int:
        return int(self.lib.dls_kv_free_pages(self.handle))

    # --- layer skip
    def set_layer_skip(self, skip=None):
        """Layers decode steps skip (a boolean per layer), or None for none."""
        if skip is None:
            self._c(self.lib.dls_set_layer_skip(self.handle, None, 0))
            return
        a = np.ascontiguousarray(np.asarray(skip, dtype=bool).astype(np.uint8))
        self._c(self.lib.dls_set_layer_skip(self.handle, a.ctypes.data, a.size))

    def layer_cosines(self, seq: int, token: int, pos: int) -> np.ndarray:
        """One decode step; cosine of each layer's output with its input."""
        out = np.zeros(self.cfg.n_layers, dtype=np.float32)
        self._c(self.lib.dls_layer_cosines(self.handle, seq, int(token), int(pos), out.ctypes.data))
        return out

    def seq_truncate(self, seq: int, length: int):
        self._c(self.lib.dls_seq_truncate(self.handle, seq, int(length)))

    def verify(self, seq: int, tokens, logits_out=None) -> np.ndarray:
        """Score tokens at the sequence end in one pass; each position's greedy pick."""
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        out = np.empty(t.size, dtype=np.int32)
        self._c(self.lib.dls_verify(self.handle, seq, t.ctypes.data, t.size, _ptr(logits_out), out.ctypes.data))
        return out

    def generate_speculative(self, seq: int, token: int, n_tokens: int, draft_skip, draft_k: int = 3):
        """Greedy self-speculative generation; (tokens [n_tokens], stats dict)."""
        mask = np.ascontiguousarray(np.asarray(draft_skip, dtype=bool).astype(np.uint8))
        if mask.size != self.cfg.n_layers:
            raise ValueError(f"draft_skip has {mask.size} entries, the model {self.cfg.n_layers} layers")
        out = np.empty(int(n_tokens), dtype=np.int32)
        st = np.zeros(3, dtype=np.int32)
        self._c(self.lib.dls_generate_speculative(self.handle, seq, int(token), int(n_tokens), mask.ctypes.data,
                                                  int(draft_k), out.ctypes.data, st.ctypes.data))
        return out, {"rounds": int(st[0]), "drafted": int(st[1]), "accepted": int(st[2])}

    # --- residency
    def set_resident_layers(self, n: int):
        self._c(self.lib.dls_set_resident_layers(self.handle, n))

    def resident_layers(self) -> int:
        return int(self.lib.dls_resident_layers(self.handle))

    def layer_bytes(self) -> int:
        return int(self.lib.dls_layer_bytes(self.handle))

    def device_bytes(self) -> int:
        return int(self.lib.dls_device_bytes(self.handle))

    def device_budget(self) -> int:
        return int(self.lib.dls_device_budget(self.handle))

    # --- hooks
    def debug_capture(self, per_layer_out):
        self._c(self.lib.dls_debug_capture(self.handle, _ptr(per_layer_out)))

    def debug_bounded_wait(self, limit_ns: int):
        """A bounded device wait that nothing satisfies (raises DLS_ERR_TIMEOUT)."""
        self._c(self.lib.dls_debug_bounded_wait(self.handle, int(limit_ns)))

    def debug_read_kv(self, seq: int, layer: int, k_out, v_out):
        self._c(self.lib.dls_debug_read_kv(self.handle, seq, layer, _ptr(k_out), _ptr(v_out)))

    def debug_dequant(self, layer: int, tensor: str, out):
        self._c(self.lib.dls_debug_dequant(self.handle, layer, TENSOR_IDS[tensor], _ptr(out)))

    def debug_gemv(self, layer: int, tensor: str, x, y):
        self._c(self.lib.dls_debug_gemv(self.handle, layer, TENSOR_IDS[tensor], _ptr(x), _ptr(y)))

    def debug_gemm(self, layer: int, tensor: str, x, y):
        """y[t] = W x[t] with the prefill GEMM; x device fp32 [T][cols], y [T][rows]."""
        self._c(self.lib.dls_debug_gemm(self.handle, layer, TENSOR_IDS[tensor], int(x.shape[0]), _ptr(x), _ptr(y)))

    def profile_step(self, seq: int, token: int, pos: int, max_kernels: int = 4096):
        """(durations_ms, kinds) of every kernel of one decode step."""
        ms = np.zeros(max_kernels, dtype=np.float32)
        kinds = np.zeros(max_kernels, dtype=np.int32)
        n = i32()
        self._c(self.lib.dls_debug_profile_step(self.handle, seq, int(token), int(pos), max_kernels, ms.ctypes.data,
                                                kinds.ctypes.data, ctypes.byref(n)))
        return ms[: n.value].copy(), kinds[: n.value].copy()

    def profile_batch(self, seqs, tokens, pos, max_kernels: int = 8192):
        """(durations_ms, kinds) of every kernel of one batched decode step."""
        n = len(seqs)
        sa = np.ascontiguousarray(seqs, dtype=np.int32)
        ta = np.ascontiguousarray(tokens, dtype=np.int32)
        pa = np.ascontiguousarray(pos, dtype=np.int32)
        ms = np.zeros(max_kernels, dtype=np.float32)
        kinds = np.zeros(max_kernels, dtype=np.int32)
        cnt = i32()
        self._c(self.lib.dls_debug_profile_batch(self.handle, n, sa.ctypes.data, ta.ctypes.data, pa.ctypes.data,
                                                 max_kernels, ms.ctypes.data, kinds.ctypes.data, ctypes.byref(cnt)))
        return ms[: cnt.value].copy(), kinds[: cnt.value].copy()

    def step_trace(self, max_entries: int = 1 << 22) -> np.ndarray:
        """Per-CTA phase timestamps of the last profiled persistent step: [phase, cta, 4] (ns)."""
        out = np.zeros(max_entries, dtype=np.uint64)
        n = ctypes.c_int32(0)
        self._c(self.lib.dls_debug_step_trace(self.handle, out.ctypes.data, max_entries, ctypes.byref(n)))
        return out[: n.value]

    def launches_per_step(self) -> int:
        return int(self.lib.dls_debug_launches_per_step(self.handle))

    def step_kernel_in_use(self):
        """(True, None) when batch-1 steps run as the persistent step kernel,
        else (False, reason)."""
        why = ctypes.c_char_p()
        used = bool(self.lib.dls_step_kernel_in_use(self.handle, ctypes.byref(why)))
        return used, (why.value.decode() if why.value else None)

    def last_error(self) -> str:
        return self.lib.dls_last_error(self.handle).decode(errors="replace")
