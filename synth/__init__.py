"""Seeded synthetic inputs for the decode-step library and its oracle.

This package is an input generator only: it draws weights and token ids and
quantises the weights into the GGUF-style Q8_0 / Q4_0 blocks that both the CUDA
library and the fp64 oracle consume.  It holds none of the decode step's
arithmetic (no dequantisation, norm, RoPE, attention or projection), and it
imports neither the library nor the oracle.

The generator itself is C (``csrc/synth.c``: SplitMix64 counters, Box-Muller
normals, block quantisers), compiled on first use with the host compiler.
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess
import threading

import numpy as np

from .configs import CONFIGS, ModelConfig, get_config  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csrc", "synth.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "libsynth.so")
_lock = threading.Lock()
_lib = None

Q8_0 = 8
Q4_0 = 4
BLOCK_BYTES = {Q8_0: 34, Q4_0: 18}


def build(force: bool = False) -> str:
    """Compile the generator into ``_lib/libsynth.so`` (gcc, OpenMP)."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-std=c11", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            u64, i64, i32, dbl = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32, ctypes.c_double
            vp = ctypes.c_void_p
            lib.synth_normal.argtypes = [u64, u64, i64, dbl, vp]
            lib.synth_normal.restype = None
            lib.synth_tokens.argtypes = [u64, i64, i32, vp]
            lib.synth_tokens.restype = None
            lib.synth_quant_matrix.argtypes = [u64, i64, i64, dbl, ctypes.c_int, vp]
            lib.synth_quant_matrix.restype = ctypes.c_int
            lib.synth_quant_matrix_k.argtypes = [u64, i64, i64, dbl, ctypes.c_int, vp]
            lib.synth_quant_matrix_k.restype = ctypes.c_int
            lib.synth_quantize.argtypes = [vp, i64, ctypes.c_int, vp]
            lib.synth_quantize.restype = ctypes.c_int
            lib.synth_f64_to_f16.argtypes = [dbl]
            lib.synth_f64_to_f16.restype = ctypes.c_uint16
            lib.synth_f16_to_f64.argtypes = [ctypes.c_uint16]
            lib.synth_f16_to_f64.restype = dbl
            _lib = lib
    return _lib


def stream_key(*parts) -> int:
    """64-bit stream key from a name path, e.g. stream_key("8b", 3, "wq")."""
    s = "/".join(str(p) for p in parts).encode()
    return int.from_bytes(hashlib.blake2b(s, digest_size=8).digest(), "little")


def normal(key: int, n: int, sigma: float = 1.0, start: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _load().synth_normal(key, start, n, sigma, out.ctypes.data)
    return out


def tokens(key: int, n: int, vocab: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    _load().synth_tokens(key, n, vocab, out.ctypes.data)
    return out


def quant_matrix(key: int, rows: int, cols: int, sigma: float, wtype: int) -> np.ndarray:
    """[rows x cols] N(0, sigma) matrix quantised to blocks (uint8, flat)."""
    nb = (cols + 31) // 32
    out = np.empty(rows * nb * BLOCK_BYTES[wtype], dtype=np.uint8)
    rc = _load().synth_quant_matrix(key, rows, cols, sigma, wtype, out.ctypes.data)
    if rc != 0:
        raise ValueError(f"bad wtype {wtype}")
    return out


KQUANT_KIND = {"q4_k": 12, "q5_k": 13, "q6_k": 14}


def quant_matrix_k(key: int, rows: int, cols: int, sigma: float, fmt: str) -> np.ndarray:
    """[rows x cols] N(0, sigma) matrix (the same draws as quant_matrix with
    this key) quantised to K-quant super-blocks (uint8, flat)."""
    if cols % 256:
        raise ValueError(f"cols={cols} is not a multiple of 256")
    out = np.empty(rows * (cols // 256) * KQUANT_BLOCK_BYTES[fmt], dtype=np.uint8)
    if _load().synth_quant_matrix_k(key, rows, cols, sigma, KQUANT_KIND[fmt], out.ctypes.data) != 0:
        raise ValueError(f"bad K-quant format {fmt}")
    return out


def quantize(x: np.ndarray, wtype: int) -> np.ndarray:
    """Quantise given values (length a multiple of 32) into blocks."""
    x = np.ascontiguousarray(x, dtype=np.float64).ravel()
    out = np.empty(x.size // 32 * BLOCK_BYTES[wtype], dtype=np.uint8)
    if _load().synth_quantize(x.ctypes.data, x.size, wtype, out.ctypes.data) != 0:
        raise ValueError("length must be a multiple of 32 and wtype 8 or 4")
    return out


def f64_to_f16_bits(v: float) -> int:
    return int(_load().synth_f64_to_f16(float(v)))


# --------------------------------------------------------------------------
# whole-model weights


def matrix_shapes(cfg: ModelConfig) -> dict:
    """Logical [rows, cols] of each per-layer matrix (cols = input features)."""
    H, hd = cfg.hidden, cfg.head_dim
    return {
        "wq": (cfg.n_heads * hd, H),
        "wk": (cfg.n_kv_heads * hd, H),
        "wv": (cfg.n_kv_heads * hd, H),
        "wo": (H, cfg.n_heads * hd),
        "w_gate": (cfg.ffn, H),
        "w_up": (cfg.ffn, H),
        "w_down": (H, cfg.ffn),
    }


LAYER_MATRICES = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")


def layer_weights(cfg: ModelConfig, layer: int) -> dict:
    out = {}
    for name, (rows, cols) in matrix_shapes(cfg).items():
        out[name] = quant_matrix(stream_key(cfg.name, layer, name), rows, cols, cfg.sigma, cfg.wtype)
    out["attn_norm"] = np.ones(cfg.hidden, dtype=np.float32)
    out["ffn_norm"] = np.ones(cfg.hidden, dtype=np.float32)
    return out


def model_weights(cfg: ModelConfig, layers=None) -> dict:
    """All weights of a config as host arrays (GGUF-style blocks).

    ``layers`` restricts which layers are generated (others are None); the
    embedding, output matrix and output norm are always generated.
    """
    H, V = cfg.hidden, cfg.vocab
    w = {
        "config": cfg,
        "tok_embd": quant_matrix(stream_key(cfg.name, "tok_embd"), V, H, cfg.sigma, cfg.wtype),
        "output_norm": np.ones(H, dtype=np.float32),
    }
    w["output"] = None if cfg.tied else quant_matrix(stream_key(cfg.name, "output"), V, H, cfg.sigma, cfg.wtype)
    sel = range(cfg.n_layers) if layers is None else layers
    w["layers"] = [layer_weights(cfg, l) if l in sel else None for l in range(cfg.n_layers)]
    return w


def with_random_gains(w: dict, cfg: ModelConfig, sigma: float = 0.2, tag: str = "gains") -> dict:
    """A copy of the weights `w` whose RMSNorm gains are seeded draws instead
    of ones: every layer's attn_norm and ffn_norm and the output_norm, each
    element N(1, sigma), stored fp32.  The matrices are shared with `w`."""
    H = cfg.hidden
    out = dict(w)
    out["output_norm"] = (1.0 + normal(stream_key(cfg.name, tag, "output_norm"), H, sigma)).astype(np.float32)
    layers = []
    for l, lw in enumerate(w["layers"]):
        if lw is None:
            layers.append(None)
            continue
        lw = dict(lw)
        for name in ("attn_norm", "ffn_norm"):
            lw[name] = (1.0 + normal(stream_key(cfg.name, tag, l, name), H, sigma)).astype(np.float32)
        layers.append(lw)
    out["layers"] = layers
    return out


# A Q4_K_M-style mix (the engine page, section 1: 70B as Q4_K_M): the value
# and down projections and the LM head in Q6_K, every other matrix in Q4_K.
Q4_K_M = {"wq": "q4_k", "wk": "q4_k", "wv": "q6_k", "wo": "q4_k", "w_gate": "q4_k", "w_up": "q4_k",
          "w_down": "q6_k", "tok_embd": "q4_k", "output": "q6_k"}


def model_weights_k(cfg: ModelConfig, formats: dict, layers=None) -> dict:
    """model_weights with matrices in per-matrix formats: `formats` maps a
    matrix name (the seven layer matrices, "tok_embd", "output") to "q4_k",
    "q5_k", "q6_k", or is missing it (the config's Q8_0 / Q4_0).  Every layer
    uses the same formats.  The result carries weights["formats"], keyed
    (layer, name) (layer None for tok_embd and output), which the oracle
    reads; the normals are those of model_weights."""
    H, V = cfg.hidden, cfg.vocab
    fm = {}

    def mat(key, rows, cols, name, layer):
        f = formats.get(name)
        if f is None:
            return quant_matrix(key, rows, cols, cfg.sigma, cfg.wtype)
        fm[(layer, name)] = f
        return quant_matrix_k(key, rows, cols, cfg.sigma, f)

    w = {"config": cfg, "output_norm": np.ones(H, dtype=np.float32),
         "tok_embd": mat(stream_key(cfg.name, "tok_embd"), V, H, "tok_embd", None)}
    w["output"] = None if cfg.tied else mat(stream_key(cfg.name, "output"), V, H, "output", None)
    sel = range(cfg.n_layers) if layers is None else layers
    shapes = matrix_shapes(cfg)
    out_layers = []
    for l in range(cfg.n_layers):
        if l not in sel:
            out_layers.append(None)
            continue
        lw = {name: mat(stream_key(cfg.name, l, name), rows, cols, name, l) for name, (rows, cols) in shapes.items()}
        lw["attn_norm"] = np.ones(H, dtype=np.float32)
        lw["ffn_norm"] = np.ones(H, dtype=np.float32)
        out_layers.append(lw)
    w["layers"] = out_layers
    w["formats"] = fm
    return w


def prompt_tokens(cfg: ModelConfig, n: int, seed: int = 1) -> np.ndarray:
    return tokens(stream_key(cfg.name, "prompt", seed), n, cfg.vocab)


# --------------------------------------------------------------------------
# K-quant super-blocks (Q4_K: 144 bytes, Q6_K: 210 bytes per 256 weights)

KQUANT_BLOCK_BYTES = {"q4_k": 144, "q5_k": 176, "q6_k": 210}


def kquant_matrix(key: int, rows: int, cols: int, fmt: str) -> np.ndarray:
    """[rows x cols] matrix of seeded K-quant super-blocks (uint8, flat,
    row-major, cols / 256 per row).  Every code and sub-block scale byte is
    uniform over its range; the fp16 super-block scales are drawn in
    [0.5, 1.5) x 2^-12 (Q4_K d and dmin), x 2^-13 (Q5_K) or x 2^-14 (Q6_K
    d), which keeps weights within about +-0.25, the spread of a trained
    model's."""
    if cols % 256:
        raise ValueError(f"cols={cols} is not a multiple of 256")
    bb = KQUANT_BLOCK_BYTES[fmt]
    nblk = rows * (cols // 256)
    raw = tokens(key, nblk * bb, 256).astype(np.uint8).reshape(nblk, bb)
    u = tokens(key ^ 0x5BD1E995, 2 * nblk, 256).astype(np.float64).reshape(nblk, 2)
    if fmt in ("q4_k", "q5_k"):
        for j, at in enumerate((0, 2)):
            d = ((0.5 + u[:, j] / 256.0) * 2.0 ** (-12 if fmt == "q4_k" else -13)).astype(np.float16).view(np.uint16)
            raw[:, at] = d & 0xFF
            raw[:, at + 1] = d >> 8
    else:
        d = ((0.5 + u[:, 0] / 256.0) * 2.0 ** -14).astype(np.float16).view(np.uint16)
        raw[:, 208] = d & 0xFF
        raw[:, 209] = d >> 8
    return raw.reshape(-1)
