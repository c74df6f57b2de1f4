"""Pins for how the oracle's layer wires its parts together: which matrix
feeds q, k, v, the attention output, gate and up; which norm gain goes where
and after the normalisation; that attention and FFN add to the residual
stream, and that the FFN normalises the stream after the attention; which
matrix the LM head reads.  (The engine page, sections 1 and 4.4: RMSNorm
with a gain, GQA attention over the KV cache, SwiGLU, residual connections.)

A one-layer micro model (hidden 32, one head of 32, FFN 32, vocab 4) is
built from hand-written Q8_0 blocks whose weights are exact: scaled
identities, a diagonal, a reversal, zero matrices.  With constant token
embeddings every quantity then has a closed form in a handful of scalars --
rho(c) = c / sqrt(c^2 + eps) for the RMSNorm of a constant vector c, silu for
SwiGLU -- so each case below is a short hand derivation, not the oracle's
code again.  eps is 0.25 so that rho depends visibly on c.  Planted swaps in
a copy of the oracle (CPU only) must each fail one of these pins.
"""
import importlib.util
import math
import sys

import numpy as np
import pytest

from oracle import model as oracle_model
from synth.configs import ModelConfig

H = 32
EPS = 0.25
CFG = ModelConfig("wiring", 1, H, 1, 1, H, H, 4, 10000.0, 8, 0.02, rms_eps=EPS)
G_ATTN, G_FFN, G_OUT = 2.0, 0.5, 4.0
TOKEN_C = [0.5, 0.25, 1.0, 0.75]        # token t's embedding is TOKEN_C[t] * ones


def _f16_bits(v: float) -> int:
    return int(np.array([v], dtype=np.float16).view(np.uint16)[0])


def _matrix(d: float, q: np.ndarray) -> np.ndarray:
    """Q8_0 blocks of a [rows x 32] matrix: weight[r, c] = d * q[r, c] with d
    a power of two (exact in fp16) and |q| <= 127."""
    q = np.asarray(q, dtype=np.int64)
    assert q.shape[1] == 32 and np.all(np.abs(q) <= 127)
    bits = _f16_bits(d)
    out = np.zeros((q.shape[0], 34), dtype=np.uint8)
    out[:, 0] = bits & 0xFF
    out[:, 1] = bits >> 8
    out[:, 2:] = (q & 0xFF).astype(np.uint8)
    return out.reshape(-1)


def _scaled_identity(scale_q: int, d: float) -> np.ndarray:
    return _matrix(d, np.eye(32, dtype=np.int64) * scale_q)


def _zero() -> np.ndarray:
    return _matrix(1.0, np.zeros((32, 32), dtype=np.int64))


def _weights(**layer) -> dict:
    """Embeddings c_t * ones (Q8_0, d = 2^-6), LM head row j = (j+1)/64 * ones;
    gains G_ATTN, G_FFN, G_OUT; layer matrices as given (zero by default)."""
    emb = _matrix(2.0 ** -6, np.array([[round(c * 64)] * 32 for c in TOKEN_C]))
    out = _matrix(2.0 ** -6, np.array([[j + 1] * 32 for j in range(4)]))
    lw = {name: _zero() for name in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")}
    lw.update(layer)
    lw["attn_norm"] = np.full(H, G_ATTN, dtype=np.float32)
    lw["ffn_norm"] = np.full(H, G_FFN, dtype=np.float32)
    return {"config": CFG, "tok_embd": emb, "output": out, "output_norm": np.full(H, G_OUT, dtype=np.float32),
            "layers": [lw]}


def rho(c: float) -> float:
    """RMSNorm of the constant vector c * ones, per element (unit gain)."""
    return c / math.sqrt(c * c + EPS)


def silu(z: float) -> float:
    return z / (1.0 + math.exp(-z))


def f16(v):
    return np.asarray(v, dtype=np.float64).astype(np.float16).astype(np.float64)


IDX = np.arange(H)
DIAG_V = (IDX + 1) / 64.0                      # Wv = diag((i+1)/64)


def _attention_model(mod):
    """Wq = 0, Wk = 0.25 I, Wv = diag((i+1)/64), Wo = 0.5 * reversal, no FFN."""
    w = _weights(wk=_scaled_identity(64, 2.0 ** -8),
                 wv=_matrix(2.0 ** -6, np.diag(IDX + 1)),
                 wo=_matrix(2.0 ** -7, np.fliplr(np.eye(32, dtype=np.int64)) * 64))
    return mod.OracleModel(CFG, w)


def pin_attention_wiring(mod=oracle_model):
    m = _attention_model(mod)
    s = m.new_seq()
    cap = []
    m.decode_step(s, 0, 0, capture=cap)
    kA = G_ATTN * rho(TOKEN_C[0])              # the normalised embedding, per element
    # the cache holds fp16(Wk xn) and fp16(Wv xn) (RoPE at position 0 is the identity)
    np.testing.assert_array_equal(s.keys(0)[0, 0], f16(np.full(H, 0.25 * kA)))
    vA = f16(kA * DIAG_V)
    np.testing.assert_array_equal(s.values(0)[0, 0], vA)
    # one key: the attention output is that key's cached value; Wo reverses
    # and halves it, and the result adds to the embedding
    np.testing.assert_allclose(cap[0], TOKEN_C[0] + 0.5 * vA[::-1], rtol=1e-14, atol=0)
    # second token at position 1: q = Wq xn = 0 gives equal scores, so the
    # output is the mean of the two cached values
    cap = []
    m.decode_step(s, 3, 1, capture=cap)
    vB = f16(G_ATTN * rho(TOKEN_C[3]) * DIAG_V)
    np.testing.assert_array_equal(s.values(0)[1, 0], vB)
    np.testing.assert_allclose(cap[0], TOKEN_C[3] + 0.5 * ((vA + vB) / 2)[::-1], rtol=1e-14, atol=0)


def _ffn_model(mod, with_attention: bool):
    """Wg = 1.0 I, Wu = 0.75 I, Wdown = 0.5 I; attention off (Wo = 0), or
    Wv = 0.5 I, Wo = 0.25 I (it adds a constant to the stream)."""
    layer = dict(w_gate=_scaled_identity(64, 2.0 ** -6), w_up=_scaled_identity(48, 2.0 ** -6),
                 w_down=_scaled_identity(64, 2.0 ** -7))
    if with_attention:
        layer.update(wv=_scaled_identity(64, 2.0 ** -7), wo=_scaled_identity(64, 2.0 ** -8))
    return mod.OracleModel(CFG, _weights(**layer))


def _ffn_closed_form(c: float, with_attention: bool):
    """Residual after the layer and the logits, for a constant input c."""
    x1 = c
    if with_attention:
        x1 = c + 0.25 * float(f16(0.5 * G_ATTN * rho(c)))   # o = the one cached value fp16(Wv xn)
    s = G_FFN * rho(x1)                                     # the FFN input, per element
    x2 = x1 + 0.5 * silu(1.0 * s) * (0.75 * s)              # down(silu(gate) * up)
    logits = np.array([G_OUT * rho(x2) * 32 * (j + 1) / 64.0 for j in range(4)])
    return x2, logits


@pytest.mark.parametrize("with_attention", [False, True])
def test_ffn_wiring_and_norm_gains(with_attention, mod=oracle_model):
    m = _ffn_model(mod, with_attention)
    for t in (0, 2):
        s = m.new_seq()
        cap = []
        lg = m.decode_step(s, t, 0, capture=cap)
        x2, logits = _ffn_closed_form(TOKEN_C[t], with_attention)
        np.testing.assert_allclose(cap[0], np.full(H, x2), rtol=1e-13, atol=0)
        np.testing.assert_allclose(lg, logits, rtol=1e-13, atol=0)


def test_attention_wiring():
    pin_attention_wiring()


def test_prefill_uses_the_same_wiring():
    # the two tokens of the attention case as one prefill: the last token's
    # residual equals the closed form of the second decode step
    m = _attention_model(oracle_model)
    s = m.new_seq()
    cap = []
    m.prefill(s, [0, 3], capture=cap)
    vA = f16(G_ATTN * rho(TOKEN_C[0]) * DIAG_V)
    vB = f16(G_ATTN * rho(TOKEN_C[3]) * DIAG_V)
    np.testing.assert_allclose(cap[0], TOKEN_C[3] + 0.5 * ((vA + vB) / 2)[::-1], rtol=1e-14, atol=0)


# Plausible wiring slips, planted in a copy of oracle/model.py on the CPU.
_MUTANTS = [
    ('ops.swiglu(self.matmul(layer, "w_gate", xn), self.matmul(layer, "w_up", xn))',
     'ops.swiglu(self.matmul(layer, "w_up", xn), self.matmul(layer, "w_gate", xn))'),        # gate <-> up
    ('xn = ops.rmsnorm(X, self.norm_gain(layer, "attn_norm"), cfg.rms_eps)',
     'xn = ops.rmsnorm(X, self.norm_gain(layer, "ffn_norm"), cfg.rms_eps)'),                  # attention reads the FFN gain
    ('xn = ops.rmsnorm(X, self.norm_gain(layer, "ffn_norm"), cfg.rms_eps)',
     'xn = ops.rmsnorm(X, self.norm_gain(layer, "attn_norm"), cfg.rms_eps)'),                 # FFN reads the attention gain
    ('q = self.matmul(layer, "wq", xn)', 'q = self.matmul(layer, "wk", xn)'),                 # q from Wk
    ('k = self.matmul(layer, "wk", xn)', 'k = self.matmul(layer, "wq", xn)'),                 # k from Wq
    ('v = self.matmul(layer, "wv", xn)', 'v = self.matmul(layer, "wk", xn)'),                 # v from Wk
    ('X = X + self.matmul(layer, "wo", o.reshape(T, nh * hd))',
     'X = self.matmul(layer, "wo", o.reshape(T, nh * hd))'),                                  # attention replaces the stream
    ('X = X + self.matmul(layer, "w_down", h)', 'X = self.matmul(layer, "w_down", h)'),       # FFN replaces the stream
    ('xn = ops.rmsnorm(X, self.norm_gain(layer, "ffn_norm"), cfg.rms_eps)',
     'xn = ops.rmsnorm(np.atleast_2d(x), self.norm_gain(layer, "ffn_norm"), cfg.rms_eps)'),   # FFN normalises the layer input
    ('xn = ops.rmsnorm(x, self.norm_gain(None, "output_norm"), self.cfg.rms_eps)',
     'xn = ops.rmsnorm(x, np.ones(self.cfg.hidden), self.cfg.rms_eps)'),                      # output gain dropped
    ('if name == "output" and self.w.get("output") is None:\n                return self.w["tok_embd"]',
     'if name == "output":\n                return self.w["tok_embd"]'),                      # LM head reads the embedding
    ('return x / np.sqrt(ms + eps) * np.asarray(g, dtype=np.float64)',
     'return x * np.asarray(g, dtype=np.float64) / np.sqrt(np.mean((x * np.asarray(g, dtype=np.float64)) ** 2, '
     'axis=-1, keepdims=True) + eps)'),                                                       # gain applied before normalising
]


def _mutant_module(old: str, new: str):
    """A copy of oracle.model (or of oracle.ops, for the gain placement) with one edit."""
    import oracle.ops as ops_mod
    target = ops_mod if old.startswith("return x / np.sqrt") else oracle_model
    src = open(target.__file__).read()
    assert src.count(old) >= 1, old
    src = src.replace(old, new, 1)
    spec = importlib.util.spec_from_loader("oracle._wiring_mutant", loader=None)
    mut = importlib.util.module_from_spec(spec)
    mut.__package__ = "oracle"
    exec(compile(src, f"{target.__name__}_mutant", "exec"), mut.__dict__)
    if target is ops_mod:
        # the model module, reading the mutated ops
        msrc = open(oracle_model.__file__).read()
        mmut = importlib.util.module_from_spec(importlib.util.spec_from_loader("oracle._wiring_mutant_m", loader=None))
        mmut.__package__ = "oracle"
        exec(compile(msrc, "oracle.model_mutant", "exec"), mmut.__dict__)
        mmut.ops = mut
        return mmut
    return mut


@pytest.mark.parametrize("old,new", _MUTANTS)
def test_wiring_pins_catch_planted_mistakes(old, new):
    mut = _mutant_module(old, new)
    pins = [lambda: pin_attention_wiring(mut),
            lambda: test_ffn_wiring_and_norm_gains(False, mut),
            lambda: test_ffn_wiring_and_norm_gains(True, mut)]
    failed = 0
    for pin in pins:
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed >= 1, f"no pin caught: {new}"


def test_unmutated_copy_passes_every_pin():
    # the copy mechanism itself changes nothing
    mut = _mutant_module('v = self.matmul(layer, "wv", xn)', 'v = self.matmul(layer, "wv", xn)')
    pin_attention_wiring(mut)
    test_ffn_wiring_and_norm_gains(False, mut)
    test_ffn_wiring_and_norm_gains(True, mut)
    assert sys.modules.get("oracle._wiring_mutant") is None
