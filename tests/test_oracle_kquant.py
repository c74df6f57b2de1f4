"""Pins for the K-quant oracle (Q4_K, Q6_K super-blocks and the dequant-GEMV).

Blocks are assembled here field by field from the layout the oracle's
docstring states, by writers that run the opposite way to its readers
(packing values into bytes rather than unpacking them), so that a swapped
field, a wrong shift or nibble, or a misplaced index fails.
"""
from fractions import Fraction

import numpy as np
import pytest

import synth
from oracle import kquant as kq


def _f16le(v: float) -> list:
    b = int(np.array([v], dtype=np.float16).view(np.uint16)[0])
    return [b & 0xFF, b >> 8]


def _pack_q4_k(d, dmin, sc, m, q):
    """One Q4_K super-block from d, dmin, eight (sc, m) pairs and 256 codes."""
    blk = np.zeros(144, dtype=np.uint8)
    blk[0:2] = _f16le(d)
    blk[2:4] = _f16le(dmin)
    s12 = [0] * 12
    for s in range(8):
        if s < 4:
            s12[s] |= sc[s]
            s12[s + 4] |= m[s]
        else:
            s12[s + 4] = (sc[s] & 15) | ((m[s] & 15) << 4)
            s12[s - 4] |= (sc[s] >> 4) << 6
            s12[s] |= (m[s] >> 4) << 6
    blk[4:16] = s12
    for i in range(256):
        g, r = divmod(i, 64)
        byte = 16 + 32 * g + (r % 32)
        blk[byte] |= q[i] if r < 32 else q[i] << 4
    return blk


def _pack_q5_k(d, dmin, sc, m, q):
    """One Q5_K super-block from d, dmin, eight (sc, m) pairs and 256 codes 0..31."""
    low = [v & 15 for v in q]
    q4 = _pack_q4_k(d, dmin, sc, m, low)
    blk = np.zeros(176, dtype=np.uint8)
    blk[0:16] = q4[0:16]
    blk[48:176] = q4[16:144]
    for i in range(256):
        g, r = divmod(i, 64)
        bit = 2 * g + (1 if r >= 32 else 0)
        blk[16 + (r % 32)] |= (q[i] >> 4) << bit
    return blk


def _pack_q6_k(d, scales, code):
    """One Q6_K super-block from d, sixteen int8 scales and 256 codes 0..63."""
    blk = np.zeros(210, dtype=np.uint8)
    for i in range(256):
        h, o = divmod(i, 128)
        g, l = divmod(o, 32)
        low, high = code[i] & 15, code[i] >> 4
        at = 64 * h + l + (32 if g % 2 else 0)
        blk[at] |= low if g < 2 else low << 4
        blk[128 + 32 * h + l] |= high << (2 * g)
    blk[192:208] = np.array(scales, dtype=np.int8).view(np.uint8)
    blk[208:210] = _f16le(d)
    return blk


def test_q4_k_uniform_block_closed_form():
    for q, a, b in [(0, 0, 0), (15, 63, 0), (7, 1, 63), (15, 63, 63), (3, 40, 17)]:
        blk = _pack_q4_k(0.5, 0.25, [a] * 8, [b] * 8, [q] * 256)
        w = kq.dequant_q4_k(blk, 1)[0]
        assert np.all(w == 0.5 * a * q - 0.25 * b), (q, a, b)


def test_q4_k_every_nibble_lands_on_its_weight():
    # one code of 1 at a time, unit scales, no minimums: exactly one weight is d
    for i in range(256):
        q = [0] * 256
        q[i] = 1
        w = kq.dequant_q4_k(_pack_q4_k(1.0, 0.0, [1] * 8, [0] * 8, q), 1)[0]
        assert w[i] == 1.0 and np.count_nonzero(w) == 1, i
    # and the byte written for weight 64g + 32 + l is the high nibble of byte 32g + l
    q = [0] * 256
    q[64 + 32 + 5] = 9
    blk = _pack_q4_k(1.0, 0.0, [1] * 8, [0] * 8, q)
    assert blk[16 + 32 + 5] == 9 << 4


@pytest.mark.parametrize("seed", range(5))
def test_q4_k_six_bit_scales_and_minimums(seed):
    rng = np.random.default_rng(seed)
    sc = [int(v) for v in rng.integers(0, 64, 8)]
    m = [int(v) for v in rng.integers(0, 64, 8)]
    sc[5], m[6] = 63, 48                        # top bits set in the split fields
    blk = _pack_q4_k(1.0, 1.0, sc, m, [1] * 256)
    got_sc, got_m = kq.q4_k_scales_mins(blk[None, 4:16])
    assert list(got_sc[0]) == sc and list(got_m[0]) == m
    w = kq.dequant_q4_k(blk, 1)[0]
    for s in range(8):
        assert np.all(w[32 * s: 32 * s + 32] == sc[s] - m[s]), s


def test_q5_k_uniform_block_closed_form():
    for q, a, b in [(0, 0, 0), (31, 63, 0), (16, 1, 63), (31, 63, 63), (17, 40, 17)]:
        blk = _pack_q5_k(0.5, 0.25, [a] * 8, [b] * 8, [q] * 256)
        w = kq.dequant_q5_k(blk, 1)[0]
        assert np.all(w == 0.5 * a * q - 0.25 * b), (q, a, b)


def test_q5_k_every_code_lands_on_its_weight():
    # 1 (low bits only) and 16 (fifth bit only) at one weight at a time
    for v in (1, 16):
        for i in range(256):
            q = [0] * 256
            q[i] = v
            w = kq.dequant_q5_k(_pack_q5_k(1.0, 0.0, [1] * 8, [0] * 8, q), 1)[0]
            assert w[i] == float(v) and np.count_nonzero(w) == 1, (v, i)
    # the fifth bit of weight 64g + 32 + l is bit 2g + 1 of qh byte l
    q = [0] * 256
    q[128 + 32 + 7] = 16
    assert _pack_q5_k(1.0, 0.0, [1] * 8, [0] * 8, q)[16 + 7] == 1 << 5


@pytest.mark.parametrize("seed", range(3))
def test_q5_k_scales_and_minimums_as_q4_k(seed):
    rng = np.random.default_rng(10 + seed)
    sc = [int(v) for v in rng.integers(0, 64, 8)]
    m = [int(v) for v in rng.integers(0, 64, 8)]
    w = kq.dequant_q5_k(_pack_q5_k(1.0, 1.0, sc, m, [17] * 256), 1)[0]
    for s_ in range(8):
        assert np.all(w[32 * s_: 32 * s_ + 32] == 17 * sc[s_] - m[s_]), s_


def test_q6_k_uniform_block_closed_form():
    for c, a in [(32, 5), (0, 1), (63, -128), (40, 127), (31, -3)]:
        blk = _pack_q6_k(0.125, [a] * 16, [c] * 256)
        w = kq.dequant_q6_k(blk, 1)[0]
        assert np.all(w == 0.125 * a * (c - 32)), (c, a)


def test_q6_k_every_code_lands_on_its_weight():
    # background code 32 (weight 0); one weight at a time gets 33 (low bits)
    # or 48 (high bits only): exactly that weight is nonzero
    for bump in (1, 16, 31):
        for i in range(256):
            code = [32] * 256
            code[i] = 32 + bump
            w = kq.dequant_q6_k(_pack_q6_k(1.0, [1] * 16, code), 1)[0]
            assert w[i] == float(bump) and np.count_nonzero(w) == 1, (bump, i)


def test_q6_k_scale_k_covers_weights_16k_to_16k_plus_15():
    scales = [int(v) for v in np.random.default_rng(3).integers(-128, 128, 16)]
    w = kq.dequant_q6_k(_pack_q6_k(2.0, scales, [33] * 256), 1)[0]
    for i in range(256):
        assert w[i] == 2.0 * scales[i // 16], i


def test_fp16_scales_are_little_endian():
    blk = _pack_q6_k(1.0, [1] * 16, [33] * 256)
    blk[208], blk[209] = 0x00, 0xC0            # 0xC000 = -2.0
    assert np.all(kq.dequant_q6_k(blk, 1)[0] == -2.0)
    blk = _pack_q4_k(1.0, 0.0, [1] * 8, [0] * 8, [1] * 256)
    blk[0], blk[1] = 0x00, 0x38                # 0x3800 = 0.5
    assert np.all(kq.dequant_q4_k(blk, 1)[0] == 0.5)


@pytest.mark.parametrize("fmt", ["q4_k", "q5_k", "q6_k"])
def test_gemv_exact_against_fractions(fmt):
    rows, cols = 3, 512
    b = synth.kquant_matrix(synth.stream_key("kq-pin", fmt), rows, cols, fmt)
    x = synth.normal(synth.stream_key("kq-pin-x", fmt), cols, 1.0)
    y = kq.gemv(b, rows, cols, fmt, x, chunk_rows=2)
    w = kq.matrix_rows(b, cols, fmt, 0, rows)
    for r in range(rows):
        exact = sum(Fraction(float(w[r, c])) * Fraction(float(x[c])) for c in range(cols))
        assert abs(Fraction(float(y[r])) - exact) <= abs(exact) * Fraction(1, 10 ** 12) + Fraction(1, 10 ** 15)
    # rows come out in order: row r of the matrix is super-blocks r*cols/256 ..
    one = kq.dequant_blocks(b[(cols // 256) * kq.BLOCK_BYTES[fmt]:], cols // 256, fmt)
    assert np.array_equal(one.reshape(-1), w[1])


def test_rejects_ragged_columns():
    with pytest.raises(ValueError):
        kq.matrix_rows(np.zeros(144, dtype=np.uint8), 300, "q4_k", 0, 1)


# Plausible mistakes, planted in a copy of the oracle on the CPU: each must
# make at least one of the pins above fail.
_MUTANTS = [
    ("((b[:, s] >> 6) << 4)", "((b[:, s - 4] >> 6) << 4)"),                       # minimum's top bits from the wrong byte
    ("= qs[:, 32 * g: 32 * g + 32] >> 4", "= qs[:, 32 * g: 32 * g + 32] & 0x0F"),  # high nibble read as low
    (">> (2 * g)) & 3", ">> (2 * (g ^ 1))) & 3"),                                 # Q6_K high bits of the wrong group
    ("np.arange(QK) // 16]", "np.arange(QK) // 16 ^ 1]"),                         # neighbouring Q6_K scale
    ("low = src & 0x0F if g < 2 else src >> 4", "low = src & 0x0F if g % 2 == 0 else src >> 4"),
    ("- dmin[:, None] * m[:, sub]\n\n\ndef dequant_q5_k", "+ dmin[:, None] * m[:, sub]\n\n\ndef dequant_q5_k"),  # minimum's sign
    ("(((qh >> (2 * g)) & 1) << 4)", "(((qh >> (2 * g + 1)) & 1) << 4)"),        # Q5_K fifth bit of the wrong weight
    ("qh = b[:, 16:48]", "qh = b[:, 48:80]"),                                      # Q5_K field offsets
]


@pytest.mark.parametrize("old,new", _MUTANTS)
def test_pins_catch_planted_mistakes(old, new, monkeypatch):
    import importlib.util
    import sys
    src = open(kq.__file__).read()
    assert src.count(old) == 1, old
    spec = importlib.util.spec_from_loader("kquant_mutant", loader=None)
    mutant = importlib.util.module_from_spec(spec)
    exec(compile(src.replace(old, new), "kquant_mutant", "exec"), mutant.__dict__)
    monkeypatch.setitem(sys.modules, "kquant_mutant", mutant)
    monkeypatch.setattr(sys.modules[__name__], "kq", mutant)
    pins = [test_q4_k_uniform_block_closed_form, test_q4_k_every_nibble_lands_on_its_weight,
            lambda: test_q4_k_six_bit_scales_and_minimums(0), test_q6_k_uniform_block_closed_form,
            test_q6_k_every_code_lands_on_its_weight, test_q6_k_scale_k_covers_weights_16k_to_16k_plus_15,
            test_q5_k_uniform_block_closed_form, test_q5_k_every_code_lands_on_its_weight,
            lambda: test_q5_k_scales_and_minimums_as_q4_k(0)]
    failed = 0
    for pin in pins:
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed >= 1


# ---------------------------------------------------------------- K-quant matrices inside the model

def _q4_0_and_q4_k(rng, rows, cols):
    """The same weights as Q4_0 blocks and as Q4_K super-blocks: every Q4_0
    block of a 256-column run shares one scale d, so the Q4_K form with
    d, dmin = d, every sub-block scale 1 and minimum 8 gives d * (q - 8)
    exactly, weight for weight."""
    nsb = cols // 256
    q = rng.integers(0, 16, size=(rows, cols))
    d = (rng.uniform(0.5, 1.5, size=(rows, nsb)) * 2.0 ** -6).astype(np.float16).astype(np.float64)
    q40 = np.zeros((rows, cols // 32, 18), dtype=np.uint8)
    q4k = np.zeros((rows, nsb, 144), dtype=np.uint8)
    for r in range(rows):
        for b in range(cols // 32):
            q40[r, b, 0:2] = _f16le(d[r, b // 8])
            for j in range(16):
                q40[r, b, 2 + j] = q[r, 32 * b + j] | (q[r, 32 * b + 16 + j] << 4)
        for s_ in range(nsb):
            q4k[r, s_] = _pack_q4_k(d[r, s_], d[r, s_], [1] * 8, [8] * 8, list(q[r, 256 * s_: 256 * s_ + 256]))
    return q40.reshape(-1), q4k.reshape(-1)


def test_a_q4_k_model_equals_the_q4_0_model_with_the_same_weights():
    from oracle.model import OracleModel
    from synth.configs import ModelConfig
    cfg = ModelConfig("kqmix", 2, 256, 4, 2, 64, 512, 48, 10000.0, 4, 0.05)
    rng = np.random.default_rng(5)
    shapes = synth.matrix_shapes(cfg)
    w40 = synth.model_weights(cfg)
    wk = dict(w40, layers=[dict(lw) for lw in w40["layers"]], formats={})
    for l in range(cfg.n_layers):
        for name in synth.LAYER_MATRICES:
            rows, cols = shapes[name]
            a, b = _q4_0_and_q4_k(rng, rows, cols)
            w40["layers"][l][name] = a
            wk["layers"][l][name] = b
            wk["formats"][(l, name)] = "q4_k"
    m40, mk = OracleModel(cfg, w40), OracleModel(cfg, wk)
    for l in range(cfg.n_layers):
        for name in synth.LAYER_MATRICES:
            assert np.array_equal(m40.matrix(l, name), mk.matrix(l, name)), (l, name)
    # the same weights give the same model (up to the BLAS summation order,
    # which may follow the arrays' placement in memory)
    toks = synth.prompt_tokens(cfg, 5, seed=2)
    s40, sk = m40.new_seq(), mk.new_seq()
    np.testing.assert_allclose(m40.prefill(s40, toks), mk.prefill(sk, toks), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(m40.decode_step(s40, 7, 5), mk.decode_step(sk, 7, 5), rtol=1e-12, atol=1e-13)


def test_a_mixed_k_quant_model_prefill_equals_sequential_decode():
    # Q4_K_M-style mix: value and down projections Q6_K, the rest Q4_K / Q5_K
    from oracle.model import OracleModel
    from synth.configs import ModelConfig
    cfg = ModelConfig("kqmix2", 2, 256, 4, 2, 64, 512, 48, 10000.0, 4, 0.05)
    shapes = synth.matrix_shapes(cfg)
    w = synth.model_weights(cfg)
    w["formats"] = {}
    for l in range(cfg.n_layers):
        for name in synth.LAYER_MATRICES:
            rows, cols = shapes[name]
            fmt = "q6_k" if name in ("wv", "w_down") else ("q5_k" if l == 1 and name == "wq" else "q4_k")
            w["layers"][l][name] = synth.kquant_matrix(synth.stream_key("kqmix2", l, name), rows, cols, fmt)
            w["formats"][(l, name)] = fmt
    m = OracleModel(cfg, w)
    toks = synth.prompt_tokens(cfg, 6, seed=4)
    s1, s2 = m.new_seq(), m.new_seq()
    lg1 = m.prefill(s1, toks)
    for i, t in enumerate(toks):
        lg2 = m.decode_step(s2, int(t), i)
    np.testing.assert_allclose(lg1, lg2, rtol=1e-12, atol=1e-13)
    # and the matrices really are read in their own formats
    assert np.array_equal(m.matrix(0, "wv"), kq.matrix_rows(w["layers"][0]["wv"], 256, "q6_k", 0, shapes["wv"][0]))
