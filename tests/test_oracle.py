"""Pins for the fp64 oracle: closed forms, invariants, special cases and brute
force, each chosen so a plausible slip in the oracle (a dropped term, a wrong
sign or index, a transposed operand, the other RoPE pairing, a missing scale)
fails at least one of them.  CPU only.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import synth
from oracle import ops, quant
from oracle.model import OracleModel
from synth.configs import ModelConfig


# ---------------------------------------------------------------- dequant

def _q8_block(d_bits: int, q) -> bytes:
    return bytes([d_bits & 0xFF, d_bits >> 8]) + bytes((int(v) & 0xFF) for v in q)


def test_q8_0_every_code_unit_scale():
    # d = 1.0 (fp16 0x3C00): every weight equals its int8 code, -128..127.
    codes = list(range(-128, 128))
    blob = b"".join(_q8_block(0x3C00, codes[i:i + 32]) for i in range(0, 256, 32))
    w = quant.dequant_q8_0(np.frombuffer(blob, np.uint8), 8).ravel()
    assert w.tolist() == [float(c) for c in codes]


@pytest.mark.parametrize("d_bits,d_val", [
    (0x3800, Fraction(1, 2)),            # 0.5
    (0xC000, Fraction(-2)),              # -2.0: negative scale
    (0x0001, Fraction(1, 2 ** 24)),      # smallest subnormal
    (0x03FF, Fraction(1023, 2 ** 24)),   # largest subnormal
    (0x7BFF, Fraction(65504)),           # largest finite
    (0x3555, Fraction(0x555 | 0x400, 2 ** 11) / 2),  # 0.333251953125
])
def test_q8_0_scale_values(d_bits, d_val):
    q = [(-1) ** i * (3 * i + 1) for i in range(32)]
    w = quant.dequant_q8_0(np.frombuffer(_q8_block(d_bits, q), np.uint8), 1)[0]
    assert [Fraction(x) for x in w] == [d_val * v for v in q]


def test_q4_0_nibble_order():
    # byte j = (high nibble 15-j) << 4 | (low nibble j): element j = j - 8,
    # element j+16 = (15-j) - 8.  Swapping halves or interleaving fails this.
    body = bytes(((15 - j) << 4) | j for j in range(16))
    blob = bytes([0x00, 0x3C]) + body            # d = 1.0
    w = quant.dequant_q4_0(np.frombuffer(blob, np.uint8), 1)[0]
    assert w[:16].tolist() == [j - 8.0 for j in range(16)]
    assert w[16:].tolist() == [7.0 - j for j in range(16)]


def test_q4_0_scale_and_offset():
    body = bytes([0x80] * 16)  # low nibble 0 -> -8, high nibble 8 -> 0
    blob = bytes([0x00, 0xB8]) + body            # d = -0.5
    w = quant.dequant_q4_0(np.frombuffer(blob, np.uint8), 1)[0]
    assert w[:16].tolist() == [4.0] * 16
    assert w[16:].tolist() == [0.0] * 16


@pytest.mark.parametrize("wtype", [8, 4])
def test_quantiser_round_trip_bound(wtype):
    x = synth.normal(synth.stream_key("pin", "roundtrip", wtype), 32 * 512, 0.02)
    blocks = synth.quantize(x, wtype)
    w = quant.dequant_blocks(blocks, 512, wtype).ravel()
    xb = x.reshape(512, 32)
    amax = np.abs(xb).max(axis=1)
    d = amax / 127.0 if wtype == 8 else amax / 8.0
    # |x - w| <= |d|/2 from rounding, plus the effect of storing d in fp16
    # (relative error <= 2^-11, times the largest code magnitude 128 or 8).
    qmax = 128.0 if wtype == 8 else 8.0
    fp16_term = qmax * 2.0 ** -11
    err = np.abs(xb - w.reshape(512, 32))
    if wtype == 8:
        assert np.all(err <= (d * (0.5 + fp16_term))[:, None] + 1e-300)
    else:
        # Q4_0 codes stop at 15 (= +7 steps), so values beyond +7.5 steps on the
        # side opposite the block's extreme element are clamped: one full step.
        steps = np.abs(xb) / d[:, None]
        opposite = np.sign(xb) != np.sign(xb[np.arange(512), np.abs(xb).argmax(1)])[:, None]
        clamped = opposite & (steps > 7.5)
        lim = np.where(clamped, 1.0, 0.5) + fp16_term
        assert np.all(err <= lim * d[:, None] + 1e-300)
        assert clamped.any()   # the clamp case is exercised
    # and the extreme element of each block is reproduced to fp16 precision
    assert np.all(np.abs(np.abs(w.reshape(512, 32)).max(axis=1) - amax) <= amax * 2.0 ** -10)


def test_matrix_padding_columns_are_zero_weights():
    # 688 columns -> 22 blocks per row; the oracle returns exactly 688 columns
    rows, cols = 3, 688
    blocks = synth.quant_matrix(synth.stream_key("pin", "pad"), rows, cols, 0.02, 8)
    full = quant.dequant_q8_0(blocks, rows * 22).reshape(rows, 704)
    assert np.all(full[:, 688:] == 0.0)
    assert quant.matrix(blocks, rows, cols, 8).shape == (rows, cols)


def test_gemv_exact_against_fractions():
    # 24 x 64 Q8_0 matrix with power-of-two scales and dyadic inputs: the
    # fp64 product is exact, so it must equal the rational triple loop.
    rng = np.random.default_rng(7)
    rows, cols = 24, 64
    blob = bytearray()
    for r in range(rows):
        for b in range(2):
            d_bits = [0x3C00, 0x3800, 0x4000, 0x3400][(r + b) % 4]   # 1, .5, 2, .25
            blob += _q8_block(d_bits, rng.integers(-127, 128, 32))
    blob = np.frombuffer(bytes(blob), np.uint8)
    x = rng.integers(-64, 65, cols) / 16.0
    W = quant.matrix(blob, rows, cols, 8)
    y = W @ x
    for r in range(rows):
        acc = Fraction(0)
        for c in range(cols):
            blk = blob[(r * 2 + c // 32) * 34:(r * 2 + c // 32 + 1) * 34]
            d = {0x3C00: Fraction(1), 0x3800: Fraction(1, 2), 0x4000: Fraction(2),
                 0x3400: Fraction(1, 4)}[int(blk[0]) | int(blk[1]) << 8]
            q = int(np.int8(blk[2 + c % 32]))
            acc += d * q * Fraction(x[c])
        assert Fraction(y[r]) == acc


# ---------------------------------------------------------------- RMSNorm

@pytest.mark.parametrize("c", [0.02, -3.0, 1e-4])
def test_rmsnorm_constant_vector(c):
    n, eps = 256, 1e-5
    g = np.linspace(0.5, 1.5, n)
    y = ops.rmsnorm(np.full(n, c), g, eps)
    np.testing.assert_allclose(y, c / math.sqrt(c * c + eps) * g, rtol=1e-14)


def test_rmsnorm_unit_rms_and_rows():
    x = synth.normal(11, 3 * 64).reshape(3, 64)
    y = ops.rmsnorm(x, np.ones(64), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, rtol=1e-14)
    # row-wise: row 1 alone gives the same result
    np.testing.assert_allclose(ops.rmsnorm(x[1], np.ones(64), 0.0), y[1], rtol=1e-15)


# ---------------------------------------------------------------- RoPE

def test_rope_pos0_identity():
    v = synth.normal(12, 4 * 64).reshape(4, 64)
    np.testing.assert_array_equal(ops.rope(v, 0, 10000.0), v)


def test_rope_preserves_pair_norms_and_composes():
    v = synth.normal(13, 8 * 128).reshape(8, 128)
    for theta in (1e4, 5e5):
        r = ops.rope(v, 8191, theta)
        n0 = v[:, 0::2] ** 2 + v[:, 1::2] ** 2
        n1 = r[:, 0::2] ** 2 + r[:, 1::2] ** 2
        np.testing.assert_allclose(n1, n0, rtol=1e-12)
        np.testing.assert_allclose(ops.rope(ops.rope(v, 37, theta), 100, theta),
                                   ops.rope(v, 137, theta), rtol=1e-9, atol=1e-12)


def test_rope_adjacent_pairing_and_frequencies():
    # hd = 4: pair 0 = dims (0, 1) at frequency 1, pair 1 = dims (2, 3) at
    # frequency theta^(-1/2).  The half-split pairing (0, 2), (1, 3) fails.
    theta, p = 10000.0, 3
    e0 = np.array([[1.0, 0.0, 0.0, 0.0]])
    np.testing.assert_allclose(ops.rope(e0, p, theta)[0], [math.cos(3), math.sin(3), 0, 0], atol=1e-15)
    e2 = np.array([[0.0, 0.0, 1.0, 0.0]])
    a = p / 100.0   # theta^(-2*1/4) = 1/100
    np.testing.assert_allclose(ops.rope(e2, p, theta)[0], [0, 0, math.cos(a), math.sin(a)], atol=1e-15)
    e3 = np.array([[0.0, 0.0, 0.0, 1.0]])
    np.testing.assert_allclose(ops.rope(e3, p, theta)[0], [0, 0, -math.sin(a), math.cos(a)], atol=1e-15)


def test_rope_relative_position():
    # q.k after rotating both depends only on the position difference
    q = synth.normal(14, 64)[None]
    k = synth.normal(15, 64)[None]
    s1 = ops.rope(q, 50, 1e4)[0] @ ops.rope(k, 20, 1e4)[0]
    s2 = ops.rope(q, 1030, 1e4)[0] @ ops.rope(k, 1000, 1e4)[0]
    assert abs(s1 - s2) < 1e-10


# ---------------------------------------------------------------- softmax / attention

def test_softmax_rows_sum_to_one_and_shift_invariant():
    s = synth.normal(16, 5 * 33, 4.0).reshape(5, 33)
    p = ops.softmax(s)
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(ops.softmax(s + 123.0), p, rtol=1e-12)
    np.testing.assert_allclose(ops.softmax(np.array([0.0, math.log(3.0)])), [0.25, 0.75], rtol=1e-15)


def test_attention_single_key_returns_value():
    q = synth.normal(17, 4 * 64).reshape(4, 64)
    k = synth.normal(18, 2 * 64).reshape(1, 2, 64)
    v = synth.normal(19, 2 * 64).reshape(1, 2, 64)
    o = ops.attention(q, k, v)
    for h in range(4):
        np.testing.assert_array_equal(o[h], v[0, h // 2])


def test_attention_equal_scores_mean_of_values():
    q = synth.normal(20, 2 * 8).reshape(2, 8)
    k = np.repeat(synth.normal(21, 8).reshape(1, 1, 8), 5, axis=0)
    v = synth.normal(22, 5 * 8).reshape(5, 1, 8)
    o = ops.attention(q, k, v)
    np.testing.assert_allclose(o, np.repeat(v[:, 0].mean(0)[None], 2, 0), rtol=1e-13)


def test_attention_scale_is_inverse_sqrt_head_dim():
    # q.k1 = 0 and q.k2 = sqrt(hd)*ln 3 -> weights exactly 1/4, 3/4
    hd = 16
    q = np.zeros((1, hd)); q[0, 0] = 1.0
    k = np.zeros((2, 1, hd)); k[1, 0, 0] = math.sqrt(hd) * math.log(3.0)
    v = np.zeros((2, 1, hd)); v[0, 0, 1] = 4.0; v[1, 0, 2] = 4.0
    o = ops.attention(q, k, v)[0]
    np.testing.assert_allclose(o[1:3], [1.0, 3.0], rtol=1e-14)


def test_attention_gqa_head_mapping():
    # 8 query heads over 2 kv heads: heads 0-3 read kv 0, heads 4-7 kv 1
    hd, n = 4, 3
    q = synth.normal(23, 8 * hd).reshape(8, hd)
    k = synth.normal(24, n * 2 * hd).reshape(n, 2, hd)
    v = np.zeros((n, 2, hd)); v[:, 0, :] = 1.0; v[:, 1, :] = -2.0
    o = ops.attention(q, k, v)
    np.testing.assert_allclose(o[:4], 1.0, rtol=1e-14)
    np.testing.assert_allclose(o[4:], -2.0, rtol=1e-14)


def _brute_attention(q, k, v):
    nh, hd = q.shape
    n, nkv, _ = k.shape
    out = [[0.0] * hd for _ in range(nh)]
    for h in range(nh):
        kv = h * nkv // nh
        s = [sum(q[h][d] * k[j][kv][d] for d in range(hd)) / math.sqrt(hd) for j in range(n)]
        m = max(s)
        e = [math.exp(x - m) for x in s]
        z = sum(e)
        for d in range(hd):
            out[h][d] = sum(e[j] / z * v[j][kv][d] for j in range(n))
    return np.array(out)


@pytest.mark.parametrize("nh,nkv,n", [(4, 2, 1), (4, 2, 5), (2, 2, 4), (6, 3, 2), (4, 1, 5)])
def test_attention_brute_force(nh, nkv, n):
    hd = 4
    q = synth.normal(25 + n, nh * hd, 2.0).reshape(nh, hd)
    k = synth.normal(35 + n, n * nkv * hd, 2.0).reshape(n, nkv, hd)
    v = synth.normal(45 + n, n * nkv * hd).reshape(n, nkv, hd)
    np.testing.assert_allclose(ops.attention(q, k, v), _brute_attention(q, k, v), rtol=1e-12, atol=1e-14)


def test_gqa_with_one_group_is_mha():
    hd, n = 8, 6
    q = synth.normal(50, 3 * hd).reshape(3, hd)
    k = synth.normal(51, n * 3 * hd).reshape(n, 3, hd)
    v = synth.normal(52, n * 3 * hd).reshape(n, 3, hd)
    o = ops.attention(q, k, v)
    for h in range(3):
        s = k[:, h] @ q[h] / math.sqrt(hd)
        p = np.exp(s - s.max()); p /= p.sum()
        np.testing.assert_allclose(o[h], p @ v[:, h], rtol=1e-13)


def test_causal_attention_rows_match_single_query_attention():
    T, nh, nkv, hd = 5, 4, 2, 8
    q = synth.normal(53, T * nh * hd).reshape(T, nh, hd)
    k = synth.normal(54, T * nkv * hd).reshape(T, nkv, hd)
    v = synth.normal(55, T * nkv * hd).reshape(T, nkv, hd)
    o = ops.causal_attention(q, k, v)
    for t in range(T):
        np.testing.assert_allclose(o[t], ops.attention(q[t], k[:t + 1], v[:t + 1]), rtol=1e-13)
    # a later key never changes an earlier row
    k2 = k.copy(); k2[-1] += 10.0
    np.testing.assert_array_equal(ops.causal_attention(q, k2, v)[:-1], o[:-1])


# ---------------------------------------------------------------- SiLU / SwiGLU / fp16

def test_silu_closed_forms():
    assert ops.silu(np.array([0.0]))[0] == 0.0
    np.testing.assert_allclose(ops.silu(np.array([math.log(3.0)])), [0.75 * math.log(3.0)], rtol=1e-15)
    np.testing.assert_allclose(ops.silu(np.array([-math.log(3.0)])), [-0.25 * math.log(3.0)], rtol=1e-15)
    np.testing.assert_allclose(ops.silu(np.array([50.0])), [50.0], rtol=1e-20)
    np.testing.assert_allclose(ops.swiglu(np.array([math.log(3.0)]), np.array([2.0])),
                               [1.5 * math.log(3.0)], rtol=1e-15)


@pytest.mark.filterwarnings("ignore:overflow encountered in cast")  # values past the fp16 range, on purpose
def test_round_f16_nearest_even():
    # 1 + 2^-11 is halfway between 1 and 1 + 2^-10 -> ties to even (1.0);
    # 1 + 3*2^-11 -> 1 + 2^-9 (even mantissa)
    assert ops.round_f16(np.array([1 + 2 ** -11]))[0] == 1.0
    assert ops.round_f16(np.array([1 + 3 * 2 ** -11]))[0] == 1 + 2 ** -9
    assert ops.round_f16(np.array([70000.0]))[0] == np.inf


# ---------------------------------------------------------------- greedy

def test_greedy_ties_lowest_index():
    assert ops.greedy(np.array([1.0, 3.0, 3.0, 2.0])) == 1
    assert ops.top2_gap(np.array([1.0, 3.0, 2.5])) == pytest.approx(0.5)


# ---------------------------------------------------------------- composed model

MICRO = ModelConfig("micro", 2, 64, 4, 2, 16, 96, 48, 10000.0, 8, 0.05)


def _micro_weights(cfg=MICRO, wtype=None):
    cfg2 = cfg if wtype is None else ModelConfig(cfg.name + f"q{wtype}", cfg.n_layers, cfg.hidden,
                                                 cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn,
                                                 cfg.vocab, cfg.rope_theta, wtype, cfg.sigma)
    return cfg2, synth.model_weights(cfg2)


@pytest.mark.parametrize("wtype", [8, 4])
def test_prefill_equals_sequential_decode(wtype):
    cfg, w = _micro_weights(wtype=wtype)
    m = OracleModel(cfg, w)
    toks = synth.prompt_tokens(cfg, 7)
    s1 = m.new_seq()
    cap1 = []
    lg1 = m.prefill(s1, toks, capture=cap1)
    s2 = m.new_seq()
    for i, t in enumerate(toks):
        cap2 = []
        lg2 = m.decode_step(s2, int(t), i, capture=cap2)
    np.testing.assert_allclose(lg1, lg2, rtol=1e-12, atol=1e-13)
    for a, b in zip(cap1, cap2):
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)
    for l in range(cfg.n_layers):
        np.testing.assert_array_equal(s1.keys(l), s2.keys(l))


def test_zero_layers_pass_residual_through():
    # with every projection zero, each layer adds Wo*o = 0 and Wdown*h = 0
    cfg, w = _micro_weights()
    for lw in w["layers"]:
        for name in synth.LAYER_MATRICES:
            lw[name] = np.zeros_like(lw[name])
    m = OracleModel(cfg, w)
    cap = []
    s = m.new_seq()
    m.decode_step(s, 5, 0, capture=cap)
    x0 = m.embed(5)
    for x in cap:
        np.testing.assert_array_equal(x, x0)
    # zero k and v are cached as zeros
    assert np.all(s.keys(0) == 0) and np.all(s.values(1) == 0)


def test_zero_output_projections_keep_residual_but_fill_cache():
    cfg, w = _micro_weights()
    for lw in w["layers"]:
        lw["wo"] = np.zeros_like(lw["wo"])
        lw["w_down"] = np.zeros_like(lw["w_down"])
    m = OracleModel(cfg, w)
    s = m.new_seq()
    cap = []
    m.decode_step(s, 9, 0, capture=cap)
    np.testing.assert_array_equal(cap[-1], m.embed(9))
    # layer-0 key at pos 0 is fp16(Wk * rmsnorm(x0)) (RoPE at pos 0 is identity)
    xn = ops.rmsnorm(m.embed(9), np.ones(cfg.hidden), cfg.rms_eps)
    k = (m.matrix(0, "wk") @ xn).reshape(cfg.n_kv_heads, cfg.head_dim)
    np.testing.assert_array_equal(s.keys(0)[0], ops.round_f16(k))


def test_fork_equals_independent_prefill_and_position_matters():
    cfg, w = _micro_weights()
    m = OracleModel(cfg, w)
    prefix = synth.prompt_tokens(cfg, 6)
    base = m.new_seq()
    m.prefill(base, prefix)
    branch = base.fork()
    lg_fork = m.decode_step(branch, 3, len(prefix))
    indep = m.new_seq()
    m.prefill(indep, prefix)
    lg_ind = m.decode_step(indep, 3, len(prefix))
    np.testing.assert_array_equal(lg_fork, lg_ind)
    # the source is untouched by the branch's decode
    assert base.length == len(prefix)
    # restarting RoPE at 0 on the fork must change the result
    m2 = OracleModel(cfg, w)
    s3 = base.fork()
    s3.truncate(0)
    lg_pos0 = m2.decode_step(s3, 3, 0)
    assert np.max(np.abs(lg_pos0 - lg_fork)) > 1e-3


def test_decode_rejects_wrong_position():
    cfg, w = _micro_weights()
    m = OracleModel(cfg, w)
    s = m.new_seq()
    with pytest.raises(ValueError):
        m.decode_step(s, 1, 1)


def test_tied_output_reads_embedding():
    cfg = ModelConfig("microtied", 1, 64, 4, 2, 16, 96, 48, 10000.0, 8, 0.05, tied=True)
    w = synth.model_weights(cfg)
    assert w["output"] is None
    m = OracleModel(cfg, w)
    x = synth.normal(60, 64)
    xn = ops.rmsnorm(x, np.ones(64), cfg.rms_eps)
    np.testing.assert_allclose(m.final_logits(x), quant.matrix(w["tok_embd"], 48, 64, 8) @ xn, rtol=1e-14)


def test_selected_logit_rows_match_full_head():
    cfg, w = _micro_weights()
    m = OracleModel(cfg, w, cache_bytes=0, chunk_rows=7)   # forces chunked, uncached path
    x = synth.normal(61, 64)
    full = m.final_logits(x)
    rows = [0, 5, 47]
    np.testing.assert_allclose(m.final_logits(x, rows=rows), full[rows], rtol=1e-14)


# ---------------------------------------------------------------- layer skip (engine page, sections 2.5, 3.5, 4.5)

def test_cosine_closed_forms():
    v = np.array([3.0, -4.0, 12.0])
    w = np.array([4.0, 3.0, 0.0])                    # orthogonal to v
    assert ops.cosine(v, v) == pytest.approx(1.0, abs=1e-15)
    assert ops.cosine(v, -v) == pytest.approx(-1.0, abs=1e-15)
    assert ops.cosine(v, w) == pytest.approx(0.0, abs=1e-15)
    assert ops.cosine(2.0 * v, 3.0 * (v + w)) == pytest.approx(169.0 / (13.0 * np.sqrt(194.0)), rel=1e-14)
    assert ops.cosine(v, np.zeros(3)) == 0.0


def test_skipping_every_layer_leaves_the_embedding_and_no_cache():
    cfg, w = _micro_weights()
    m = OracleModel(cfg, w)
    s = m.new_seq()
    lg = m.decode_step(s, 7, 0, skip=set(range(cfg.n_layers)))
    np.testing.assert_array_equal(lg, m.final_logits(m.embed(7)))
    # no layer wrote the cache, but the step consumed position 0
    assert s.lens == [0] * cfg.n_layers and s.length == 1


def test_skipping_an_identity_layer_changes_nothing():
    # a layer with zero output projections adds nothing to the residual:
    # skipping it is exact, and its cosine (output vs input) is exactly 1
    cfg, w = _micro_weights()
    w["layers"][1]["wo"] = np.zeros_like(w["layers"][1]["wo"])
    w["layers"][1]["w_down"] = np.zeros_like(w["layers"][1]["w_down"])
    m = OracleModel(cfg, w)
    toks = synth.prompt_tokens(cfg, 5)
    a, b, c = m.new_seq(), m.new_seq(), m.new_seq()
    for i, t in enumerate(toks):
        la = m.decode_step(a, int(t), i)
        lb = m.decode_step(b, int(t), i, skip={1})
    np.testing.assert_array_equal(la, lb)
    assert b.lens == [5, 0]                              # the skipped layer appended nothing
    m.prefill(c, toks[:4])
    cos = m.layer_cosines(c, int(toks[4]), 4)
    assert cos[1] == pytest.approx(1.0, abs=1e-15)
    assert -1.0 <= cos[0] < 1.0


def test_layer_cosines_follow_the_captured_residuals():
    cfg, w = _micro_weights()
    m = OracleModel(cfg, w)
    s1, s2 = m.new_seq(), m.new_seq()
    cos = m.layer_cosines(s1, 9, 0)
    cap = []
    m.decode_step(s2, 9, 0, capture=cap)
    x0 = m.embed(9)
    # layer l: angle between what entered and what left
    for l, (xin, xout) in enumerate(zip([x0] + cap[:-1], cap)):
        num = sum(float(p) * float(q) for p, q in zip(xin, xout))
        den = np.sqrt(sum(float(p) ** 2 for p in xin)) * np.sqrt(sum(float(q) ** 2 for q in xout))
        assert cos[l] == pytest.approx(num / den, rel=1e-12)


# ---------------------------------------------------------------- self-speculative decoding (engine page, sections 3.5, 5.3)

DEEP = ModelConfig("deep", 4, 64, 4, 2, 16, 96, 48, 10000.0, 8, 0.05)


def test_prefill_rows_match_sequential_decode_logits():
    cfg, w = _micro_weights()
    m = OracleModel(cfg, w)
    toks = synth.prompt_tokens(cfg, 6)
    s1, s2 = m.new_seq(), m.new_seq()
    m.prefill(s1, toks[:2])
    m.prefill(s2, toks[:2])
    rows = m.prefill(s1, toks[2:], all_logits=True)
    assert rows.shape == (4, cfg.vocab) and s1.length == 6
    for i, t in enumerate(toks[2:]):
        np.testing.assert_allclose(rows[i], m.decode_step(s2, int(t), 2 + i), rtol=1e-12, atol=1e-13)


def test_truncate_then_decode_is_as_if_the_tail_never_ran():
    cfg, w = _micro_weights()
    m = OracleModel(cfg, w)
    toks = synth.prompt_tokens(cfg, 9)
    a, b = m.new_seq(), m.new_seq()
    m.prefill(a, toks[:5])
    m.prefill(b, toks[:5])
    for i in range(5, 9):
        m.decode_step(a, int(toks[i]), i)
    a.truncate(5)
    assert a.length == 5 and a.lens == [5, 5]
    np.testing.assert_array_equal(m.decode_step(a, 11, 5), m.decode_step(b, 11, 5))
    with pytest.raises(ValueError):
        a.truncate(7)


def _spec_setup(wtype=8, n_prompt=5):
    cfg, w = _micro_weights(DEEP, wtype)
    m = OracleModel(cfg, w)
    prompt = synth.prompt_tokens(cfg, n_prompt, seed=3)
    s = m.new_seq()
    first = ops.greedy(m.prefill(s, prompt))
    return cfg, m, prompt, s, first


@pytest.mark.parametrize("k", [1, 2, 3, 5])
@pytest.mark.parametrize("skip", [(), (3,), (1, 2), (0, 1, 2, 3)])
def test_speculative_tokens_are_the_full_greedy_tokens(k, skip):
    cfg, m, prompt, s, first = _spec_setup()
    ref = s.fork()
    n = 12
    want, _ = m.greedy_decode(ref, first, n)
    got, st = m.speculative_decode(s, first, n, skip, k)
    assert got == want
    assert s.length == ref.length == len(prompt) + n
    assert st["rounds"] + st["accepted"] == n and st["accepted"] <= st["drafted"]
    for l in range(cfg.n_layers):
        np.testing.assert_allclose(s.keys(l), ref.keys(l), rtol=1e-3, atol=1e-6)
        np.testing.assert_allclose(s.values(l), ref.values(l), rtol=1e-3, atol=1e-6)


@pytest.mark.parametrize("k", [1, 3, 4])
def test_speculative_with_the_full_model_as_draft_accepts_every_token(k):
    cfg, m, prompt, s, first = _spec_setup()
    n = 11
    _, st = m.speculative_decode(s, first, n, (), k)
    assert st["accepted"] == st["drafted"]
    assert st["rounds"] == -(-n // (k + 1))


@pytest.mark.parametrize("skip,k", [((3,), 3), ((1, 2), 2), ((0, 1, 2, 3), 3)])
def test_speculative_acceptance_matches_brute_force(skip, k):
    # rebuild every round from scratch: the cache holds the prompt and the
    # tokens emitted so far; the draft's greedy run is compared with the full
    # model's greedy tokens, and the common prefix is what a round accepts
    cfg, m, prompt, s, first = _spec_setup()
    n = 12
    full, _ = m.greedy_decode(s.fork(), first, n)
    _, st = m.speculative_decode(s, first, n, skip, k)
    emitted = [first] + full
    e = rounds = accepted = drafted = 0
    while e < n:
        r = min(k, n - e - 1)
        seq = m.new_seq()
        m.prefill(seq, list(prompt) + emitted[:e])
        drafts, _ = m.greedy_decode(seq, emitted[e], r, skip=set(skip))
        a = 0
        while a < r and drafts[a] == full[e + a]:
            a += 1
        e += a + 1
        rounds += 1
        accepted += a
        drafted += r
    assert (st["rounds"], st["drafted"], st["accepted"]) == (rounds, drafted, accepted)
    assert accepted < drafted       # this draft is wrong somewhere, so rejection is exercised


# ---------------------------------------------------------------- split softmax (cascade attention over a shared prefix)

@pytest.mark.parametrize("cuts", [[], [0], [5], [1, 2, 9], [11], [3, 3, 7]])
def test_merged_partials_equal_attention_over_all_keys(cuts):
    rng = np.random.default_rng(len(cuts) + sum(cuts))
    nh, nkv, hd, n = 4, 2, 16, 11
    q = rng.normal(size=(nh, hd))
    k = rng.normal(size=(n, nkv, hd)) * 2.0
    v = rng.normal(size=(n, nkv, hd))
    bounds = [0] + list(cuts) + [n]
    parts = [ops.attention_partial(q, k[a:b], v[a:b]) for a, b in zip(bounds[:-1], bounds[1:])]
    np.testing.assert_allclose(ops.merge_partials(parts), ops.attention(q, k, v), rtol=1e-12, atol=1e-14)
    # the order of the parts does not matter
    np.testing.assert_allclose(ops.merge_partials(parts[::-1]), ops.attention(q, k, v), rtol=1e-12, atol=1e-14)


def test_partial_of_one_key_and_of_none():
    q = np.array([[1.0, 0.0], [0.0, 2.0]])
    k = np.array([[[3.0, 4.0]]])
    v = np.array([[[5.0, -6.0]]])
    o, m, l = ops.attention_partial(q, k, v)
    # one key: the score itself is the maximum, its weight exp(0) = 1
    assert list(m) == pytest.approx([3.0 / np.sqrt(2.0), 8.0 / np.sqrt(2.0)], rel=1e-15)
    assert list(l) == [1.0, 1.0]
    np.testing.assert_array_equal(o, [[5.0, -6.0], [5.0, -6.0]])
    o0, m0, l0 = ops.attention_partial(q, k[:0], v[:0])
    assert np.all(m0 == -np.inf) and np.all(l0 == 0) and np.all(o0 == 0)


def test_prefix_and_branch_parts_rebuild_a_forked_decode_step():
    # a fork's branch attends over the shared prefix and its own positions:
    # the two parts merged give the oracle's decode-step attention
    cfg, w = _micro_weights()
    m = OracleModel(cfg, w)
    toks = synth.prompt_tokens(cfg, 9)
    base = m.new_seq()
    m.prefill(base, toks[:6])
    br = base.fork()
    for i, t in enumerate(toks[6:]):
        m.decode_step(br, int(t), 6 + i)
    q = synth.normal(77, cfg.n_heads * cfg.head_dim).reshape(cfg.n_heads, cfg.head_dim)
    k, v = br.keys(1), br.values(1)
    whole = ops.attention(q, k, v)
    merged = ops.merge_partials([ops.attention_partial(q, k[:6], v[:6]), ops.attention_partial(q, k[6:], v[6:])])
    np.testing.assert_allclose(merged, whole, rtol=1e-12, atol=1e-14)
