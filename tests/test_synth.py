"""The seeded input generator: determinism, distribution, formats.  CPU only."""
import numpy as np
import pytest

import synth
from synth.configs import CONFIGS


def test_normal_is_counter_based():
    key = synth.stream_key("t", 1)
    a = synth.normal(key, 1000)
    b = synth.normal(key, 600, start=400)
    np.testing.assert_array_equal(a[400:], b)
    assert not np.array_equal(a, synth.normal(synth.stream_key("t", 2), 1000))


def test_normal_moments():
    x = synth.normal(synth.stream_key("moments"), 1 << 20, 0.02)
    assert abs(x.mean()) < 1e-4
    assert abs(x.std() - 0.02) < 1e-4
    # fourth moment of a normal is 3 sigma^4
    assert abs(np.mean(x ** 4) / 0.02 ** 4 - 3.0) < 0.05


def test_quant_matrix_matches_quantize_of_normals():
    key = synth.stream_key("qm")
    rows, cols = 5, 96
    x = synth.normal(key, rows * cols, 0.02)
    for wt in (8, 4):
        np.testing.assert_array_equal(synth.quant_matrix(key, rows, cols, 0.02, wt), synth.quantize(x, wt))


@pytest.mark.filterwarnings("ignore:overflow encountered in cast")  # values past the fp16 range, on purpose
def test_f16_conversion_matches_numpy():
    v = np.concatenate([synth.normal(3, 20000, 1.0), synth.normal(4, 20000, 1e-5),
                        synth.normal(5, 2000, 3e4), [0.0, -0.0, 65504.0, 65519.99, 2 ** -25, 3 * 2 ** -26]])
    ours = np.array([synth.f64_to_f16_bits(x) for x in v], dtype=np.uint16)
    ref = v.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


def test_tokens_in_range():
    t = synth.tokens(synth.stream_key("tok"), 10000, 128256)
    assert t.min() >= 0 and t.max() < 128256
    assert len(np.unique(t)) > 9000


def test_config_parameter_counts():
    # per-layer parameter counts of the shapes
    assert CONFIGS["8b"].layer_params() == 218_103_808
    assert CONFIGS["70b"].layer_params() == 855_638_016
    assert CONFIGS["1b"].layer_params() == 60_817_408


def test_random_gains_are_seeded_and_leave_matrices_shared():
    cfg = CONFIGS["tiny"]
    w = synth.model_weights(cfg)
    g1 = synth.with_random_gains(w, cfg)
    g2 = synth.with_random_gains(w, cfg)
    for l in range(cfg.n_layers):
        a, f = g1["layers"][l]["attn_norm"], g1["layers"][l]["ffn_norm"]
        assert a.dtype == np.float32 and a.shape == (cfg.hidden,)
        np.testing.assert_array_equal(a, g2["layers"][l]["attn_norm"])
        assert not np.array_equal(a, f)                       # distinct per norm
        assert np.all(w["layers"][l]["attn_norm"] == 1.0)     # the source is untouched
        assert g1["layers"][l]["wq"] is w["layers"][l]["wq"]
    assert not np.array_equal(g1["layers"][0]["attn_norm"], g1["layers"][1]["attn_norm"])
    allg = np.concatenate([g1["output_norm"]] + [g1["layers"][l][n] for l in range(cfg.n_layers)
                                                 for n in ("attn_norm", "ffn_norm")])
    assert abs(allg.mean() - 1.0) < 0.03 and abs(allg.std() - 0.2) < 0.03


def test_k_quant_matrices_round_trip_and_share_the_normals():
    # the K-quant generator quantises the very normals of the Q8_0 generator
    # (same key, same element order); the oracle's reader turns its blocks
    # back into weights within each format's step
    from oracle import kquant
    key = synth.stream_key("kq-roundtrip")
    rows, cols = 6, 768
    x = synth.normal(key, rows * cols, 0.02).reshape(rows, cols)
    for fmt, bound in (("q4_k", 0.08), ("q5_k", 0.04), ("q6_k", 0.02)):
        b = synth.quant_matrix_k(key, rows, cols, 0.02, fmt)
        assert b.size == rows * (cols // 256) * synth.KQUANT_BLOCK_BYTES[fmt]
        w = kquant.matrix_rows(b, cols, fmt, 0, rows)
        assert np.max(np.abs(w - x)) <= bound * np.max(np.abs(x)), fmt
        assert abs(w.std() - x.std()) < 0.05 * x.std()
    with pytest.raises(ValueError):
        synth.quant_matrix_k(key, 2, 300, 0.02, "q4_k")


def test_q4_k_m_model_weights_carry_their_formats():
    cfg = CONFIGS["tiny"]
    import dataclasses
    cfgk = dataclasses.replace(cfg, ffn=768)
    w = synth.model_weights_k(cfgk, synth.Q4_K_M)
    assert w["formats"][(0, "wv")] == "q6_k" and w["formats"][(1, "wq")] == "q4_k"
    assert w["formats"][(None, "output")] == "q6_k" and w["formats"][(None, "tok_embd")] == "q4_k"
    assert w["layers"][0]["w_down"].size == cfgk.hidden * (768 // 256) * 210
