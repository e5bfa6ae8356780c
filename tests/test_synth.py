"""The seeded input generator: determinism, slicing, rounding and shape of the
distributions it promises."""
import numpy as np

import synth


def test_deterministic_and_prefix_stable():
    a = synth.normal_bf16(7, 5, (1000,), 0.02)
    b = synth.normal_bf16(7, 5, (1000,), 0.02)
    np.testing.assert_array_equal(a, b)
    c = synth.normal_bf16(7, 5, (301,), 0.02)      # odd length: the last pair is split
    np.testing.assert_array_equal(a[:301], c)
    assert not np.array_equal(a, synth.normal_bf16(7, 6, (1000,), 0.02))
    assert not np.array_equal(a, synth.normal_bf16(8, 5, (1000,), 0.02))


def test_thread_split_invariance():
    big = synth.normal_bf16(3, 1, (300001,), 1.0)  # multi-threaded path
    words = synth.words(3, 1, 10)
    assert len(set(words.tolist())) == 10
    np.testing.assert_array_equal(big[:1000], synth.normal_bf16(3, 1, (1000,), 1.0))
    np.testing.assert_array_equal(big[-5:], synth.normal_bf16(3, 1, (300001,), 1.0)[-5:])


def test_bf16_rounding_is_rne_of_f32():
    f = synth.normal_f32(1, 2, (10000,), 1.0)
    bits = synth.normal_bf16(1, 2, (10000,), 1.0)
    np.testing.assert_array_equal(synth.f32_to_bf16_bits(f), bits)
    # ties to even on hand-picked float32 bit patterns
    pats = np.array([0x3F808000, 0x3F818000, 0x3F80C000, 0xBF808000, 0x3F807FFF], dtype=np.uint32)
    got = synth.f32_to_bf16_bits(pats.view(np.float32))
    np.testing.assert_array_equal(got, np.array([0x3F80, 0x3F82, 0x3F81, 0xBF80, 0x3F80], dtype=np.uint16))
    back = synth.bf16_bits_to_f32(np.array([0x3F80, 0xC000, 0x4278], dtype=np.uint16))
    np.testing.assert_array_equal(back, np.array([1.0, -2.0, 62.0], dtype=np.float32))


def test_normal_moments():
    x = synth.normal_f32(7, 9, (400000,), 0.02).astype(np.float64)
    assert abs(x.mean()) < 0.02 * 0.01
    assert abs(x.std() / 0.02 - 1.0) < 0.01
    z = x / 0.02
    assert abs(np.mean(z ** 4) - 3.0) < 0.05           # normal kurtosis
    assert abs(np.mean(np.abs(z) < 1.0) - 0.682689) < 0.003


def test_uniform_ids():
    ids = synth.uniform_ids(99, 0, (200000,), 49152)
    assert ids.dtype == np.int32 and ids.min() >= 0 and ids.max() < 49152
    hist = np.bincount(ids // 4096, minlength=12)
    assert np.all(np.abs(hist / hist.mean() - 1.0) < 0.05)


def test_weights_layout():
    cfg = synth.tiny_config("gemma")
    w = synth.make_weights(cfg)
    assert w["embed"].shape == (cfg.vocab, cfg.hidden)
    assert w["L0.wq"].shape == (cfg.n_q_heads * cfg.head_dim, cfg.hidden)
    assert w["L2.w_down"].shape == (cfg.hidden, cfg.intermediate)
    assert "lm_head" not in w and "L1.q_norm" in w and "L1.post_ffn_norm" in w
    assert np.all(w["final_norm"] == 0x3F80)
    # each tensor is reproducible alone
    np.testing.assert_array_equal(synth.make_tensor(cfg, "L1.w_up"), w["L1.w_up"])
