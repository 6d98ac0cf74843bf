"""The seeded input generators: determinism and bf16 rounding."""
import numpy as np

import workloads as wl


def test_bf16_round_to_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 0.0, -0.0, 3.0e38], dtype=np.float32)
    bits = wl.f32_to_bf16(x)
    # 1+2^-8 is a tie between 0x3F80 and 0x3F81: to even (0x3F80); 1+3*2^-8 rounds up to 0x3F82
    assert list(bits) == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x0000, 0x8000, 0x7F62]
    np.testing.assert_array_equal(wl.bf16_to_f32(bits[:4]), [1.0, 1.0, 1.0 + 2 ** -6, -2.5])


def test_generators_are_deterministic_and_per_stream():
    cfg = wl.scaled(wl.HEADLINE, N=3, V=4096, d=64, E=64, r=32, H=32)
    a, b = wl.logits(cfg), wl.logits(cfg)
    np.testing.assert_array_equal(a, b)
    assert not np.array_equal(a[0], a[1])
    np.testing.assert_array_equal(a[1], wl.stream_logits(cfg, 1))
    one = wl.scaled(wl.HEADLINE, N=1, V=4096, d=64, E=64, r=32, H=32)
    np.testing.assert_array_equal(wl.logits(one)[0], a[0])
    w1, w2 = wl.weights(cfg), wl.weights(cfg)
    for k in wl.WEIGHT_NAMES:
        np.testing.assert_array_equal(w1[k], w2[k])
    assert np.all(wl.weights(cfg, "delta_zero")["w2"] == 0)


def test_distributions():
    cfg = wl.scaled(wl.QWEN3_8B, V=20000, d=512, E=512, r=64, H=64)
    x = wl.to_f64(wl.logits(cfg), "bf16")
    assert abs(x.std() - 3.0) < 0.05
    e = wl.to_f64(wl.embedding(cfg), "bf16")
    assert abs(e.std() - 0.02) < 0.001
    u = wl.uniforms(cfg)
    assert u.dtype == np.float32 and u.min() >= 0 and u.max() < 1
    q = wl.verifier_probs(cfg.replace(N=2, V=1000))
    np.testing.assert_allclose(q.sum(axis=2), 1.0, rtol=1e-5)
    W = wl.to_f64(wl.lm_head(cfg), "bf16")
    assert W.shape == (cfg.V, cfg.d)
    assert abs(W.std() - 3.0 / np.sqrt(cfg.d)) < 0.002


def test_grid_logits():
    x = wl.grid_logits([[1.0, 2.0], [3.0, 4.0], [5.0, 6.0]], V=16)
    assert x.shape == (1, 3, 16)
    assert x[0, 1, 2] == 3.0 and x[0, 2, 5] == 6.0 and x[0, 0, 7] == -100.0
