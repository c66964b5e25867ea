"""The seeded input generator: determinism, shapes, planted structure."""
import numpy as np

from dspark_draft_sampling_gb300 import synth


def test_deterministic_and_shaped():
    a = synth.markov_inputs(2, 3, 1000, 64, seed=5, d2t="injective", tie_frac=0.01)
    b = synth.markov_inputs(2, 3, 1000, 64, seed=5, d2t="injective", tie_frac=0.01)
    for key in ("base", "w1", "w2", "d2t", "prev0", "ties"):
        np.testing.assert_array_equal(a[key], b[key])
    assert a["base"].shape == (2, 3, 1000) and a["base"].dtype == np.float32
    assert a["w1"].shape == (1000, 64) and a["w1"].dtype == np.uint16
    assert a["prev0"].dtype == np.int64 and np.all((a["prev0"] >= 0) & (a["prev0"] < 1000))
    c = synth.markov_inputs(2, 3, 1000, 64, seed=6)
    assert not np.array_equal(a["base"], c["base"])


def test_d2t_injective_into_target_vocab():
    a = synth.markov_config("reduced_vocab")
    d = a["d2t"]
    assert d.shape == (32000,) and d.dtype == np.int32
    assert len(np.unique(d)) == 32000
    assert d.min() >= 0 and d.max() < synth.TARGET_VOCAB


def test_planted_ties():
    a = synth.markov_config("reduced_vocab")
    ties = a["ties"]
    assert len(ties) == 160
    assert np.all(ties[:, 0] < ties[:, 1])
    assert len(np.unique(ties)) == 320
    np.testing.assert_array_equal(a["w2"][ties[:, 0]], a["w2"][ties[:, 1]])
    np.testing.assert_array_equal(a["base"][:, :, ties[:, 0]], a["base"][:, :, ties[:, 1]])
    assert a["spiked_steps"] == [0, 2, 4, 6, 8]


def test_bf16_rounding_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1.0 + 2 ** -9], np.float32)
    bits = synth.f32_to_bf16_bits(x)
    back = (bits.astype(np.uint32) << 16).view(np.float32)
    np.testing.assert_array_equal(back, [1.0, 1.0, 1.0 + 2 ** -6, -2.5, 1.0])


def test_probe_layout():
    p = synth.probe_inputs(3, 7424, seed=0)
    assert p["wq"].shape == (232 * 34,)
    blk = p["wq"].reshape(232, 34)
    d = blk[:, :2].copy().view("<u2").reshape(-1).view(np.float16)
    assert np.all(d == np.float16(1e-3))
    q = blk[:, 2:].copy().view(np.int8)
    assert q.min() >= -127 and q.max() <= 127
    assert p["hidden"].shape == (3, 7424)
    assert 0.0 < p["threshold"] < 1.0


def test_ws_inputs():
    w = synth.ws_inputs(7, 64, 128, seed=1)
    assert w["W"].shape == (64, 128) and w["W"].dtype == np.uint16
    assert w["X"].shape == (7, 128)
