"""Pins of the confidence-probe oracle (Q8_0 dot + logit-space gate)."""
import math

import numpy as np
import pytest

import oracle
from oracle import brute
from dspark_draft_sampling_gb300 import synth


def _blocks(inp):
    nb = inp["K"] // 32
    b = inp["wq"].reshape(nb, 34)
    d = b[:, :2].copy().view("<u2").reshape(nb).view(np.float16).astype(np.float64)
    q = b[:, 2:].copy().view(np.int8).astype(np.float64)
    return d, q


def test_one_hot_hidden_exact(oracle_lib):
    inp = synth.probe_inputs(1, 256, seed=1, random_scales=True)
    d, q = _blocks(inp)
    for (b, j) in [(0, 0), (3, 31), (7, 5)]:
        x = np.zeros((1, 256), np.float32)
        x[0, 32 * b + j] = 1.0
        z, _ = oracle.conf_probe(inp["wq"], x, inp["bias"], 0.5)
        assert z[0] == inp["bias"] + d[b] * q[b, j]


def test_all_ones_hidden_exact(oracle_lib):
    inp = synth.probe_inputs(1, 7424, seed=2, random_scales=True)
    d, q = _blocks(inp)
    z, _ = oracle.conf_probe(inp["wq"], np.ones((1, 7424), np.float32), inp["bias"], 0.5)
    expect = inp["bias"] + sum(d[b] * q[b].sum() for b in range(len(d)))
    assert z[0] == pytest.approx(expect, rel=1e-15, abs=1e-15)


@pytest.mark.parametrize("seed,K,t", [(3, 64, 0.5), (4, 128, 0.8), (5, 256, 0.3)])
def test_brute_force_rational(oracle_lib, seed, K, t):
    inp = synth.probe_inputs(6, K, seed=seed, scale=0.05, random_scales=True, threshold=t)
    z, gate = oracle.conf_probe(inp["wq"], inp["hidden"], inp["bias"], t)
    zs, gates = brute.conf_probe(inp["wq"], inp["hidden"], inp["bias"], t)
    for p in range(6):
        assert z[p] == pytest.approx(float(zs[p]), rel=1e-14, abs=1e-14)
        if abs(float(zs[p]) - math.log(t / (1 - t))) > 1e-9:
            assert gate[p] == gates[p]


def test_half_threshold_is_sign(oracle_lib):
    inp = synth.probe_inputs(64, 7424, seed=6)
    z, gate = oracle.conf_probe(inp["wq"], inp["hidden"], inp["bias"], 0.5)
    np.testing.assert_array_equal(gate, (z >= 0).astype(np.int32))
    assert 0 < gate.sum() < 64


def test_sigmoid_gate_other_threshold(oracle_lib):
    inp = synth.probe_inputs(64, 7424, seed=7)
    z, gate = oracle.conf_probe(inp["wq"], inp["hidden"], inp["bias"], 0.9)
    sig = 1.0 / (1.0 + np.exp(-z))
    far = np.abs(z - math.log(9.0)) > 1e-9
    np.testing.assert_array_equal(gate[far], (sig[far] >= 0.9).astype(np.int32))


def test_sign_flip_flips_gate(oracle_lib):
    inp = synth.probe_inputs(32, 7424, seed=8)
    z, gate = oracle.conf_probe(inp["wq"], inp["hidden"], inp["bias"], 0.5)
    z2, gate2 = oracle.conf_probe(inp["wq"], -inp["hidden"], -inp["bias"], 0.5)
    np.testing.assert_allclose(z2, -z, rtol=0, atol=1e-12)
    nz = np.abs(z) > 1e-9
    np.testing.assert_array_equal(gate2[nz], 1 - gate[nz])


def test_rejects_bad_threshold(oracle_lib):
    inp = synth.probe_inputs(1, 64, seed=9)
    for t in (0.0, 1.0, -0.5):
        with pytest.raises(ValueError):
            oracle.conf_probe(inp["wq"], inp["hidden"], inp["bias"], t)
