"""Pins of the weight-stationary matvec oracle (Y = X W^T from fp16)."""
import numpy as np
import pytest

import oracle
from oracle import brute
from dspark_draft_sampling_gb300 import synth


@pytest.mark.parametrize("M,N,K,seed", [(3, 5, 16, 0), (7, 4, 24, 1), (1, 9, 8, 2)])
def test_brute_force_exact(oracle_lib, M, N, K, seed):
    inp = synth.ws_inputs(M, N, K, seed=seed, w_sd=1.0)
    Y, _ = oracle.ws_matvec(inp["W"], inp["X"])
    exact = brute.ws_matvec(inp["W"], inp["X"])
    for m in range(M):
        for n in range(N):
            assert Y[m, n] == float(exact[m][n])  # the fp64 sum is exact at these sizes


def test_m1_is_plain_gemv(oracle_lib):
    inp = synth.ws_inputs(1, 64, 512, seed=3)
    Y, _ = oracle.ws_matvec(inp["W"], inp["X"])
    Wf = inp["W"].view(np.float16).astype(np.float64)
    xf = inp["X"].view(np.float16).astype(np.float64)[0]
    np.testing.assert_allclose(Y[0], Wf @ xf, rtol=1e-12, atol=1e-12)


def test_identity_weight_returns_x(oracle_lib):
    K = 64
    W = synth.f32_to_f16_bits(np.eye(K, dtype=np.float32))
    X = synth.ws_inputs(5, K, K, seed=4)["X"]
    Y, Y16 = oracle.ws_matvec(W, X)
    np.testing.assert_array_equal(Y, X.view(np.float16).astype(np.float64))
    np.testing.assert_array_equal(Y16, X)


def test_rows_independent_of_m(oracle_lib):
    inp = synth.ws_inputs(6, 32, 256, seed=5)
    Y, _ = oracle.ws_matvec(inp["W"], inp["X"])
    for m in range(6):
        Ym, _ = oracle.ws_matvec(inp["W"], inp["X"][m:m + 1])
        np.testing.assert_array_equal(Ym[0], Y[m])


def test_orientation(oracle_lib):
    """W is [N, K] (out x in): a W with one nonzero column k0 picks X[:, k0]."""
    N, K = 6, 16
    Wf = np.zeros((N, K), np.float32)
    Wf[:, 5] = np.arange(1, N + 1)
    X = synth.ws_inputs(3, N, K, seed=6)["X"]
    Y, _ = oracle.ws_matvec(synth.f32_to_f16_bits(Wf), X)
    xk = X.view(np.float16).astype(np.float64)[:, 5]
    np.testing.assert_array_equal(Y, xk[:, None] * np.arange(1, N + 1)[None, :])


def test_fp16_output_is_rne_of_exact(oracle_lib):
    inp = synth.ws_inputs(4, 16, 64, seed=7)
    Y, Y16 = oracle.ws_matvec(inp["W"], inp["X"])
    np.testing.assert_array_equal(Y16, Y.astype(np.float16).view(np.uint16))


@pytest.mark.parametrize("M,N,K,seed", [(2, 3, 64, 0), (3, 2, 96, 1)])
def test_q8_brute_force(oracle_lib, M, N, K, seed):
    inp = synth.ws_q8_inputs(M, N, K, seed=seed, d_sd=0.05)
    Y = oracle.ws_matvec_q8(inp["Wq8"], inp["X"])
    exact = brute.ws_matvec_q8(inp["Wq8"], inp["X"], N, K)
    for m in range(M):
        for n in range(N):
            assert Y[m, n] == pytest.approx(float(exact[m][n]), rel=1e-13, abs=1e-13)


def test_q8_reduces_to_fp16_matvec(oracle_lib):
    """With power-of-two scales every d*q is an fp16 number, so the quantized matvec must
    equal the fp16 matvec of the dequantized weight exactly."""
    M, N, K = 5, 40, 256
    inp = synth.ws_q8_inputs(M, N, K, seed=2, power_of_two_scales=True)
    blk = inp["Wq8"].reshape(N, K // 32, 34)
    d = blk[:, :, :2].copy().view("<u2").reshape(N, K // 32).view(np.float16).astype(np.float64)
    q = blk[:, :, 2:].copy().view(np.int8).astype(np.float64)
    Wd = (d[:, :, None] * q).reshape(N, K)
    W16 = Wd.astype(np.float16)
    assert np.array_equal(W16.astype(np.float64), Wd)
    Yq = oracle.ws_matvec_q8(inp["Wq8"], inp["X"])
    Yf, _ = oracle.ws_matvec(W16.view(np.uint16), inp["X"])
    np.testing.assert_array_equal(Yq, Yf)


def test_q8_one_hot_activation(oracle_lib):
    M, N, K = 1, 6, 128
    inp = synth.ws_q8_inputs(M, N, K, seed=3)
    X = np.zeros((1, K), np.float32)
    X[0, 70] = 1.0
    Y = oracle.ws_matvec_q8(inp["Wq8"], synth.f32_to_f16_bits(X))
    blk = inp["Wq8"].reshape(N, K // 32, 34)
    d = blk[:, 2, :2].copy().view("<u2").reshape(N).view(np.float16).astype(np.float64)
    q = blk[:, 2, 2 + 6].view(np.int8).astype(np.float64)
    np.testing.assert_array_equal(Y[0], d * q)
