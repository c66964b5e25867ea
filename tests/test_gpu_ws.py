"""GPU weight-stationary matvec vs the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

from dspark_draft_sampling_gb300 import api, synth
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(dspark_lib):
    return dspark_lib


def _dev(inp):
    W = torch.from_numpy(inp["W"].view(np.int16)).cuda().view(torch.float16)
    X = torch.from_numpy(inp["X"].view(np.int16)).cuda().view(torch.float16)
    return W, X


def _run(inp):
    W, X = _dev(inp)
    y32 = api.ws_matvec(W, X, out_fp32=True)
    y16 = api.ws_matvec(W, X)
    torch.cuda.synchronize()
    return y32.cpu().numpy(), y16.cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("K,N", synth.WS_SHAPES)
def test_qwen3_8b_projection_shapes(K, N):
    inp = synth.ws_inputs(7, N, K, seed=K + N)
    y32, y16 = _run(inp)
    parity.check_ws(inp, y32=y32, y16=y16)


@pytest.mark.parametrize("K,N", synth.WS_SHAPES)
def test_exact_inputs_fp16_is_the_oracles_rne(K, N):
    """Inputs whose every partial sum is exact in fp32: any correct accumulation order gives
    Y itself, so the fp32 output must equal the oracle's Y and the fp16 output the oracle's
    RNE(Y), bit for bit -- including values exactly halfway between two fp16 numbers."""
    inp = synth.ws_exact_inputs(7, N, K, seed=K + N)
    y32, y16 = _run(inp)
    rep = parity.check_ws(inp, y32=y32, y16=y16, exact=True)
    Y, Y16 = parity.oracle.ws_matvec(inp["W"], inp["X"])
    h = Y16.view(np.float16).astype(np.float64)
    up = np.nextafter(Y16.view(np.float16), np.float16(np.inf)).astype(np.float64)
    n_rounded = int((h != Y).sum())
    n_ties = int((np.abs(Y - h) == (up - h) / 2).sum())
    print(f"{K}x{N}: {rep['fp16_total']} outputs, {n_rounded} rounded, {n_ties} exact ties")
    assert n_rounded > rep["fp16_total"] // 4 and n_ties > 0


@pytest.mark.parametrize("M,N,K", [(1, 1, 8), (2, 100, 64), (3, 1000, 2056), (5, 153, 4104),
                                   (8, 4096, 512), (9, 300, 1024), (16, 777, 4096), (7, 1, 12288),
                                   (4, 5000, 8)])
def test_ragged_shapes(M, N, K):
    inp = synth.ws_inputs(M, N, K, seed=M * 7 + N)
    y32, y16 = _run(inp)
    parity.check_ws(inp, y32=y32, y16=y16)


def test_rows_independent_of_m_bitwise():
    inp = synth.ws_inputs(16, 1000, 4096, seed=3)
    W, X = _dev(inp)
    full = api.ws_matvec(W, X, out_fp32=True)
    for M in (1, 2, 3, 7, 9):
        part = api.ws_matvec(W, X[:M].contiguous(), out_fp32=True)
        torch.cuda.synchronize()
        assert torch.equal(part.view(torch.int32), full[:M].view(torch.int32)), M
    for m in (0, 5, 15):
        one = api.ws_matvec(W, X[m:m + 1].contiguous(), out_fp32=True)
        assert torch.equal(one[0].view(torch.int32), full[m].view(torch.int32))


def test_close_to_cublas():
    inp = synth.ws_inputs(7, 4096, 4096, seed=4)
    W, X = _dev(inp)
    y = api.ws_matvec(W, X, out_fp32=True)
    ref = torch.matmul(X.float(), W.float().t())
    assert torch.allclose(y, ref, rtol=1e-3, atol=2e-3)


def test_repeat_bit_identical():
    inp = synth.ws_inputs(7, 12288, 4096, seed=5)
    W, X = _dev(inp)
    a = api.ws_matvec(W, X, out_fp32=True)
    b = api.ws_matvec(W, X, out_fp32=True)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_workspace_shared_across_shapes():
    """One zero-filled workspace serves calls of different shapes in any order (it holds only
    the status word; split-K partials are reduced in distributed shared memory)."""
    shapes = [(7, 1024, 4096), (7, 4096, 4096), (3, 12288, 4096), (7, 4096, 12288)]
    size = max(api.ws_matvec_workspace_bytes(*s) for s in shapes)
    ws = torch.zeros(size, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        for (M, N, K) in shapes:
            inp = synth.ws_inputs(M, N, K, seed=N + K)
            W, X = _dev(inp)
            y = api.ws_matvec(W, X, out_fp32=True, workspace=ws)
            ref = api.ws_matvec(W, X, out_fp32=True)  # its own fresh workspace
            torch.cuda.synchronize()
            assert torch.equal(y.view(torch.int32), ref.view(torch.int32)), (M, N, K)


def test_workspace_status_reports_a_wait_that_gave_up():
    """Failure detection without a fault: the debug launch makes the epilogue wait 2 ms on a
    barrier nothing signals; the kernel records a timeout in the workspace status word and
    returns.  The status is read once, then cleared, and the context stays usable."""
    inp = synth.ws_inputs(7, 1024, 4096, seed=11)
    W, X = _dev(inp)
    ws = api.new_ws_workspace(7, 1024, 4096)
    y = torch.empty((7, 1024), dtype=torch.float32, device="cuda")
    lib = api.load_library()
    st = lib.dspark_ws_matvec_debug(api._ptr(W, "W"), api._ptr(X, "X"), api._ptr(y, "y"), 1, 7, 1024, 4096,
                                    api._ptr(ws, "ws"), ws.numel(), 2000, api._stream(None))
    assert st == 0
    assert api.ws_matvec_status(ws) == api.DSPARK_ERR_TIMEOUT
    assert "timed out" in lib.dspark_last_error().decode()
    assert api.ws_matvec_status(ws) == 0  # reported once
    y2 = api.ws_matvec(W, X, out_fp32=True, workspace=ws)
    assert api.ws_matvec_status(ws) == 0
    parity.check_ws(inp, y32=y2.cpu().numpy())
    assert int(ws[:256].count_nonzero()) == 0


def _problems(shapes, seed, fp32):
    probs, inps = [], []
    for i, (M, N, K) in enumerate(shapes):
        inp = synth.ws_inputs(M, N, K, seed=seed + i)
        W, X = _dev(inp)
        Y = torch.empty((M, N), dtype=torch.float32 if fp32 else torch.float16, device="cuda")
        probs.append((W, X, Y))
        inps.append(inp)
    return probs, inps


@pytest.mark.parametrize("shapes", [
    [(7, N, K) for (K, N) in synth.WS_SHAPES],
    [(3, 100, 64), (16, 777, 4096), (1, 1, 8), (9, 4099, 2056), (7, 12288, 4096)],
])
def test_grouped_matches_separate_calls_bitwise(shapes):
    for fp32 in (True, False):
        probs, inps = _problems(shapes, seed=50, fp32=fp32)
        api.ws_matvec_grouped(probs)
        torch.cuda.synchronize()
        for (W, X, Y), inp in zip(probs, inps):
            ref = api.ws_matvec(W, X, out_fp32=fp32)
            torch.cuda.synchronize()
            view = torch.int32 if fp32 else torch.int16
            assert torch.equal(Y.view(view), ref.view(view))
            if fp32:
                parity.check_ws(inp, y32=Y.cpu().numpy())


def test_grouped_workspace_reuse_and_empty_problems():
    shapes = [(7, N, K) for (K, N) in synth.WS_SHAPES]
    probs, inps = _problems(shapes, seed=60, fp32=True)
    empty = (probs[0][0], probs[0][1][:0], torch.empty((0, probs[0][0].shape[0]), dtype=torch.float32, device="cuda"))
    group = probs[:2] + [empty] + probs[2:]
    ws = torch.zeros(api.ws_matvec_grouped_workspace_bytes(group), dtype=torch.uint8, device="cuda")
    for _ in range(3):
        for (_, _, Y) in probs:
            Y.zero_()
        api.ws_matvec_grouped(group, workspace=ws)
        torch.cuda.synchronize()
        for (W, X, Y), inp in zip(probs, inps):
            parity.check_ws(inp, y32=Y.cpu().numpy())
    assert api.ws_matvec_status(ws) == 0
    assert int(ws[:256].count_nonzero()) == 0
