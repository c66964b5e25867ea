"""GPU quantized (Q8_0) weight-stationary matvec and its repack vs the fp64 oracle."""
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
    raw = torch.from_numpy(inp["Wq8"]).cuda()
    q, d = api.q8_0_repack(raw, inp["N"], inp["K"])
    X = torch.from_numpy(inp["X"].view(np.int16)).cuda().view(torch.float16)
    return q, d, X


def _run(inp):
    q, d, X = _dev(inp)
    y32 = api.ws_matvec_q8(q, d, X, out_fp32=True)
    y16 = api.ws_matvec_q8(q, d, X)
    torch.cuda.synchronize()
    return y32.cpu().numpy(), y16.cpu().view(torch.int16).numpy().view(np.uint16)


def test_repack_is_a_byte_exact_split():
    N, K = 37, 1024
    inp = synth.ws_q8_inputs(3, N, K, seed=1)
    q, d, _ = _dev(inp)
    blk = inp["Wq8"].reshape(N, K // 32, 34)
    np.testing.assert_array_equal(q.cpu().numpy(), blk[:, :, 2:].view(np.int8).reshape(N, K))
    np.testing.assert_array_equal(d.cpu().numpy().view(np.uint16),
                                  blk[:, :, :2].copy().view("<u2").reshape(N, K // 32))


@pytest.mark.parametrize("K,N", synth.WS_SHAPES)
def test_qwen3_8b_projection_shapes(K, N):
    inp = synth.ws_q8_inputs(7, N, K, seed=K + N)
    y32, y16 = _run(inp)
    parity.check_ws_q8(inp, y32=y32, y16=y16)


@pytest.mark.parametrize("M,N,K", [(1, 1, 256), (2, 100, 512), (3, 1000, 2304), (5, 153, 4352),
                                   (8, 4096, 256), (9, 300, 1024), (16, 777, 4096), (7, 1, 12288),
                                   (4, 5000, 256), (6, 151, 6400)])
def test_ragged_shapes(M, N, K):
    inp = synth.ws_q8_inputs(M, N, K, seed=M * 7 + N)
    y32, y16 = _run(inp)
    parity.check_ws_q8(inp, y32=y32, y16=y16)


def test_extreme_scales_and_codes():
    """Largest fp16 scales next to subnormal ones, codes at +-127 and 0: the dequantized
    weights must come out exactly (no overflow, no flush of subnormal scales)."""
    M, N, K = 3, 64, 512
    inp = synth.ws_q8_inputs(M, N, K, seed=9)
    blk = inp["Wq8"].reshape(N, K // 32, 34)
    d = np.abs(np.random.default_rng(9).standard_normal((N, K // 32))).astype(np.float32)
    d[0::4] = 60000.0
    d[1::4] = np.float32(2.0 ** -24) * 3.0
    d[2::4] = 1.0
    blk[:, :, 0:2] = synth.f32_to_f16_bits(d).astype("<u2").view(np.uint8).reshape(N, K // 32, 2)
    blk[:, 0, 2:] = np.uint8(127)
    blk[:, 1, 2:] = np.int8(-127).view(np.uint8)
    blk[:, 2, 2:] = 0
    inp["Wq8"] = blk.reshape(-1).copy()
    x = np.zeros((M, K), np.float32)
    x[:, 0:96] = np.random.default_rng(10).standard_normal((M, 96)).astype(np.float32) * 1e-3
    inp["X"] = synth.f32_to_f16_bits(x)
    y32, _ = _run(inp)
    parity.check_ws_q8(inp, y32=y32)


def test_rows_independent_of_m_bitwise():
    inp = synth.ws_q8_inputs(16, 1000, 4096, seed=3)
    q, d, X = _dev(inp)
    full = api.ws_matvec_q8(q, d, X, out_fp32=True)
    for M in (1, 2, 3, 7, 8, 9):
        part = api.ws_matvec_q8(q, d, X[:M].contiguous(), out_fp32=True)
        torch.cuda.synchronize()
        assert torch.equal(part.view(torch.int32), full[:M].view(torch.int32)), M


def test_repeat_is_bit_identical():
    inp = synth.ws_q8_inputs(7, 4096, 4096, seed=4)
    q, d, X = _dev(inp)
    a = api.ws_matvec_q8(q, d, X, out_fp32=True)
    b = api.ws_matvec_q8(q, d, X, out_fp32=True)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_close_to_dequantized_torch_reference():
    """Plain PyTorch fp32 reference of the same op: dequantize, then matmul."""
    inp = synth.ws_q8_inputs(7, 2048, 4096, seed=5)
    q, d, X = _dev(inp)
    y = api.ws_matvec_q8(q, d, X, out_fp32=True)
    W = (q.float().view(2048, 128, 32) * d.view(torch.float16).float()[:, :, None]).view(2048, 4096)
    ref = X.float() @ W.t()
    torch.cuda.synchronize()
    assert torch.allclose(y, ref, atol=2e-3, rtol=1e-3)


def test_shared_workspace_across_shapes_and_repeats():
    """One zero-filled workspace serves every shape in turn: each call leaves it zero-filled."""
    shapes = [(7, 4096, 4096), (7, 1024, 4096), (3, 300, 12288), (7, 4096, 4096)]
    nbytes = max(api.ws_matvec_q8_workspace_bytes(M, N, K) for M, N, K in shapes)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    for i, (M, N, K) in enumerate(shapes):
        inp = synth.ws_q8_inputs(M, N, K, seed=20 + i)
        q, d, X = _dev(inp)
        for _ in range(2):
            y = api.ws_matvec_q8(q, d, X, out_fp32=True, workspace=ws)
            torch.cuda.synchronize()
            parity.check_ws_q8(inp, y32=y.cpu().numpy())
    assert int(ws[:256].count_nonzero()) == 0


def test_workspace_status_reports_a_wait_that_gave_up():
    """As for the fp16 matvec: a debug launch whose epilogue first waits 2 ms on a barrier
    nothing signals records a timeout, reports it once and leaves the context usable."""
    inp = synth.ws_q8_inputs(7, 1024, 4096, seed=12)
    q, d, X = _dev(inp)
    ws = api.new_ws_q8_workspace(7, 1024, 4096)
    y = torch.empty((7, 1024), dtype=torch.float32, device="cuda")
    lib = api.load_library()
    st = lib.dspark_ws_matvec_q8_debug(api._ptr(q, "q"), api._ptr(d, "d"), api._ptr(X, "X"), api._ptr(y, "y"), 1,
                                       7, 1024, 4096, api._ptr(ws, "ws"), ws.numel(), 2000, api._stream(None))
    assert st == 0
    assert api.ws_matvec_status(ws) == api.DSPARK_ERR_TIMEOUT
    assert api.ws_matvec_status(ws) == 0
    y2 = api.ws_matvec_q8(q, d, X, out_fp32=True, workspace=ws)
    assert api.ws_matvec_status(ws) == 0
    parity.check_ws_q8(inp, y32=y2.cpu().numpy())


def _grouped(inps, fp32_flags):
    devs = [_dev(inp) for inp in inps]
    outs = [torch.empty((inp["M"], inp["N"]), dtype=torch.float32 if f else torch.float16, device="cuda")
            for inp, f in zip(inps, fp32_flags)]
    api.ws_matvec_q8_grouped([(q, d, X, Y) for (q, d, X), Y in zip(devs, outs)])
    torch.cuda.synchronize()
    return [Y.cpu().numpy() if Y.dtype == torch.float32 else Y.cpu().view(torch.int16).numpy().view(np.uint16)
            for Y in outs]


def test_grouped_qwen3_8b_shapes():
    """The four projections in one launch (stream-K over all their row blocks), within
    tolerance of the oracle, the fp16 outputs the rounding of the fp32 ones."""
    inps = [synth.ws_q8_inputs(7, N, K, seed=K + N) for (K, N) in synth.WS_SHAPES]
    g32 = _grouped(inps, [True] * 4)
    g16 = _grouped(inps, [False] * 4)
    for inp, a32, a16 in zip(inps, g32, g16):
        parity.check_ws_q8(inp, y32=a32, y16=a16)


@pytest.mark.parametrize("shapes", [
    [(1, 40000, 512), (16, 300, 2304), (3, 1, 256)],                  # one problem wider than the SMs
    [(7, 1000, 4096), (2, 153, 12288), (9, 5000, 256), (4, 64, 1024)],  # row blocks of 1 .. 48 superblocks
    [(5, 777, 6400), (8, 128, 768)],                                    # 178 superblocks
    [(3, 300, 512), (2, 200, 256)],                                     # 8 superblocks: 8 CTAs
    [(2, 128, 16384), (1, 128, 256)],                                   # one row block over 64 CTAs
])
def test_grouped_ragged_mixed(shapes):
    inps = [synth.ws_q8_inputs(M, N, K, seed=M + N + K) for (M, N, K) in shapes]
    flags = [i % 2 == 0 for i in range(len(inps))]
    outs = _grouped(inps, flags)
    for inp, f, y in zip(inps, flags, outs):
        if f:
            parity.check_ws_q8(inp, y32=y)
        else:
            parity.check_ws_q8(inp, y16=y)


def test_grouped_skips_empty_problems_and_repeats_bitwise():
    inps = [synth.ws_q8_inputs(3, 500, 1024, seed=5), synth.ws_q8_inputs(6, 2048, 2048, seed=6)]
    a = _grouped(inps, [True, True])
    b = _grouped(inps, [True, True])
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x.view(np.uint32), y.view(np.uint32))
    q, d, X = _dev(inps[0])
    Y = torch.full((3, 500), 7.0, device="cuda")
    Ye = torch.full((0, 500), 7.0, device="cuda")
    api.ws_matvec_q8_grouped([(q, d, X, Y), (q, d, X[:0], Ye)])
    torch.cuda.synchronize()
    # one live problem: the plan of a single call, so the bits of dspark_ws_matvec_q8
    y32, _ = _run(inps[0])
    np.testing.assert_array_equal(Y.cpu().numpy().view(np.uint32), y32.view(np.uint32))
    parity.check_ws_q8(inps[0], y32=a[0])


def test_grouped_wait_for_a_withheld_partial_gives_up():
    """Failure detection without a fault: one CTA of the stream-K launch writes its partial
    sums but never sets its flag; the CTA finishing that row block waits 2 ms, gives up,
    leaves the row block's outputs alone and records DSPARK_ERR_TIMEOUT.  Every other output
    is right, and after the workspace is zero-filled again the next launch is whole."""
    from tests.test_streamk_partition import pieces_of, range_begin, superblock_k

    inps = [synth.ws_q8_inputs(7, N, K, seed=K + N) for (K, N) in synth.WS_SHAPES]
    sk = superblock_k()
    problems, total = [], 0
    for inp in inps:
        nrb, nsb = -(-inp["N"] // 128), inp["K"] // sk
        problems.append(dict(nrb=nrb, nsb=nsb, sb_base=total))
        total += nrb * nsb
    G = min(torch.cuda.get_device_properties(0).multi_processor_count, total)
    # a CTA whose range starts inside a row block: its first piece is a later part
    c = next(c for c in range(1, G) if pieces_of(c, problems, total, G)[0][2] > 0)
    p, rb = pieces_of(c, problems, total, G)[0][:2]
    head = max(h for h in range(c) if range_begin(h, total, G) <= problems[p]["sb_base"] + rb * problems[p]["nsb"])

    devs = [_dev(inp) for inp in inps]
    outs = [torch.full((inp["M"], inp["N"]), 7.0, dtype=torch.float32, device="cuda") for inp in inps]
    group = [(q, d, X, Y) for (q, d, X), Y in zip(devs, outs)]
    ws = api.new_ws_q8_grouped_workspace()
    api.ws_matvec_q8_grouped_debug(group, ws, withheld_cta=c, timeout_us=2000)
    assert api.ws_matvec_status(ws) == api.DSPARK_ERR_TIMEOUT
    lo, hi = rb * 128, min((rb + 1) * 128, inps[p]["N"])
    for i, (inp, Y) in enumerate(zip(inps, outs)):
        y = Y.cpu().numpy()
        if i == p:
            assert np.all(y[:, lo:hi] == 7.0), f"row block {rb} of problem {p} (finished by CTA {head}) was written"
            ref = parity.oracle.ws_matvec_q8(inp["Wq8"], inp["X"])
            keep = np.ones(inp["N"], bool)
            keep[lo:hi] = False
            ok, err, nbad = parity.within_tol(y[:, keep], ref[:, keep])
            assert ok, (i, err, nbad)
        else:
            parity.check_ws_q8(inp, y32=y)
    ws.zero_()
    api.ws_matvec_q8_grouped(group, workspace=ws)
    assert api.ws_matvec_status(ws) == 0
    for inp, Y in zip(inps, outs):
        parity.check_ws_q8(inp, y32=Y.cpu().numpy())
