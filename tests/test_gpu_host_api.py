"""Host-buffer forms of the three operations: inputs from and outputs to pinned host memory
give the same bits as the device-pointer forms (and so the same parity with the oracle)."""
import numpy as np
import pytest
import torch

from dspark_draft_sampling_gb300 import api, synth
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(dspark_lib):
    return dspark_lib


def _scratch(nbytes, zero=False):
    return (torch.zeros if zero else torch.empty)(nbytes, dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("lane", ["reduced_vocab", "tiny"])
def test_markov_draft_host_matches_device_form(lane):
    inp = synth.markov_config(lane)
    base_h = torch.from_numpy(inp["base"]).pin_memory()
    prev_h = torch.from_numpy(inp["prev0"].copy()).pin_memory()
    B, k, V = inp["base"].shape
    ids_h = torch.empty((B, k), dtype=torch.int64).pin_memory()
    w1 = torch.from_numpy(inp["w1"].view(np.int16)).cuda()
    w2 = torch.from_numpy(inp["w2"].view(np.int16)).cuda()
    d2t = None if inp["d2t"] is None else torch.from_numpy(inp["d2t"]).cuda()
    scratch = _scratch(api.markov_draft_host_scratch_bytes(B, k, V, inp["rank"]))
    api.markov_draft_host(base_h, w1, w2, d2t, prev_h, ids_h, scratch)
    torch.cuda.synchronize()
    prev_d = torch.from_numpy(inp["prev0"].copy()).cuda()
    ids_d = api.markov_draft(torch.from_numpy(inp["base"]).cuda(), w1, w2, d2t, prev_d)
    torch.cuda.synchronize()
    assert torch.equal(ids_h, ids_d.cpu())
    assert torch.equal(prev_h, prev_d.cpu())


def test_conf_probe_host_matches_device_form():
    inp = synth.probe_inputs(64, 7424, seed=3, random_scales=True, scale=0.01)
    wq = torch.from_numpy(inp["wq"]).cuda()
    hid_h = torch.from_numpy(inp["hidden"]).pin_memory()
    gate_h = torch.empty(64, dtype=torch.int32).pin_memory()
    z_h = torch.empty(64, dtype=torch.float32).pin_memory()
    scratch = _scratch(api.conf_probe_host_scratch_bytes(7424, 64))
    api.conf_probe_host(wq, hid_h, inp["bias"], inp["threshold"], gate_h, scratch, logit_h=z_h)
    torch.cuda.synchronize()
    z_d, g_d = api.conf_probe(wq, hid_h.cuda(), inp["bias"], inp["threshold"])
    torch.cuda.synchronize()
    assert torch.equal(z_h.view(torch.int32), z_d.cpu().view(torch.int32))
    assert torch.equal(gate_h, g_d.cpu())
    parity.check_probe(inp, z_h.numpy(), gate_h.numpy())


def test_ws_matvec_host_matches_device_form_and_shares_scratch():
    shapes = [(7, 4096, 4096), (7, 1024, 4096), (3, 300, 12288)]
    nbytes = max(api.ws_matvec_host_scratch_bytes(M, N, K) for M, N, K in shapes)
    scratch = _scratch(nbytes, zero=True)
    for i, (M, N, K) in enumerate(shapes):
        inp = synth.ws_inputs(M, N, K, seed=30 + i)
        W = torch.from_numpy(inp["W"].view(np.int16)).cuda().view(torch.float16)
        X_h = torch.from_numpy(inp["X"].view(np.int16)).view(torch.float16).pin_memory()
        for dt in (torch.float32, torch.float16):
            Y_h = torch.empty((M, N), dtype=dt).pin_memory()
            api.ws_matvec_host(W, X_h, Y_h, scratch)
            torch.cuda.synchronize()
            Y_d = api.ws_matvec(W, X_h.cuda(), out_fp32=dt == torch.float32)
            torch.cuda.synchronize()
            assert torch.equal(Y_h.view(torch.int16 if dt == torch.float16 else torch.int32),
                               Y_d.cpu().view(torch.int16 if dt == torch.float16 else torch.int32))
    assert int(scratch[:256].count_nonzero()) == 0


def test_inputs_copied_event_orders_another_stream():
    """The optional event is recorded after the input copies: a second stream waiting on it
    starts only then (a never-recorded torch event is created by the binding first)."""
    inp = synth.markov_config("tiny")
    B, k, V = inp["base"].shape
    base_h = torch.from_numpy(inp["base"]).pin_memory()
    prev_h = torch.from_numpy(inp["prev0"].copy()).pin_memory()
    ids_h = torch.empty((B, k), dtype=torch.int64).pin_memory()
    w1 = torch.from_numpy(inp["w1"].view(np.int16)).cuda()
    w2 = torch.from_numpy(inp["w2"].view(np.int16)).cuda()
    scratch = _scratch(api.markov_draft_host_scratch_bytes(B, k, V, inp["rank"]))
    ev = torch.cuda.Event()
    assert not ev.cuda_event
    api.markov_draft_host(base_h, w1, w2, None, prev_h, ids_h, scratch, inputs_copied=ev)
    assert ev.cuda_event
    other = torch.cuda.Stream()
    other.wait_event(ev)
    marker = torch.zeros(1, device="cuda")
    with torch.cuda.stream(other):
        marker += 1
    torch.cuda.synchronize()
    assert ev.query() and float(marker.item()) == 1.0


def test_ws_matvec_grouped_host_matches_grouped_device_form():
    shapes = [(7, N, K) for (K, N) in synth.WS_SHAPES] + [(3, 300, 12288)]
    host_probs, dev_probs = [], []
    for i, (M, N, K) in enumerate(shapes):
        inp = synth.ws_inputs(M, N, K, seed=80 + i)
        W = torch.from_numpy(inp["W"].view(np.int16)).cuda().view(torch.float16)
        X_h = torch.from_numpy(inp["X"].view(np.int16)).view(torch.float16).pin_memory()
        dt = torch.float32 if i % 2 else torch.float16
        host_probs.append((W, X_h, torch.empty((M, N), dtype=dt).pin_memory()))
        dev_probs.append((W, X_h.cuda(), torch.empty((M, N), dtype=dt, device="cuda")))
    scratch = _scratch(api.ws_matvec_grouped_host_scratch_bytes(host_probs), zero=True)
    for _ in range(2):
        api.ws_matvec_grouped_host(host_probs, scratch)
        api.ws_matvec_grouped(dev_probs)
        torch.cuda.synchronize()
        for (_, _, Yh), (_, _, Yd) in zip(host_probs, dev_probs):
            v = torch.int32 if Yh.dtype == torch.float32 else torch.int16
            assert torch.equal(Yh.view(v), Yd.cpu().view(v))
    assert api.ws_matvec_status(scratch) == 0
    assert int(scratch[:256].count_nonzero()) == 0
