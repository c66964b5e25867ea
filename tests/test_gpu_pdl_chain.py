"""Kernels launched back to back with programmatic dependent launch must still see their
predecessor's writes: each chain below feeds one call's output into the next call on the
same stream, and must give bit-identical results to the same calls separated by a full
device synchronization."""
import numpy as np
import pytest
import torch

from dspark_draft_sampling_gb300 import api, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(dspark_lib):
    return dspark_lib


def _f16(a):
    return torch.from_numpy(a.view(np.int16)).cuda().view(torch.float16)


def _ws_pair(N1, K1, N2, seed):
    a = synth.ws_inputs(7, N1, K1, seed=seed)
    b = synth.ws_inputs(7, N2, N1, seed=seed + 1)
    return _f16(a["W"]), _f16(a["X"]), _f16(b["W"])


def test_fp16_matvec_chain():
    W1, X, W2 = _ws_pair(4096, 4096, 1024, seed=1)
    ws1 = api.new_ws_workspace(7, 4096, 4096)
    ws2 = api.new_ws_workspace(7, 1024, 4096)
    y1 = torch.empty((7, 4096), dtype=torch.float16, device="cuda")
    y2 = torch.empty((7, 1024), dtype=torch.float32, device="cuda")
    api.ws_matvec(W1, X, out=y1, workspace=ws1)
    torch.cuda.synchronize()
    api.ws_matvec(W2, y1, out=y2, workspace=ws2)
    torch.cuda.synchronize()
    ref = y2.clone()
    for _ in range(5):
        y1.zero_()
        y2.zero_()
        torch.cuda.synchronize()
        api.ws_matvec(W1, X, out=y1, workspace=ws1)
        api.ws_matvec(W2, y1, out=y2, workspace=ws2)  # consumes y1 with no host sync
        torch.cuda.synchronize()
        assert torch.equal(y2.view(torch.int32), ref.view(torch.int32))


def test_q8_then_fp16_chain():
    inp = synth.ws_q8_inputs(7, 4096, 4096, seed=3)
    q, d = api.q8_0_repack(torch.from_numpy(inp["Wq8"]).cuda(), 4096, 4096)
    X = _f16(inp["X"])
    W2 = _f16(synth.ws_inputs(7, 2048, 4096, seed=4)["W"])
    y1 = torch.empty((7, 4096), dtype=torch.float16, device="cuda")
    y2 = torch.empty((7, 2048), dtype=torch.float32, device="cuda")
    wsq = api.new_ws_q8_workspace(7, 4096, 4096)
    ws2 = api.new_ws_workspace(7, 2048, 4096)
    api.ws_matvec_q8(q, d, X, out=y1, workspace=wsq)
    torch.cuda.synchronize()
    api.ws_matvec(W2, y1, out=y2, workspace=ws2)
    torch.cuda.synchronize()
    ref = y2.clone()
    for _ in range(5):
        y1.zero_()
        y2.zero_()
        torch.cuda.synchronize()
        api.ws_matvec_q8(q, d, X, out=y1, workspace=wsq)
        api.ws_matvec(W2, y1, out=y2, workspace=ws2)
        torch.cuda.synchronize()
        assert torch.equal(y2.view(torch.int32), ref.view(torch.int32))


def test_matvec_then_probe_chain():
    """The probe reads a hidden vector the matvec has just written (fp32, 7424 wide)."""
    K = synth.PROBE_K
    a = synth.ws_inputs(1, K, 4096, seed=5)
    W, X = _f16(a["W"]), _f16(a["X"])
    pr = synth.probe_inputs(1, K, seed=6)
    wq = torch.from_numpy(pr["wq"]).cuda()
    hid = torch.empty((1, K), dtype=torch.float32, device="cuda")
    ws = api.new_ws_workspace(1, K, 4096)
    z = torch.empty(1, dtype=torch.float32, device="cuda")
    g = torch.empty(1, dtype=torch.int32, device="cuda")
    api.ws_matvec(W, X, out=hid, workspace=ws)
    torch.cuda.synchronize()
    api.conf_probe(wq, hid, pr["bias"], 0.5, logit_out=z, gate_out=g)
    torch.cuda.synchronize()
    zref, gref = z.clone(), g.clone()
    for _ in range(5):
        hid.zero_()
        z.zero_()
        torch.cuda.synchronize()
        api.ws_matvec(W, X, out=hid, workspace=ws)
        api.conf_probe(wq, hid, pr["bias"], 0.5, logit_out=z, gate_out=g)
        torch.cuda.synchronize()
        assert torch.equal(z.view(torch.int32), zref.view(torch.int32))
        assert torch.equal(g, gref)
