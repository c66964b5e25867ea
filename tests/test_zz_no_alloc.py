"""The allocation-free Markov entry point (dspark_markov_draft_noalloc).

Some callers cannot call cudaMalloc or lend device scratch (an engine plugin whose
device memory belongs to the host engine's allocator, or a latency-critical loop where
cudaMalloc's implicit synchronization is not acceptable).  For them the library keeps
the Markov kernel's scratch in a static device array.  This test calls that entry point
through the C ABI twice in a row -- the second call continuing from the prev the first
left on the device -- and checks it against dspark_markov_draft with a workspace.
Draft ids are compared exactly (the same kernel runs on the same inputs).
"""
import ctypes

import numpy as np
import pytest
import torch

from dspark_draft_sampling_gb300 import api, synth
from tests import parity

pytestmark = pytest.mark.gpu


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, t, B, k, V, R, out):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.dspark_markov_draft_noalloc(_p(t["base"]), _p(t["w1"]), _p(t["w2"]), _p(t["d2t"]),
                                         _p(t["prev"]), B, k, V, R, _p(out), stream)
    assert st == 0, lib.dspark_last_error().decode()


@pytest.mark.parametrize("lane,num_reqs", [("reduced_vocab", 1), ("tiny", 1), ("qwen3_8b", 3)])
def test_noalloc_matches_workspace_entry_two_calls(dspark_lib, lane, num_reqs):
    lib = dspark_lib
    inp = synth.markov_config(lane, num_reqs=num_reqs, seed=1)
    B, k, V = inp["base"].shape
    R = inp["w2"].shape[1]
    a = parity.markov_to_device(inp)   # driven through the allocation-free entry point
    b = parity.markov_to_device(inp)   # driven through dspark_markov_draft + workspace
    ws = api.new_markov_workspace(B, k, V, R)
    first = None
    for call in range(2):
        out_a = torch.full((B, k), -7, dtype=torch.int64, device="cuda")
        _noalloc(lib, a, B, k, V, R, out_a)
        out_b = api.markov_draft(b["base"], b["w1"], b["w2"], b["d2t"], b["prev"], workspace=ws)
        torch.cuda.synchronize()
        assert api.markov_status(ws) == 0
        # every position finished: the entry point sets out_ids to -1 before its kernel
        assert (out_a >= 0).all()
        np.testing.assert_array_equal(out_a.cpu().numpy(), out_b.cpu().numpy())
        np.testing.assert_array_equal(a["prev"].cpu().numpy(), b["prev"].cpu().numpy())
        if call == 0:
            first = dict(out_ids=out_a.cpu().numpy(), prev=a["prev"].cpu().numpy(),
                         logits=None, bias=None, status=0)
    # the first call of the pair also matches the oracle directly
    parity.check_markov(inp, first, values=False)


def test_noalloc_at_its_limits(dspark_lib):
    """k = 64 positions (the static scratch's limit) and num_reqs = 8 (the kernel's limit)."""
    lib = dspark_lib
    inp = synth.markov_inputs(8, 64, 5000, 128, base_sd=1.0, w_sd=0.3, d2t="injective", seed=5)
    B, k, V = inp["base"].shape
    a = parity.markov_to_device(inp)
    out = torch.full((B, k), -7, dtype=torch.int64, device="cuda")
    _noalloc(lib, a, B, k, V, 128, out)
    torch.cuda.synchronize()
    assert (out >= 0).all()
    rep = parity.check_markov(inp, dict(out_ids=out.cpu().numpy(), prev=a["prev"].cpu().numpy(), logits=None,
                                        bias=None, status=0), values=False)
    assert rep["n_exempt"] <= 2


def test_noalloc_allocates_no_device_memory(dspark_lib):
    """After a first call (which may load the library's device code), further calls leave the
    device's free memory unchanged: the entry point itself allocates nothing."""
    lib = dspark_lib
    inp = synth.markov_config("tiny", seed=3)
    B, k, V = inp["base"].shape
    R = inp["w2"].shape[1]
    t = parity.markov_to_device(inp)
    out = torch.empty((B, k), dtype=torch.int64, device="cuda")
    _noalloc(lib, t, B, k, V, R, out)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        _noalloc(lib, t, B, k, V, R, out)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert (out >= 0).all()


def test_noalloc_rejects_too_many_positions(dspark_lib):
    lib = dspark_lib
    inp = synth.markov_inputs(1, 65, 64, 64, seed=2)
    t = parity.markov_to_device(inp)
    out = torch.empty((1, 65), dtype=torch.int64, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.dspark_markov_draft_noalloc(_p(t["base"]), _p(t["w1"]), _p(t["w2"]), None,
                                         _p(t["prev"]), 1, 65, 64, 64, _p(out), stream)
    assert st == api.DSPARK_ERR_UNSUPPORTED
    assert "64" in lib.dspark_last_error().decode()
