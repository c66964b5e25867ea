"""Device-side base logits: lm_head matvec -> Markov draft in one CUDA graph, vs the oracle."""
import numpy as np
import pytest
import torch

from dspark_draft_sampling_gb300 import api, synth
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(dspark_lib):
    return dspark_lib


@pytest.mark.parametrize("B,k,V,H,R,d2t", [(1, 9, 32000, 2048, 256, "injective"),
                                           (2, 7, 20000, 1024, 128, "identity"),
                                           (1, 15, 248320, 512, 256, "identity")])
def test_lm_head_then_markov(B, k, V, H, R, d2t):
    head = synth.ws_inputs(B * k, V, H, seed=V + H)           # W = lm_head, X = draft hidden states
    mk = synth.markov_inputs(B, k, V, R, d2t=d2t, w_sd=0.2, seed=B * 10 + k)
    dev = "cuda"
    lm_head = torch.from_numpy(head["W"].view(np.int16)).to(dev).view(torch.float16)
    hidden = torch.from_numpy(head["X"].view(np.int16)).to(dev).view(torch.float16)
    t = parity.markov_to_device(mk)
    plan = api.DraftPlan(lm_head, hidden, t["w1"], t["w2"], t["d2t"], t["prev"], k)
    plan.launch()
    torch.cuda.synchronize()
    assert api.markov_status(plan.markov_ws) == 0
    base = plan.base.cpu().numpy()
    # (1) the base logits are the lm_head projection of the hidden states
    if V * H * B * k <= 2e9:
        Y, _ = parity.oracle.ws_matvec(head["W"], head["X"])
        ok, err, nbad = parity.within_tol(base.reshape(B * k, V), Y)
        assert ok, f"{nbad} base logits outside tolerance (max err {err:.3e})"
    # (2) the draft ids are the Markov chain on exactly those base logits
    chained = dict(mk)
    chained["base"] = base
    g = dict(out_ids=plan.out_ids.cpu().numpy(), prev=t["prev"].cpu().numpy(), logits=None,
             bias=None, status=0)
    rep = parity.check_markov(chained, g, values=False)
    assert rep["n_exempt"] == 0
    plan.close()


def test_plan_relaunch_continues_from_prev():
    B, k, V, H, R = 1, 4, 8000, 256, 64
    head = synth.ws_inputs(B * k, V, H, seed=3)
    mk = synth.markov_inputs(B, k, V, R, w_sd=0.5, base_sd=0.1, seed=4)
    lm_head = torch.from_numpy(head["W"].view(np.int16)).cuda().view(torch.float16)
    hidden = torch.from_numpy(head["X"].view(np.int16)).cuda().view(torch.float16)
    t = parity.markov_to_device(mk)
    plan = api.DraftPlan(lm_head, hidden, t["w1"], t["w2"], None, t["prev"], k)
    first = plan.launch().clone()
    second = plan.launch().clone()
    torch.cuda.synchronize()
    base = plan.base.cpu().numpy()
    chained = dict(mk)
    chained["base"] = base
    chained["prev0"] = first.cpu().numpy()[:, -1].copy()
    g = dict(out_ids=second.cpu().numpy(), prev=t["prev"].cpu().numpy(), logits=None, bias=None,
             status=0)
    parity.check_markov(chained, g, values=False)
    plan.close()
