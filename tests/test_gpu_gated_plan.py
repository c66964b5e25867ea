"""Probe-gated draft: the conditional graph node runs the Markov draft only when the
probe's gate is open, with no host readback in between."""
import numpy as np
import pytest
import torch

from dspark_draft_sampling_gb300 import api, synth
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(dspark_lib):
    return dspark_lib


def _setup(bias):
    mk = synth.markov_config("reduced_vocab", seed=3)
    pr = synth.probe_inputs(1, 7424, seed=5)
    t = parity.markov_to_device(mk)
    wq = torch.from_numpy(pr["wq"]).cuda()
    x = torch.from_numpy(pr["hidden"][0].copy()).cuda()
    plan = api.GatedDraftPlan(wq, x, bias, 0.5, t["base"], t["w1"], t["w2"], t["d2t"], t["prev"])
    plan.out_ids.fill_(-7)
    return mk, pr, t, x, plan


def test_gate_open_runs_the_draft():
    mk, pr, t, x, plan = _setup(bias=50.0)
    plan.launch()
    torch.cuda.synchronize()
    assert int(plan.gate[0]) == 1
    g = dict(out_ids=plan.out_ids.cpu().numpy(), prev=t["prev"].cpu().numpy(), logits=None,
             bias=None, status=api.markov_status(plan.workspace))
    parity.check_markov(mk, g, values=False)
    plan.close()


def test_gate_closed_skips_the_draft():
    mk, pr, t, x, plan = _setup(bias=-50.0)
    plan.launch()
    torch.cuda.synchronize()
    assert int(plan.gate[0]) == 0
    assert torch.all(plan.out_ids == -7)
    np.testing.assert_array_equal(t["prev"].cpu().numpy(), mk["prev0"])
    plan.close()


def test_gate_follows_the_probe_input_between_launches():
    mk, pr, t, x, plan = _setup(bias=0.0)
    z0, g0 = parity.oracle.conf_probe(pr["wq"], pr["hidden"], 0.0, 0.5)
    for flip in (False, True, False):
        x.copy_(torch.from_numpy(-pr["hidden"][0] if flip else pr["hidden"][0]).cuda())
        t["prev"].copy_(torch.from_numpy(mk["prev0"]))
        plan.out_ids.fill_(-7)
        plan.launch()
        torch.cuda.synchronize()
        want = int(g0[0]) if not flip else 1 - int(g0[0])
        assert int(plan.gate[0]) == want
        if want:
            assert torch.all(plan.out_ids >= 0)
        else:
            assert torch.all(plan.out_ids == -7)
    plan.close()
