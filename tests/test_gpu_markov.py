"""GPU Markov block draft vs the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

from dspark_draft_sampling_gb300 import api, synth
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(dspark_lib):
    return dspark_lib


def test_tiny_lane():
    inp = synth.markov_config("tiny")
    rep = parity.check_markov(inp, parity.gpu_markov(inp))
    assert rep["n_exempt"] == 0


def test_reduced_vocab_lane_with_ties():
    inp = synth.markov_config("reduced_vocab")
    g = parity.gpu_markov(inp)
    rep = parity.check_markov(inp, g)
    assert rep["n_exempt"] == 0
    gd = parity.draft_from_target(inp, g["out_ids"])
    for i in inp["spiked_steps"]:
        v1, _ = inp["ties"][(i // 2) % len(inp["ties"])]
        assert gd[0, i] == v1  # lowest index of the planted exact tie


def test_qwen3_8b_lane():
    inp = synth.markov_config("qwen3_8b")
    rep = parity.check_markov(inp, parity.gpu_markov(inp))
    assert rep["n_exempt"] == 0


@pytest.mark.slow
@pytest.mark.parametrize("B", [1, 4, 8])
def test_full_vocab_27b_lane(B):
    inp = synth.markov_config("full_vocab_27b", num_reqs=B)
    g = parity.gpu_markov(inp, dbg=True, dbg_bias=False)
    rep = parity.check_markov(inp, g)
    assert rep["n_exempt"] <= 1


@pytest.mark.slow
@pytest.mark.parametrize("B", [4, 8])
def test_full_vocab_27b_lane_production_kernel(B):
    """The kernel instantiation the benchmark times (no debug outputs) on the full 27B lane:
    ids and the final prev against the oracle, with the near-tie exemption reported."""
    inp = synth.markov_config("full_vocab_27b", num_reqs=B)
    g = parity.gpu_markov(inp, dbg=False)
    rep = parity.check_markov(inp, g, values=False)
    print(f"num_reqs={B}: n_exempt={rep['n_exempt']} {rep['exempt']}")
    assert rep["n_exempt"] <= 1


@pytest.mark.parametrize("B,k,V,R,d2t", [
    (3, 5, 1000, 64, "identity"),
    (5, 3, 777, 128, "injective"),
    (7, 2, 4099, 256, "identity"),
    (2, 1, 100, 256, "identity"),     # fewer rows than CTAs
    (1, 3, 1, 64, "identity"),        # a single vocab row
    (8, 2, 153, 64, "injective"),
    (6, 4, 20000, 256, "injective"),
    (2, 6, 3001, 128, "identity"),
    (1, 9, 60000, 128, "identity"),   # rank 128: 6 tile slots, wrapped many times
    (4, 5, 100000, 64, "injective"),  # rank 64: 12 tile slots
])
def test_ragged_shapes(B, k, V, R, d2t):
    inp = synth.markov_inputs(B, k, V, R, base_sd=1.0, w_sd=0.3, d2t=d2t, seed=B * 100 + k)
    rep = parity.check_markov(inp, parity.gpu_markov(inp))
    assert rep["n_exempt"] == 0


# The single-cluster kernel (vocabularies whose markov_w1 + markov_w2 fit in one cluster's
# shared memory), named explicitly so that each case runs it whatever the auto choice.
@pytest.mark.parametrize("B,k,V,R,d2t", [
    (1, 4, 4096, 64, "identity"),     # the tiny lane's shape
    (3, 5, 1000, 64, "injective"),    # 8 tiles, the last one ragged
    (8, 3, 8192, 64, "identity"),     # 64 tiles, 8 requests
    (2, 6, 2048, 128, "injective"),
    (2, 2, 2048, 256, "identity"),    # rank 256
    (2, 1, 100, 256, "identity"),     # a single CTA
    (7, 9, 508, 64, "identity"),      # 4 tiles, ragged
    (4, 20, 3000, 64, "injective"),   # more positions than base buffers
])
def test_cluster_kernel(B, k, V, R, d2t):
    inp = synth.markov_inputs(B, k, V, R, base_sd=1.0, w_sd=0.3, d2t=d2t, seed=B * 31 + k)
    rep = parity.check_markov(inp, parity.gpu_markov(inp, kernel="cluster"))
    assert rep["n_exempt"] == 0


def test_cluster_kernel_production_form_and_ties():
    """Without debug outputs, with planted exact ties decided by the lowest index."""
    inp = synth.markov_inputs(3, 8, 6000, 64, base_sd=1.0, w_sd=0.3, tie_frac=0.005,
                              d2t="injective", seed=41)
    g = parity.gpu_markov(inp, dbg=False, kernel="cluster")
    rep = parity.check_markov(inp, g, values=False)
    assert rep["n_exempt"] == 0
    gd = parity.draft_from_target(inp, g["out_ids"])
    for i in inp["spiked_steps"]:
        v1, _ = inp["ties"][(i // 2) % len(inp["ties"])]
        assert np.all(gd[:, i] == v1)


def test_tiny_lane_on_both_kernels():
    inp = synth.markov_config("tiny")
    assert api.markov_kernel_for(1, 4, 4096, 64) == "cluster"
    for kernel in ("grid", "cluster"):
        rep = parity.check_markov(inp, parity.gpu_markov(inp, kernel=kernel))
        assert rep["n_exempt"] == 0


@pytest.mark.parametrize("B,k,V,R", [(1, 4, 4096, 64), (6, 5, 3000, 128), (8, 7, 8192, 64),
                                     (2, 3, 2040, 256)])
def test_cluster_and_grid_kernels_bit_identical(B, k, V, R):
    """Both kernels issue the same tensor-core instructions for every bias value, so logits,
    biases and ids agree bit for bit (the automatic choice, which depends on the shared
    memory the exchange needs for num_reqs, cannot change a result)."""
    inp = synth.markov_inputs(B, k, V, R, base_sd=1.0, w_sd=0.3, seed=B + k + R)
    g = parity.gpu_markov(inp, kernel="grid")
    c = parity.gpu_markov(inp, kernel="cluster")
    np.testing.assert_array_equal(g["out_ids"], c["out_ids"])
    np.testing.assert_array_equal(g["prev"], c["prev"])
    np.testing.assert_array_equal(g["logits"].view(np.uint32), c["logits"].view(np.uint32))
    np.testing.assert_array_equal(g["bias"].view(np.uint32), c["bias"].view(np.uint32))


def test_cluster_kernel_choice_and_refusal():
    assert api.markov_kernel_for(1, 9, 32000, 256) == "grid"
    assert api.markov_kernel_for(8, 15, 248320, 256) == "grid"
    assert api.markov_kernel_for(1, 4, 4098, 64) == "grid"  # vocab not a multiple of 4
    inp = synth.markov_inputs(1, 2, 20000, 256, seed=42)
    t = parity.markov_to_device(inp)
    with pytest.raises(api.DsparkError) as e:
        api.markov_draft(t["base"], t["w1"], t["w2"], None, t["prev"], kernel="cluster")
    assert e.value.status == api.DSPARK_ERR_UNSUPPORTED


def test_cluster_kernel_batch_invariance_bitwise():
    inp = synth.markov_inputs(5, 3, 4000, 128, w_sd=0.3, seed=43)
    full = parity.gpu_markov(inp, kernel="cluster")
    for r in range(5):
        one = dict(inp)
        one["base"] = inp["base"][r:r + 1]
        one["prev0"] = inp["prev0"][r:r + 1]
        g = parity.gpu_markov(one, kernel="cluster")
        np.testing.assert_array_equal(g["out_ids"][0], full["out_ids"][r])
        np.testing.assert_array_equal(g["logits"][0].view(np.uint32),
                                      full["logits"][r].view(np.uint32))


def test_cluster_kernel_in_a_graph_plan():
    """The single-cluster kernel recorded in a CUDA graph: replays match a direct call and
    continue the chain from the prev they leave on the device."""
    inp = synth.markov_config("tiny")
    assert api.markov_kernel_for(1, 4, 4096, 64) == "cluster"
    direct = parity.gpu_markov(inp, dbg=False)
    t = parity.markov_to_device(inp)
    plan = api.MarkovPlan(t["base"], t["w1"], t["w2"], t["d2t"], t["prev"])
    for _ in range(3):
        t["prev"].copy_(torch.from_numpy(inp["prev0"]))
        out = plan.launch()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(out.cpu().numpy(), direct["out_ids"])
        assert api.markov_status(plan.workspace) == 0
    second = plan.launch().cpu().numpy()
    o = parity.oracle.markov_draft(inp["base"], inp["w1"], inp["w2"], None, direct["prev"])
    np.testing.assert_array_equal(second, o["out_ids"])
    plan.close()


def test_cluster_kernel_resets_the_status_word():
    """A grid-kernel draft that timed out leaves DSPARK_ERR_TIMEOUT in the workspace; the
    next draft on the same workspace through the cluster kernel reports its own status."""
    inp = synth.markov_inputs(1, 3, 4096, 64, seed=44)
    t = parity.markov_to_device(inp)
    ws = api.new_markov_workspace(1, 3, 4096, 64)
    out = torch.empty((1, 3), dtype=torch.int64, device="cuda")
    api.markov_draft_debug(t["base"], t["w1"], t["w2"], None, t["prev"], out, ws,
                           missing_arrivals=1, timeout_us=20000)
    assert api.markov_status(ws) == api.DSPARK_ERR_TIMEOUT
    t["prev"].copy_(torch.from_numpy(inp["prev0"]))
    g = api.markov_draft(t["base"], t["w1"], t["w2"], None, t["prev"], workspace=ws,
                         kernel="cluster")
    assert api.markov_status(ws) == 0
    o = parity.oracle.markov_draft(inp["base"], inp["w1"], inp["w2"], None, inp["prev0"])
    np.testing.assert_array_equal(g.cpu().numpy(), o["out_ids"])


def test_strong_bias_chain():
    """Large markov weights make the bias dominate the base row, so every position's id
    really depends on the previous one (the chain is exercised, not just argmax(base))."""
    inp = synth.markov_inputs(4, 8, 5000, 256, base_sd=0.1, w_sd=0.2, seed=21)
    o = parity.oracle.markov_draft(inp["base"], inp["w1"], inp["w2"], None, inp["prev0"])
    assert np.any(o["out_ids"] != np.argmax(inp["base"], axis=2))
    rep = parity.check_markov(inp, parity.gpu_markov(inp))
    assert rep["n_exempt"] == 0


def test_repeat_runs_bit_identical():
    inp = synth.markov_inputs(3, 4, 30000, 256, w_sd=0.3, seed=22)
    a = parity.gpu_markov(inp)
    b = parity.gpu_markov(inp)
    np.testing.assert_array_equal(a["out_ids"], b["out_ids"])
    np.testing.assert_array_equal(a["logits"].view(np.uint32), b["logits"].view(np.uint32))


def test_batch_invariance_bitwise():
    inp = synth.markov_inputs(5, 3, 9000, 256, w_sd=0.3, seed=23)
    full = parity.gpu_markov(inp)
    for r in range(5):
        one = dict(inp)
        one["base"] = inp["base"][r:r + 1]
        one["prev0"] = inp["prev0"][r:r + 1]
        g = parity.gpu_markov(one)
        np.testing.assert_array_equal(g["out_ids"][0], full["out_ids"][r])
        np.testing.assert_array_equal(g["logits"][0].view(np.uint32),
                                      full["logits"][r].view(np.uint32))


def test_debug_outputs_do_not_change_ids():
    inp = synth.markov_inputs(2, 5, 12000, 128, w_sd=0.3, seed=24)
    a = parity.gpu_markov(inp, dbg=True)
    b = parity.gpu_markov(inp, dbg=False)
    np.testing.assert_array_equal(a["out_ids"], b["out_ids"])


def test_plan_matches_direct_call():
    inp = synth.markov_config("reduced_vocab")
    direct = parity.gpu_markov(inp, dbg=False)
    t = parity.markov_to_device(inp)
    plan = api.MarkovPlan(t["base"], t["w1"], t["w2"], t["d2t"], t["prev"])
    for _ in range(3):
        t["prev"].copy_(torch.from_numpy(inp["prev0"]))
        out = plan.launch()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(out.cpu().numpy(), direct["out_ids"])
        assert api.markov_status(plan.workspace) == 0
    # prev stays on the device: a second draft continues from the last id
    plan.launch()
    torch.cuda.synchronize()
    plan.close()


def test_out_of_range_prev_reports_index_error():
    inp = synth.markov_inputs(2, 3, 2000, 64, w_sd=0.3, seed=25)
    bad = dict(inp)
    bad["prev0"] = np.array([2000, inp["prev0"][1]], np.int64)
    g = parity.gpu_markov(bad, dbg=False)
    assert g["status"] == api.DSPARK_ERR_INDEX
    assert np.all(g["out_ids"][0] == -1)
    assert g["prev"][0] == 2000  # untouched
    good = dict(inp)
    good["base"] = inp["base"][1:2]
    good["prev0"] = inp["prev0"][1:2]
    ref = parity.gpu_markov(good, dbg=False)
    np.testing.assert_array_equal(g["out_ids"][1], ref["out_ids"][0])


def test_negative_d2t_reports_index_error():
    inp = synth.markov_inputs(1, 3, 500, 64, seed=26)
    inp["d2t"] = np.full(500, -1, np.int32)
    t = parity.markov_to_device(inp)
    ws = api.new_markov_workspace(1, 3, 500, 64)
    out = api.markov_draft(t["base"], t["w1"], t["w2"], t["d2t"], t["prev"], workspace=ws)
    assert api.markov_status(ws) == api.DSPARK_ERR_INDEX
    assert np.all(out.cpu().numpy() == -1)


def test_empty_calls_enqueue_nothing():
    inp = synth.markov_inputs(1, 2, 300, 64, seed=27)
    t = parity.markov_to_device(inp)
    out = torch.full((1, 0), 7, dtype=torch.int64, device="cuda")
    api.markov_draft(t["base"][:, :0].contiguous(), t["w1"], t["w2"], None, t["prev"],
                     out_ids=out)
    torch.cuda.synchronize()
    assert int(t["prev"][0]) == int(inp["prev0"][0])


def test_device_wait_limit_reports_timeout():
    """Fault injection on the host side of the wait: the step barrier is told to expect
    one more CTA than exists, so it can never complete; the kernel must give up after the
    limit, record DSPARK_ERR_TIMEOUT and leave the context usable."""
    inp = synth.markov_inputs(1, 3, 5000, 64, seed=28)
    t = parity.markov_to_device(inp)
    ws = api.new_markov_workspace(1, 3, 5000, 64)
    out = torch.empty((1, 3), dtype=torch.int64, device="cuda")
    api.markov_draft_debug(t["base"], t["w1"], t["w2"], None, t["prev"], out, ws,
                           missing_arrivals=1, timeout_us=20000)
    assert api.markov_status(ws) == api.DSPARK_ERR_TIMEOUT
    # the same workspace works again afterwards
    t["prev"].copy_(torch.from_numpy(inp["prev0"]))
    g = api.markov_draft(t["base"], t["w1"], t["w2"], None, t["prev"], workspace=ws)
    assert api.markov_status(ws) == 0
    o = parity.oracle.markov_draft(inp["base"], inp["w1"], inp["w2"], None, inp["prev0"])
    np.testing.assert_array_equal(g.cpu().numpy(), o["out_ids"])
