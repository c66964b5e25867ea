"""GPU confidence probe vs the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

from dspark_draft_sampling_gb300 import api, synth
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(dspark_lib):
    return dspark_lib


def test_batched_cycle_workload():
    """2 probes per cycle x 1024 cycles, 7424-wide, threshold 0.5."""
    inp = synth.probe_inputs(2048, 7424, seed=0)
    z, gate = parity.gpu_probe(inp)
    rep = parity.check_probe(inp, z, gate)
    assert rep["n_gate_mismatch"] == 0
    assert rep["n_near_threshold"] <= 2
    assert rep["max_z_err"] < 1e-4
    assert 0 < gate.sum() < 2048


@pytest.mark.parametrize("n,K,t,seed", [(1, 7424, 0.5, 1), (7, 32, 0.5, 2), (33, 7424, 0.8, 3),
                                        (100, 4096, 0.2, 4), (5, 7456, 0.5, 5)])
def test_shapes_and_thresholds(n, K, t, seed):
    inp = synth.probe_inputs(n, K, seed=seed, threshold=t, random_scales=True, scale=0.01)
    z, gate = parity.gpu_probe(inp)
    parity.check_probe(inp, z, gate)


def test_one_hot_is_exact():
    inp = synth.probe_inputs(1, 7424, seed=6, random_scales=True)
    x = np.zeros((3, 7424), np.float32)
    for p, (b, j) in enumerate([(0, 0), (100, 17), (231, 31)]):
        x[p, 32 * b + j] = 1.0
    inp["hidden"] = x
    z, _ = parity.gpu_probe(inp)
    zo, _ = parity.oracle.conf_probe(inp["wq"], x, inp["bias"], 0.5)
    np.testing.assert_array_equal(z.astype(np.float64), zo.astype(np.float32).astype(np.float64))


def test_repeat_bit_identical():
    inp = synth.probe_inputs(64, 7424, seed=7)
    a, ga = parity.gpu_probe(inp)
    b, gb = parity.gpu_probe(inp)
    np.testing.assert_array_equal(a.view(np.uint32), b.view(np.uint32))
    np.testing.assert_array_equal(ga, gb)


def test_gate_readback_is_four_bytes():
    inp = synth.probe_inputs(1, 7424, seed=8)
    wq = torch.from_numpy(inp["wq"]).cuda()
    hid = torch.from_numpy(inp["hidden"]).cuda()
    gate = torch.empty(1, dtype=torch.int32, device="cuda")
    api.conf_probe(wq, hid, inp["bias"], 0.5, gate_out=gate)
    host = gate.cpu()
    assert host.numel() * host.element_size() == 4
    _, go = parity.oracle.conf_probe(inp["wq"], inp["hidden"], inp["bias"], 0.5)
    assert int(host[0]) == int(go[0])


def test_rejects_misaligned_hidden():
    inp = synth.probe_inputs(2, 64, seed=9)
    wq = torch.from_numpy(inp["wq"]).cuda()
    flat = torch.from_numpy(inp["hidden"].reshape(-1)).cuda()
    with pytest.raises(api.DsparkError):
        api.conf_probe(wq, flat[1:65], inp["bias"], 0.5)


def test_split_input_matches_concatenated():
    """[hidden(7168); markov_state(256)] given as two buffers (strided views of a wider
    buffer for the hidden part) gives bit-identical logits to the contiguous probe."""
    inp = synth.probe_inputs(512, 7424, seed=10)
    full = torch.from_numpy(inp["hidden"]).cuda()
    wq = torch.from_numpy(inp["wq"]).cuda()
    wide = torch.zeros((512, 7168 + 64), dtype=torch.float32, device="cuda")
    wide[:, :7168] = full[:, :7168]
    hidden = wide[:, :7168]                 # row stride 7232 floats
    state = full[:, 7168:].contiguous()     # [512, 256]
    z_split, g_split = api.conf_probe_split(wq, hidden, state, inp["bias"], 0.5)
    z_full, g_full = api.conf_probe(wq, full, inp["bias"], 0.5)
    torch.cuda.synchronize()
    assert torch.equal(z_split.view(torch.int32), z_full.view(torch.int32))
    assert torch.equal(g_split, g_full)
    parity.check_probe(inp, z_split.cpu().numpy(), g_split.cpu().numpy())


def test_odd_aligned_weight_row():
    """Q8_0 rows are 34-byte blocks with no alignment requirement: a row starting at an odd
    address must give the same logits, bit for bit, as an aligned copy."""
    inp = synth.probe_inputs(6, 7424, seed=8, random_scales=True, scale=0.01)
    hid = torch.from_numpy(inp["hidden"]).cuda()
    wq = torch.from_numpy(inp["wq"]).cuda()
    buf = torch.zeros(wq.numel() + 1, dtype=torch.uint8, device="cuda")
    buf[1:] = wq
    odd = buf[1:]
    assert odd.data_ptr() % 2 == 1
    z1, g1 = api.conf_probe(wq, hid, inp["bias"], inp["threshold"])
    z2, g2 = api.conf_probe(odd, hid, inp["bias"], inp["threshold"])
    torch.cuda.synchronize()
    assert torch.equal(z1.view(torch.int32), z2.view(torch.int32))
    assert torch.equal(g1, g2)
    parity.check_probe(inp, z2.cpu().numpy(), g2.cpu().numpy())


def test_gate_into_pinned_host_memory():
    """gate_out in pinned host memory: the kernel's own 4-byte store is the readback."""
    inp = synth.probe_inputs(3, 7424, seed=9)
    wq = torch.from_numpy(inp["wq"]).cuda()
    hid = torch.from_numpy(inp["hidden"]).cuda()
    _, g_dev = api.conf_probe(wq, hid, inp["bias"], 0.5)
    g_host = torch.full((3,), -1, dtype=torch.int32).pin_memory()
    api.conf_probe(wq, hid, inp["bias"], 0.5, gate_out=g_host)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(g_host.numpy(), g_dev.cpu().numpy())
    _, go = parity.oracle.conf_probe(inp["wq"], inp["hidden"], inp["bias"], 0.5)
    np.testing.assert_array_equal(g_host.numpy(), go)


@pytest.mark.parametrize("split", [False, True])
def test_large_batch_ring_matches_small_batches_bitwise(split):
    """A batch large enough for the persistent bulk-copy ring kernel (2048 probes) gives the
    same bits, probe by probe, as the same probes run 64 at a time (one CTA per probe, every
    load in flight); with split=True both run over the two-piece input (the ring then copies
    each row in two pieces), with random block scales and an odd number of probes."""
    n = 2047
    inp = synth.probe_inputs(n, 7424, seed=11, random_scales=True, scale=0.01)
    wq = torch.from_numpy(inp["wq"]).cuda()
    full = torch.from_numpy(inp["hidden"]).cuda()

    def run(lo, hi):
        if not split:
            return api.conf_probe(wq, full[lo:hi], inp["bias"], 0.5)
        wide = torch.zeros((hi - lo, 7168 + 64), dtype=torch.float32, device="cuda")
        wide[:, :7168] = full[lo:hi, :7168]
        return api.conf_probe_split(wq, wide[:, :7168], full[lo:hi, 7168:].contiguous(), inp["bias"], 0.5)

    z_big, g_big = run(0, n)
    torch.cuda.synchronize()
    for lo in range(0, n, 64):
        z, g = run(lo, min(n, lo + 64))
        torch.cuda.synchronize()
        assert torch.equal(z.view(torch.int32), z_big[lo:lo + 64].view(torch.int32)), lo
        assert torch.equal(g, g_big[lo:lo + 64]), lo
    parity.check_probe(inp, z_big.cpu().numpy(), g_big.cpu().numpy())


def test_prepared_probe_call_decides_like_the_oracle():
    """api.ProbeCall: arguments marshalled once; decide() launches and polls the decisions the
    kernel stores into pinned host memory, call after call, as the oracle decides them."""
    inp = synth.probe_inputs(5, 7424, seed=12)
    wq = torch.from_numpy(inp["wq"]).cuda()
    hid = torch.from_numpy(inp["hidden"]).cuda()
    _, go = parity.oracle.conf_probe(inp["wq"], inp["hidden"], inp["bias"], 0.5)
    z = torch.empty(5, dtype=torch.float32, device="cuda")
    call = api.ProbeCall(wq, hid, inp["bias"], 0.5, logit_out=z)
    for _ in range(3):
        np.testing.assert_array_equal(call.decide(), go)
    torch.cuda.synchronize()
    parity.check_probe(inp, z.cpu().numpy(), go)
    one = api.ProbeCall(wq, hid[0], inp["bias"], 0.5)  # a single probe: one 4-byte decision
    assert one.decide().tolist() == [int(go[0])]
    dev_gate = torch.empty(5, dtype=torch.int32, device="cuda")
    on_device = api.ProbeCall(wq, hid, inp["bias"], 0.5, gate_out=dev_gate)
    on_device.launch()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(dev_gate.cpu().numpy(), go)
    with pytest.raises(ValueError):
        on_device.decide()
