"""Pins of the Markov-draft oracle against facts fixed independently of it.

Each test would fail for a plausible slip in the oracle: a transposed GEMV (w1 vs w2
roles), a wrong base row, a dropped bias or base term, highest- instead of lowest-index
tie-break, prev carried in target space instead of draft space, or a d2t applied twice.
"""
import numpy as np
import pytest

import oracle
from oracle import brute
from dspark_draft_sampling_gb300 import synth


def _tiny(seed, B, k, V, R, *, d2t=False, w_sd=1.0, ties=0):
    rng = np.random.default_rng(seed)
    base = rng.standard_normal((B, k, V)).astype(np.float32)
    w1 = synth.f32_to_bf16_bits(rng.standard_normal((V, R)).astype(np.float32) * w_sd)
    w2 = synth.f32_to_bf16_bits(rng.standard_normal((V, R)).astype(np.float32) * w_sd)
    for _ in range(ties):
        a, b = sorted(rng.choice(V, 2, replace=False))
        w2[b] = w2[a]
        base[:, :, b] = base[:, :, a]
    prev0 = rng.integers(0, V, size=B).astype(np.int64)
    d = rng.permutation(3 * V)[:V].astype(np.int32) if d2t else None
    return base, w1, w2, d, prev0


@pytest.mark.parametrize("seed,B,k,V,R,d2t,ties", [
    (0, 1, 4, 8, 2, False, 0),
    (1, 2, 3, 16, 4, True, 0),
    (2, 2, 4, 12, 3, True, 2),
    (3, 1, 4, 5, 1, False, 1),
    (4, 2, 2, 16, 4, False, 3),
])
def test_brute_force_exact(oracle_lib, seed, B, k, V, R, d2t, ties):
    base, w1, w2, d, prev0 = _tiny(seed, B, k, V, R, d2t=d2t, ties=ties)
    got = oracle.markov_draft(base, w1, w2, d, prev0, want_logits=True)
    out, draft, logits = brute.markov_draft(base, w1, w2, d, prev0)
    np.testing.assert_array_equal(got["draft_ids"], draft)
    np.testing.assert_array_equal(got["out_ids"], out)
    for r in range(B):
        for i in range(k):
            exact = np.array([float(x) for x in logits[r][i]])
            np.testing.assert_allclose(got["logits"][r, i], exact, rtol=1e-13, atol=1e-13)


def test_hand_worked_chain(oracle_lib):
    """vocab 3, rank 2, k 2: every quantity is a small dyadic number, so the expected
    draft follows from the definition by hand.

    w1 = [[1,0],[0,1],[1,1]], w2 = [[2,0],[0,2],[-1,-1]] (all exact in bf16), prev0 = 0.
    Position 0: h = w1[0] = (1,0); bias = (2, 0, -1); base row (0, 1.5, 0) -> logits
    (2, 1.5, -1) -> id 0.  Position 1: h = w1[0] = (1,0) again; base row (0, 2, 3) ->
    logits (2, 2, 2): a three-way tie -> lowest index 0.  With d2t = (7, 8, 9) the
    target ids are (7, 7).  A transposed GEMV (bias[v] = sum_j w1[v,j] w2[p,j]) would give
    bias (2, 0, 2) at position 0 and pick id 0 then id 2; highest-index tie-break picks 2.
    """
    w1 = synth.f32_to_bf16_bits(np.array([[1, 0], [0, 1], [1, 1]], np.float32))
    w2 = synth.f32_to_bf16_bits(np.array([[2, 0], [0, 2], [-1, -1]], np.float32))
    base = np.array([[[0, 1.5, 0], [0, 2, 3]]], np.float32)
    prev0 = np.array([0], np.int64)
    d2t = np.array([7, 8, 9], np.int32)
    got = oracle.markov_draft(base, w1, w2, d2t, prev0, want_logits=True, want_bias=True)
    np.testing.assert_array_equal(got["draft_ids"], [[0, 0]])
    np.testing.assert_array_equal(got["out_ids"], [[7, 7]])
    np.testing.assert_array_equal(got["bias"][0, 0], [2.0, 0.0, -1.0])
    np.testing.assert_array_equal(got["logits"][0, 1], [2.0, 2.0, 2.0])


def test_prev_is_draft_space(oracle_lib):
    """The gather uses the draft-space id, not the d2t image: with d2t mapping every id
    out of the draft vocabulary, a target-space prev would be out of range."""
    base, w1, w2, _, prev0 = _tiny(7, 1, 4, 16, 4)
    d2t = (np.arange(16) + 1000).astype(np.int32)
    got = oracle.markov_draft(base, w1, w2, d2t, prev0)
    ident = oracle.markov_draft(base, w1, w2, None, prev0)
    np.testing.assert_array_equal(got["out_ids"], ident["out_ids"] + 1000)


def test_zero_w2_closed_form(oracle_lib):
    """markov_w2 = 0 makes every bias 0: the ids are d2t[argmax base row], whatever prev."""
    inp = synth.markov_inputs(2, 5, 3000, 64, base_sd=2.0, d2t="injective", seed=3)
    w2 = np.zeros_like(inp["w2"])
    expect = inp["d2t"][np.argmax(inp["base"], axis=2)]
    for prev0 in (inp["prev0"], np.array([0, 2999], np.int64)):
        got = oracle.markov_draft(inp["base"], inp["w1"], w2, inp["d2t"], prev0)
        np.testing.assert_array_equal(got["out_ids"], expect)


def test_zero_w1_closed_form(oracle_lib):
    inp = synth.markov_inputs(1, 4, 2000, 64, seed=4)
    w1 = np.zeros_like(inp["w1"])
    got = oracle.markov_draft(inp["base"], w1, inp["w2"], None, inp["prev0"])
    np.testing.assert_array_equal(got["out_ids"], np.argmax(inp["base"], axis=2))


def test_d2t_identity_vs_injective(oracle_lib):
    inp = synth.markov_inputs(2, 6, 4000, 64, base_sd=2.0, w_sd=0.2, d2t="injective", seed=5)
    a = oracle.markov_draft(inp["base"], inp["w1"], inp["w2"], None, inp["prev0"])
    b = oracle.markov_draft(inp["base"], inp["w1"], inp["w2"], inp["d2t"], inp["prev0"])
    np.testing.assert_array_equal(a["draft_ids"], b["draft_ids"])
    np.testing.assert_array_equal(b["out_ids"], inp["d2t"][a["out_ids"]])
    ident = np.arange(4000, dtype=np.int32)
    c = oracle.markov_draft(inp["base"], inp["w1"], inp["w2"], ident, inp["prev0"])
    np.testing.assert_array_equal(c["out_ids"], a["out_ids"])


def test_planted_ties_lowest_index(oracle_lib):
    inp = synth.markov_inputs(1, 7, 3000, 64, base_sd=2.0, w_sd=0.02, tie_frac=0.005, seed=6)
    got = oracle.markov_draft(inp["base"], inp["w1"], inp["w2"], None, inp["prev0"],
                              want_logits=True)
    ties = inp["ties"]
    for i in inp["spiked_steps"]:
        v1, v2 = ties[(i // 2) % len(ties)]
        assert got["logits"][0, i, v1] == got["logits"][0, i, v2]
        assert got["draft_ids"][0, i] == v1


def test_argmax_certificate(oracle_lib):
    inp = synth.markov_inputs(2, 4, 5000, 128, w_sd=0.3, seed=8)
    got = oracle.markov_draft(inp["base"], inp["w1"], inp["w2"], None, inp["prev0"],
                              want_logits=True)
    L = got["logits"]
    for r in range(2):
        for i in range(4):
            v = got["draft_ids"][r, i]
            assert np.all(L[r, i] <= L[r, i, v])
            assert np.all(L[r, i, :v] < L[r, i, v])


def test_batch_invariance(oracle_lib):
    inp = synth.markov_inputs(3, 5, 2500, 64, w_sd=0.3, seed=9)
    full = oracle.markov_draft(inp["base"], inp["w1"], inp["w2"], None, inp["prev0"])
    for r in range(3):
        one = oracle.markov_draft(inp["base"][r:r + 1], inp["w1"], inp["w2"], None,
                                  inp["prev0"][r:r + 1])
        np.testing.assert_array_equal(one["out_ids"][0], full["out_ids"][r])


def test_power_of_two_scaling(oracle_lib):
    """Doubling base and markov_w2 doubles every logit exactly (bf16 exponent + 1)."""
    inp = synth.markov_inputs(2, 5, 3000, 64, w_sd=0.3, seed=10)
    w2x2 = inp["w2"].copy()
    nz = (w2x2 & 0x7F80) != 0
    w2x2[nz] += 0x80
    a = oracle.markov_draft(inp["base"], inp["w1"], inp["w2"], None, inp["prev0"],
                            want_logits=True)
    b = oracle.markov_draft(inp["base"] * 2, inp["w1"], w2x2, None, inp["prev0"],
                            want_logits=True)
    np.testing.assert_array_equal(a["out_ids"], b["out_ids"])
    np.testing.assert_array_equal(b["logits"], 2 * a["logits"])


def test_vocab_permutation_equivariance(oracle_lib):
    inp = synth.markov_inputs(2, 5, 2000, 64, w_sd=0.3, d2t="injective", seed=11)
    V = 2000
    pi = np.random.default_rng(12).permutation(V)  # old id v -> new id pi[v]
    inv = np.argsort(pi)
    w1p, w2p = inp["w1"][inv], inp["w2"][inv]
    basep = inp["base"][:, :, inv]
    d2tp = inp["d2t"][inv]
    a = oracle.markov_draft(inp["base"], inp["w1"], inp["w2"], inp["d2t"], inp["prev0"])
    b = oracle.markov_draft(basep, w1p, w2p, d2tp, pi[inp["prev0"]])
    np.testing.assert_array_equal(b["out_ids"], a["out_ids"])
    np.testing.assert_array_equal(b["draft_ids"], pi[a["draft_ids"]])


def test_teacher_forcing(oracle_lib):
    """Forcing prev to the oracle's own ids changes nothing; forcing another sequence makes
    each position equal a one-step draft from the forced prev."""
    inp = synth.markov_inputs(1, 4, 1500, 64, w_sd=0.5, seed=13)
    a = oracle.markov_draft(inp["base"], inp["w1"], inp["w2"], None, inp["prev0"],
                            forced_prev=None)
    b = oracle.markov_draft(inp["base"], inp["w1"], inp["w2"], None, inp["prev0"],
                            forced_prev=a["draft_ids"])
    np.testing.assert_array_equal(a["out_ids"], b["out_ids"])
    forced = np.array([[3, 77, 1499, 0]], np.int64)
    c = oracle.markov_draft(inp["base"], inp["w1"], inp["w2"], None, inp["prev0"],
                            forced_prev=forced)
    prevs = [inp["prev0"][0], 3, 77, 1499]
    for i in range(4):
        one = oracle.markov_draft(inp["base"][:, i:i + 1], inp["w1"], inp["w2"], None,
                                  np.array([prevs[i]], np.int64))
        assert one["out_ids"][0, 0] == c["out_ids"][0, i]


def test_rejects_out_of_range_prev(oracle_lib):
    inp = synth.markov_inputs(1, 2, 100, 64, seed=14)
    with pytest.raises(ValueError):
        oracle.markov_draft(inp["base"], inp["w1"], inp["w2"], None, np.array([100], np.int64))
