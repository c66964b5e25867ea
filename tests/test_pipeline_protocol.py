"""The mbarrier protocol of the Q8_0 weight-stationary kernel, model-checked on the host.

The kernel's roles wait on mbarriers by phase parity: a wait for the k-th completion of a
barrier passes as soon as the number of completed phases c has the other parity than k,
which is right only while c is k or k + 1.  This test models the roles (TMA producer,
converter groups, MMA issuers, epilogue), the asynchronous events (a stage's copies landing,
a stage's MMAs completing) and the barriers with exactly those semantics, explores many
random interleavings, and checks that every wait that passes sees the phase it waits for
and that every run finishes.  The ring sizes and role counts are read from the kernel
source, so the check follows the kernel.
"""
import os
import random
import re

import pytest

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "dspark_draft_sampling_gb300",
                   "csrc", "ws_q8.cu")


def kernel_constants():
    text = open(SRC).read()

    def const(name):
        m = re.search(rf"constexpr int {name} = (\d+);", text)
        assert m, name
        return int(m.group(1))

    return dict(stages=const("kStages"), aslots=const("kASlots"), issuers=const("kMmaIssuers"),
                conv_groups=const("kConvWarps") // 4)


class Barrier:
    def __init__(self):
        self.completed = 0


def run(stages, aslots, issuers, conv_groups, n_stages, rng):
    """One random interleaving.  Returns None, or a description of the first wait that
    passed on the wrong phase (or of a deadlock)."""
    full_r = [Barrier() for _ in range(stages)]   # stage's copies landed
    done = [Barrier() for _ in range(stages)]     # stage's MMAs completed (one commit)
    full_a = [Barrier() for _ in range(aslots)]   # A tile written by its converter group
    empty_t = [Barrier() for _ in range(aslots)]  # accumulator group drained by the epilogue

    def passes(bar, k):
        """Parity wait for the k-th completion (0-based) of `bar`."""
        return (bar.completed & 1) != (k & 1)

    def exact(bar, k):
        return bar.completed == k + 1

    # per-role cursor (next stage) and, for roles with two waits per stage, which wait is
    # next (each wait is its own step, as in the kernel: the second starts after the first
    # passed, and the first is not checked again); pending asynchronous completions
    prod = 0
    conv = [g for g in range(conv_groups)]     # next stage of each group
    conv_w = [0] * conv_groups
    iss = [i for i in range(issuers)]
    iss_w = [0] * issuers
    epi = 0
    pending_land, pending_mma = [], []
    error = None

    def wait(bar, k, who):
        """One parity wait; records an error if it passes on a phase other than k."""
        nonlocal error
        if not passes(bar, k):
            return False
        if not exact(bar, k) and error is None:
            error = f"{who}: passed with {bar.completed} completed phases, wanted {k + 1}"
        return True

    def step_producer():
        nonlocal prod
        J = prod
        if J >= n_stages:
            return False
        if J >= stages and not wait(done[J % stages], J // stages - 1, f"producer stage {J}"):
            return False
        pending_land.append(J)
        prod += 1
        return True

    def step_converter(g):
        J = conv[g]
        if J >= n_stages:
            return False
        if conv_w[g] == 0:
            if not wait(full_r[J % stages], J // stages, f"converter stage {J} (copies)"):
                return False
            conv_w[g] = 1
            return True
        if J >= aslots:
            jp = J - aslots
            if not wait(done[jp % stages], jp // stages, f"converter stage {J} (A slot free)"):
                return False
        full_a[J % aslots].completed += 1
        conv[g] += conv_groups
        conv_w[g] = 0
        return True

    def step_issuer(i):
        J = iss[i]
        if J >= n_stages:
            return False
        g, k = J % aslots, J // aslots
        if iss_w[i] == 0:
            if not wait(full_a[g], k, f"issuer {i} stage {J} (A written)"):
                return False
            iss_w[i] = 1
            return True
        if J >= aslots and not wait(empty_t[g], k - 1, f"issuer {i} stage {J} (accumulators drained)"):
            return False
        pending_mma.append(J)
        iss[i] += issuers
        iss_w[i] = 0
        return True

    def step_epilogue():
        nonlocal epi
        J = epi
        if J >= n_stages:
            return False
        if not wait(done[J % stages], J // stages, f"epilogue stage {J}"):
            return False
        empty_t[J % aslots].completed += 1
        epi += 1
        return True

    def land(idx):
        J = pending_land.pop(idx)
        full_r[J % stages].completed += 1
        return True

    def mma_complete(idx):
        # one commit per stage; an issuer's commits complete in its issue order
        J = pending_mma[idx]
        mine = [x for x in pending_mma if x % issuers == J % issuers]
        if J != min(mine):
            return False
        pending_mma.pop(idx)
        done[J % stages].completed += 1
        return True

    while error is None:
        actions = [step_producer, step_epilogue]
        actions += [lambda g=g: step_converter(g) for g in range(conv_groups)]
        actions += [lambda i=i: step_issuer(i) for i in range(issuers)]
        actions += [lambda x=x: land(x) for x in range(len(pending_land))]
        actions += [lambda x=x: mma_complete(x) for x in range(len(pending_mma))]
        rng.shuffle(actions)
        if not any(a() for a in actions):
            break
    if error:
        return error
    if epi < n_stages:
        return f"deadlock: epilogue at stage {epi} of {n_stages}"
    return None


def check(stages, aslots, issuers, conv_groups, trials=300, n_stages=48, seed=0):
    rng = random.Random(seed)
    for _ in range(trials):
        err = run(stages, aslots, issuers, conv_groups, n_stages, rng)
        if err:
            return err
    return None


def test_kernel_protocol_is_exact_under_random_interleavings():
    c = kernel_constants()
    assert check(c["stages"], c["aslots"], c["issuers"], c["conv_groups"]) is None


def test_other_issuer_counts_that_divide_the_slots_are_exact():
    c = kernel_constants()
    for issuers in (1, 4):
        assert check(c["stages"], c["aslots"], issuers, c["conv_groups"], trials=100) is None


@pytest.mark.parametrize("issuers", [3])
def test_an_issuer_count_that_does_not_divide_the_slots_is_caught(issuers):
    # the race the kernel once had: the issuer of stage J did not own stage J - 4, the
    # previous use of its A slot, and its first parity wait passed a whole phase early
    c = kernel_constants()
    err = check(c["stages"], c["aslots"], issuers, c["conv_groups"], trials=2000)
    assert err is not None and "(A written)" in err
