"""The mbarrier protocols of the Q8_0 weight-stationary kernel, the grid Markov kernel and
the single-cluster Markov kernel's exchange, model-checked on the host.

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


# ---------------------------------------------------------------- Markov draft kernel ---
MARKOV_SRC = os.path.join(os.path.dirname(SRC), "markov_tc.cu")


def markov_slots(rank, nb=8):
    """Tile slots of the Markov kernel's ring at this rank and request count: kRingBudget
    bytes of slots, each one [128 x rank] bf16 tile (one 16 KB box per 64 columns) plus the
    tile's base rows (nb x 128 fp32, rounded up to 1 KB), at most kMaxSlots."""
    text = open(MARKOV_SRC).read()
    budget = re.search(r"constexpr int kRingBudget = (\d+) \* 1024;", text)
    cap = re.search(r"constexpr int kMaxSlots = (\d+);", text)
    assert budget and cap
    slot = (rank // 64) * 16384 + (nb * 128 * 4 + 1023) // 1024 * 1024
    return min(int(cap.group(1)), int(budget.group(1)) * 1024 // slot)


class Barrier2(Barrier):
    """An mbarrier whose phase completes after `count` arrivals."""

    def __init__(self, count):
        super().__init__()
        self.count = count
        self.arrived = 0

    def arrive(self):
        self.arrived += 1
        if self.arrived == self.count:
            self.arrived = 0
            self.completed += 1


def run_markov(nslots, k, ntiles, rng, epi_warps=4, epilogue_holds_slot=True, issuers=2):
    """One random interleaving of the Markov kernel's roles for one CTA: the TMA producer
    (one copy of tile + base rows per slot, running ahead across positions), the MMA issuers
    (issuer p takes the tiles tc with tc % issuers == p and accumulator p; per position every
    issuer waits for H; per own tile: wait for its accumulator to be drained, then for the
    slot; its completion commits to the slot and to the accumulator; each issuer's commits
    complete in its issue order, the issuers' in any interleaving), and each epilogue warp
    (per tile: wait for the slot to land, read the base rows and arrive on the slot's empty
    barrier, wait for the accumulator, read it and arrive on its empty barrier; after the last
    tile of a position: the next position's H).  The slot's empty barrier completes after the
    commit and every epilogue warp (with epilogue_holds_slot=False, after the commit alone).
    Returns an error string or None."""
    full = [Barrier() for _ in range(nslots)]
    empty = [Barrier2(1 + (epi_warps if epilogue_holds_slot else 0)) for _ in range(nslots)]
    acc_full = [Barrier() for _ in range(2)]
    acc_empty = [Barrier2(epi_warps) for _ in range(2)]
    h_full = [Barrier2(epi_warps) for _ in range(2)]
    h_full[0].completed = 1  # the epilogue builds position 0's H before the loop
    total = k * ntiles
    error = None

    def wait(bar, kk, who):
        nonlocal error
        if (bar.completed & 1) == (kk & 1):
            return False
        if bar.completed != kk + 1 and error is None:
            error = f"{who}: passed with {bar.completed} completed phases, wanted {kk + 1}"
        return True

    st = dict(prod=0)
    iss = [dict(q=0, w=0) for _ in range(issuers)]  # q: next tile counter this issuer looks at
    epi = [dict(q=0, step=0) for _ in range(epi_warps)]
    pending_land = []
    pending_mma = [[] for _ in range(issuers)]

    def producer():
        q = st["prod"]
        if q >= total:
            return False
        if q >= nslots and not wait(empty[q % nslots], q // nslots - 1, f"producer tile {q}"):
            return False
        pending_land.append(q)
        st["prod"] += 1
        return True

    def issuer(p):
        me = iss[p]
        q = me["q"]
        if q >= total:
            return False
        i, t = divmod(q, ntiles)
        if me["w"] == 0:  # the position's H (every issuer, first tile of each position)
            if t == 0 and not wait(h_full[i & 1], i >> 1, f"issuer {p} position {i} (H)"):
                return False
            me["w"] = 1
            return True
        if q % issuers != p:  # another issuer's tile
            me["q"] += 1
            me["w"] = 0
            return True
        if me["w"] == 1:  # accumulator p drained (its previous use)
            u = q // issuers
            if u >= 1 and not wait(acc_empty[p], u - 1, f"issuer {p} tile {q} (accumulator)"):
                return False
            me["w"] = 2
            return True
        if not wait(full[q % nslots], q // nslots, f"issuer {p} tile {q} (tile landed)"):
            return False
        pending_mma[p].append(q)
        me["q"] += 1
        me["w"] = 0
        return True

    def epilogue(w):
        e = epi[w]
        q = e["q"]
        if q >= total:
            return False
        if e["step"] == 0:  # slot landed: read the base rows, release the slot
            if not wait(full[q % nslots], q // nslots, f"epilogue warp {w} tile {q} (base rows)"):
                return False
            if epilogue_holds_slot:
                empty[q % nslots].arrive()
            e["step"] = 1
            return True
        if not wait(acc_full[q % issuers], q // issuers, f"epilogue warp {w} tile {q} (accumulator)"):
            return False
        acc_empty[q % issuers].arrive()
        i, t = divmod(q, ntiles)
        if t == ntiles - 1 and i + 1 < k:
            h_full[(i + 1) & 1].arrive()
        e["q"] += 1
        e["step"] = 0
        return True

    def land(x):
        q = pending_land.pop(x)
        full[q % nslots].completed += 1
        return True

    def mma_complete(p):
        if not pending_mma[p]:
            return False
        q = pending_mma[p].pop(0)  # one issuer's commits complete in its issue order
        empty[q % nslots].arrive()
        acc_full[p].completed += 1
        return True

    while error is None:
        actions = [producer] + [lambda p=p: issuer(p) for p in range(issuers)]
        actions += [lambda w=w: epilogue(w) for w in range(epi_warps)]
        actions += [lambda x=x: land(x) for x in range(len(pending_land))]
        actions += [lambda p=p: mma_complete(p) for p in range(issuers)]
        rng.shuffle(actions)
        if not any(a() for a in actions):
            break
    if error:
        return error
    if any(e["q"] < total for e in epi):
        return f"deadlock: epilogue at tiles {[e['q'] for e in epi]} of {total}"
    return None


@pytest.mark.parametrize("rank", [64, 128, 256])
def test_markov_protocol_is_exact_under_random_interleavings(rank):
    nslots = markov_slots(rank)
    assert nslots == {64: 10, 128: 5, 256: 3}[rank]
    rng = random.Random(rank)
    for _ in range(150):
        k = rng.randint(1, 6)
        ntiles = rng.randint(1, 14)
        err = run_markov(nslots, k, ntiles, rng)
        assert err is None, (rank, nslots, k, ntiles, err)


def test_markov_model_catches_a_slot_freed_by_the_mma_alone():
    # if the MMAs' commit alone freed a slot, the producer could refill it before a slow
    # epilogue warp has read the tile's base rows; the model must see that wait pass a phase
    # late, and the kernel's ring must keep at least three slots
    rng = random.Random(7)
    assert any(run_markov(3, 4, 6, rng, epilogue_holds_slot=False) for _ in range(300))
    assert min(markov_slots(r, nb) for r in (64, 128, 256) for nb in (1, 2, 4, 8)) >= 3


# ---- the single-cluster Markov kernel's exchange (csrc/markov_cluster.cu) ----------------
# Every CTA sends, per position, its message to every CTA of the cluster (itself included)
# with stores whose bytes complete on the receiver's inbox barrier for that position's parity;
# a CTA waits only for its own inbox (parity wait), reads it, re-arms that barrier for the
# position two ahead (arrive.expect_tx), and only then sends the next position.  The barriers
# of positions 0 and 1 are armed before any CTA sends.  The model delivers each message at a
# random later moment and checks that every delivery lands on an armed phase of the right
# position, that every wait that passes sees exactly its phase, and that a CTA reads its
# whole inbox of the position it waited for.

class ArmedBarrier:
    """mbarrier of arrival count 1 with a transaction count."""

    def __init__(self):
        self.completed = 0  # completed phases
        self.pending = 1    # arrivals still expected in the current phase
        self.tx = 0         # transaction bytes still expected (may run ahead of the arm)

    def arrive_expect(self, n):
        self.pending -= 1
        self.tx += n
        self._maybe_complete()

    def complete_tx(self, n):
        self.tx -= n
        self._maybe_complete()

    def _maybe_complete(self):
        if self.pending == 0 and self.tx == 0:
            self.completed += 1
            self.pending = 1


def run_cluster_exchange(C, k, rng, nbuf=2):
    bars = [[ArmedBarrier() for _ in range(nbuf)] for _ in range(C)]
    inbox = [[[None] * C for _ in range(nbuf)] for _ in range(C)]
    for r in range(C):  # armed before the first cluster barrier
        for p in range(min(k, nbuf)):
            bars[r][p % nbuf].arrive_expect(C)
    pos = [0] * C
    state = ["send"] * C  # send -> wait -> read -> (next position)
    in_flight = []        # (sender, receiver, position)
    error = None
    while True:
        actions = [("cta", c) for c in range(C) if pos[c] < k]
        actions += [("deliver", j) for j in range(len(in_flight))]
        if not actions:
            break
        enabled = []
        for kind, x in actions:
            if kind == "deliver":
                enabled.append((kind, x))
                continue
            c = x
            if state[c] == "wait":
                i = pos[c]
                b = bars[c][i % nbuf]
                if (b.completed & 1) == ((i // nbuf) & 1):
                    continue  # the parity wait does not pass yet
            enabled.append((kind, x))
        if not enabled:
            return "deadlock"
        kind, x = rng.choice(enabled)
        if kind == "deliver":
            s, r, p = in_flight.pop(x)
            b = bars[r][p % nbuf]
            if (b.completed != p // nbuf or b.pending != 0) and error is None:
                error = f"message of position {p} from CTA {s} landed on phase {b.completed} (armed: {b.pending == 0})"
            inbox[r][p % nbuf][s] = p
            b.complete_tx(1)
            continue
        c = x
        i = pos[c]
        if state[c] == "send":
            in_flight += [(c, r, i) for r in range(C)]
            state[c] = "wait"
        elif state[c] == "wait":
            b = bars[c][i % nbuf]
            if b.completed != i // nbuf + 1 and error is None:
                error = f"CTA {c} passed its wait of position {i} with {b.completed} completed phases"
            state[c] = "read"
        else:
            if any(inbox[c][i % nbuf][s] != i for s in range(C)) and error is None:
                error = f"CTA {c} read an incomplete inbox at position {i}: {inbox[c][i % nbuf]}"
            if i + nbuf < k:
                bars[c][i % nbuf].arrive_expect(C)
            pos[c] += 1
            state[c] = "send"
        if error:
            return error
    return error


@pytest.mark.parametrize("C,k", [(2, 6), (4, 9), (16, 5)])
def test_cluster_exchange_protocol_is_exact_under_random_interleavings(C, k):
    rng = random.Random(C * 100 + k)
    for _ in range(200):
        assert run_cluster_exchange(C, k, rng) is None


def test_cluster_exchange_model_catches_a_single_inbox():
    """With one inbox (and one barrier) a fast CTA's next message can land on the phase a slow
    CTA is still collecting; the model must find such an interleaving."""
    rng = random.Random(7)
    found = any(run_cluster_exchange(3, 6, rng, nbuf=1) is not None for _ in range(300))
    assert found
