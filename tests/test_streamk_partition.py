"""The stream-K partition of the grouped Q8_0 matvec launch, model-checked on the host.

The grouped launch (`dspark_ws_matvec_q8_grouped`, csrc/ws_q8.cu) lays the 128-row blocks of
all problems, each over all of its K, end to end as one sequence of 256-k superblocks and
gives CTA c of G the contiguous range [c T / G, (c + 1) T / G).  A range falls into pieces at
row-block boundaries.  The kernel relies on these properties, checked here for many random
groups and grid sizes with the same integer arithmetic:

  * every superblock of every row block belongs to exactly one piece;
  * a piece that starts inside a row block (a later part) is the first piece of its CTA, and
    a piece that starts a row block but does not finish it (a first part) is the last piece
    of its CTA, so each CTA writes at most one partial and waits at most once;
  * the first part's CTA waits exactly for the CTAs j > c with range_begin(j) < row-block end,
    and those are exactly the CTAs whose first piece is a later part of that row block: every
    partial is read by one CTA and every flag is reset once, and a CTA only ever waits for
    higher-numbered CTAs, whose later parts need nothing from anyone (no wait cycle);
  * a row block no boundary cuts is one whole piece (summed exactly as an unsplit unit).
"""
import os
import random
import re

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "dspark_draft_sampling_gb300",
                   "csrc", "ws_q8.cu")


def superblock_k():
    text = open(SRC).read()
    ks = re.search(r"constexpr int kKS = (\d+);", text)
    sup = re.search(r"constexpr int kSuper = (\d+);", text)
    assert ks and sup
    return int(ks.group(1)) * int(sup.group(1))


def range_begin(c, total, G):
    return c * total // G


def pieces_of(c, problems, total, G):
    """The pieces of CTA c's range: (problem, row block, first superblock, count)."""
    out = []
    g, end = range_begin(c, total, G), range_begin(c + 1, total, G)
    while g < end:
        p = 0
        while p + 1 < len(problems) and g >= problems[p + 1]["sb_base"]:
            p += 1
        a = problems[p]
        off = g - a["sb_base"]
        rb, sb0 = divmod(off, a["nsb"])
        n = min(a["nsb"] - sb0, end - g)
        out.append((p, rb, sb0, n))
        g += n
    return out


def check(shapes, sms):
    sk = superblock_k()
    problems, total = [], 0
    for (N, K) in shapes:
        nrb, nsb = -(-N // 128), K // sk
        problems.append(dict(nrb=nrb, nsb=nsb, sb_base=total))
        total += nrb * nsb
    G = min(sms, total)
    covered = {}
    writers, readers = {}, {}
    for c in range(G):
        ps = pieces_of(c, problems, total, G)
        assert ps, f"CTA {c} has an empty range"
        for idx, (p, rb, sb0, n) in enumerate(ps):
            a = problems[p]
            assert rb < a["nrb"] and n >= 1
            for s in range(sb0, sb0 + n):
                key = (p, rb, s)
                assert key not in covered, f"superblock {key} in CTAs {covered[key]} and {c}"
                covered[key] = c
            if sb0 == 0 and n == a["nsb"]:
                continue
            if sb0 > 0:
                assert idx == 0, f"CTA {c}: a later part that is not its first piece"
                writers[c] = (p, rb)
            else:
                assert idx == len(ps) - 1, f"CTA {c}: a first part that is not its last piece"
                unit_end = a["sb_base"] + (rb + 1) * a["nsb"]
                j = c + 1
                while j < G and range_begin(j, total, G) < unit_end:
                    assert j not in readers, f"the partial of CTA {j} is read twice"
                    readers[j] = (p, rb)
                    j += 1
                assert j > c + 1, f"CTA {c}: a first part with nobody to wait for"
    assert len(covered) == total
    assert writers == readers, "a partial written but never read, or read but never written"
    return G, total, len(writers)


def test_the_four_qwen3_8b_projections():
    shapes = [(4096, 4096), (1024, 4096), (12288, 4096), (4096, 12288)]  # (N, K)
    G, total, cut = check(shapes, 152)
    assert (G, total) == (152, 3712) and cut > 0
    for sms in (148, 132, 100, 8, 1):
        check(shapes, sms)


def test_random_groups_and_grids():
    rng = random.Random(5)
    sk = superblock_k()
    for _ in range(3000):
        n = rng.randint(2, 8)
        shapes = [(rng.randint(1, 20000), sk * rng.choice([1, 2, 3, 16, 48, rng.randint(1, 200)])) for _ in range(n)]
        check(shapes, rng.choice([152, 148, 132, 17, 7, 2, 1]))


def test_more_ctas_than_superblocks_leaves_none_empty():
    # tiny groups: the grid is min(SMs, superblocks), so every range holds a superblock
    sk = superblock_k()
    G, total, _ = check([(1, sk), (130, sk)], 152)
    assert G == total == 3
