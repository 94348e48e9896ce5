"""Host model of the dP1 reduce warps' per-tile decision (no GPU).

Both tensor-core backward kernels drain the dP1 partial with four warps that
meet twice per 32-column panel at named barrier 1 (``bar.sync 1, 128``), which
has no time limit.  Each tile starts with a bounded wait on the MMA's
``dq_full`` barrier; after another role's wait has expired (abort), that wait
can succeed for one warp and give up for another.  If each warp decided alone,
the warp that left would never reach the next ``bar.sync 1, 128`` and the other
three would wait there forever: the CTA would never return.  The kernels
therefore take the decision as one 128-thread vote on barrier 1
(``barrier.cta.red.and.pred``): all four warps stay or all four leave.

The model enumerates every pattern of wait results over a few tiles and checks
that every instance of barrier 1 is reached by all four warps.  A planted
mistake (per-warp decisions) must produce a hang in the model.  A second check
reads the kernel sources and requires the vote before the reduce loop's named
barriers, so the fix cannot silently disappear.
"""
import itertools
import os
import re

WARPS = 4
PANELS = {"bwd_tc64.cu": 2, "bwd_tc.cu": 4}  # 32-column panels per tile (d_h 64; d_h 80/128)
CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "relation_token_mixing_gb300", "csrc")


def _barrier_sequences(ok, panels, vote):
    """Barrier-1 instructions each warp executes, given wait results ok[warp][tile]."""
    seqs = [[] for _ in range(WARPS)]
    tiles = len(ok[0])
    alive = [True] * WARPS
    for t in range(tiles):
        if vote:
            for w in range(WARPS):
                seqs[w].append("vote")
            stay = all(ok[w][t] for w in range(WARPS))
            decision = [stay] * WARPS
        else:
            decision = [ok[w][t] for w in range(WARPS)]
        for w in range(WARPS):
            if not alive[w]:
                continue
            if not decision[w]:
                alive[w] = False
                continue
            seqs[w].extend(["bar"] * (2 * panels))
    return seqs


def _completes(seqs):
    """Every instance of barrier 1 completes iff all warps execute the same number of
    barrier-1 instructions (a warp that leaves early strands the others at the next one)."""
    return len({len(s) for s in seqs}) == 1 and all(s == seqs[0] for s in seqs)


def _patterns(tiles):
    for bits in itertools.product([True, False], repeat=WARPS * tiles):
        yield [list(bits[w * tiles:(w + 1) * tiles]) for w in range(WARPS)]


def test_vote_never_strands_a_warp():
    for panels in set(PANELS.values()):
        for tiles in (1, 2, 3):
            for ok in _patterns(tiles):
                assert _completes(_barrier_sequences(ok, panels, vote=True)), (panels, ok)


def test_per_warp_decision_hangs_in_the_model():
    """Planted mistake: the decision each warp took before the vote strands warps."""
    hangs = sum(not _completes(_barrier_sequences(ok, 2, vote=False)) for ok in _patterns(2))
    assert hangs > 0
    # One warp giving up on the first tile while three go on is one such pattern.
    ok = [[False, True], [True, True], [True, True], [True, True]]
    assert not _completes(_barrier_sequences(ok, 2, vote=False))


def _reduce_loop(src):
    start = src.index("dP1 partial reduce")
    end = src.index("__syncthreads", start)
    return src[start:end]


def test_kernels_take_the_decision_by_vote():
    """Every early exit of the reduce loop follows a vote: the per-tile vote itself, and in the
    persistent d_h <= 64 kernel also the flag it sets (leaving the key-tile loop) and the vote on
    the next key tile.  No other break may appear, and the flag is set only where a vote failed."""
    for name in PANELS:
        with open(os.path.join(CSRC, name)) as f:
            loop = _reduce_loop(f.read())
        vote = loop.find("bar_vote_all<1, 128>")
        first_bar = loop.find("bar.sync 1, 128")
        assert vote >= 0 and first_bar > vote, name
        allowed = [
            r"if \(!ptx::bar_vote_all<1, 128>\([^()]*(?:\([^()]*\))?[^()]*\)\) break;",
            r"if \(!ptx::bar_vote_all<1, 128>\(\w+\)\) \{\s*left = true;\s*break;\s*\}",
            r"if \(left\) break;",
        ]
        rest = loop
        for pat in allowed:
            rest = re.sub(pat, "", rest)
        assert not re.findall(r"\bbreak;", rest), name
        assert len(re.findall(r"left = true;", loop)) == len(
            re.findall(r"if \(!ptx::bar_vote_all<1, 128>\(\w+\)\) \{\s*left = true;", loop)), name
        assert re.search(r"if \(!ptx::bar_vote_all<1, 128>\(\w+\)\)", loop), name
