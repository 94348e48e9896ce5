"""Host model of the forward's softmax turns at D = 128 (no GPU).

In the 128-column forward kernel the two query tiles' softmax warps that share
a sub-partition take turns on its special-function unit: tile 0's step j, then
tile 1's step j, for the first n_pair = min(n_0, n_1) steps.  Each tile t owns
one count-1 mbarrier ``turn[t]``; before the tanh / ex2 loops of a paired step
j it waits on ``turn[t]`` with parity (j + t - 1) & 1 (tile 0 skips the wait at
j = 0), and after them it arrives on ``turn[1 - t]``.

An mbarrier parity wait only sees the low bit of the completed-phase count, so
the protocol is correct only if, whenever a wait is made, the count is the one
the wait needs or one short of it (never two ahead).  The model explores every
interleaving of the two warps for small step counts and checks that:

- both warps finish (no wait is left unsatisfied);
- no wait is satisfied by a phase count other than the intended one;
- the paired sections never overlap and run in the order 0, 1, 0, 1, ...

Two planted mistakes (tile 1 not waiting; pairing the longer tile's steps
too) must be caught.  A last check reads the kernel source so that the modelled
parities and gating cannot drift from the code.
"""
import functools
import os
import re

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "relation_token_mixing_gb300", "csrc")


def _program(t, n_t, n_pair, tile1_waits=True):
    """Actions of tile t's warp: ('wait', parity, needed) / ('enter', j) / ('exit', j) / ('arrive',)."""
    prog = []
    for j in range(n_t):
        paired = j < n_pair
        if paired and j + t > 0 and (t == 0 or tile1_waits):
            prog.append(("wait", (j + t - 1) & 1, j + t))
        prog.append(("enter", j, paired))
        prog.append(("exit", j, paired))
        if paired:
            prog.append(("arrive",))
    return tuple(prog)


def _explore(n0, n1, n_pair, tile1_waits=True):
    """Returns the list of protocol violations found over all interleavings."""
    progs = (_program(0, n0, n_pair, tile1_waits), _program(1, n1, n_pair, tile1_waits))
    problems = set()

    @functools.lru_cache(maxsize=None)
    def step(pc0, pc1, done0, done1, inside, order):
        # done[t]: completed phases of turn[t]; inside: tile in a paired section or -1;
        # order: tiles of the paired sections entered so far (last few only).
        pcs, done = (pc0, pc1), (done0, done1)
        if pc0 == len(progs[0]) and pc1 == len(progs[1]):
            return
        moved = False
        for w in (0, 1):
            if pcs[w] == len(progs[w]):
                continue
            act = progs[w][pcs[w]]
            npc = list(pcs)
            npc[w] += 1
            ndone = list(done)
            ninside, norder = inside, order
            if act[0] == "wait":
                parity, needed = act[1], act[2]
                if (done[w] & 1) == parity:  # try_wait.parity: not yet complete
                    continue
                if done[w] != needed:
                    problems.add(f"tile {w} wait satisfied at phase count {done[w]}, needs {needed}")
            elif act[0] == "enter" and act[2]:
                if inside >= 0:
                    problems.add("paired sections overlap")
                if order and order[-1] == w:
                    problems.add("paired sections out of turn")
                if not order and w != 0:
                    problems.add("tile 1 took the first turn")
                ninside, norder = w, (order + (w,))[-2:]
            elif act[0] == "exit" and act[2]:
                ninside = -1
            elif act[0] == "arrive":
                ndone[1 - w] += 1
            moved = True
            step(npc[0], npc[1], ndone[0], ndone[1], ninside, norder)
        if not moved:
            problems.add(f"deadlock at pcs {pcs}")

    step(0, 0, 0, 0, -1, ())
    return sorted(problems)


STEP_COUNTS = [(0, 0), (0, 1), (1, 1), (1, 2), (2, 3), (3, 4), (3, 3), (4, 4), (2, 0)]


def test_turns_alternate_without_aliasing_or_deadlock():
    for n0, n1 in STEP_COUNTS:
        assert _explore(n0, n1, min(n0, n1)) == [], (n0, n1)


def test_planted_mistakes_are_caught():
    # Tile 1 entering its paired sections without waiting: sections overlap.
    assert any("overlap" in p or "out of turn" in p for p in _explore(3, 4, 3, tile1_waits=False))
    # Pairing the longer tile's extra step: its wait is never satisfied.
    assert any("deadlock" in p for p in _explore(3, 4, 4))


def test_kernel_source_matches_the_model():
    src = open(os.path.join(CSRC, "fwd_tc.cu")).read()
    # n_pair is min(n_0, n_1) for the 128-column kernel and 0 (no turns) at D = 64.
    assert re.search(r"n_pair\s*=\s*C::kSepP\s*\?\s*0\s*:\s*min\(n_t\[0\],\s*n_t\[1\]\)", src)
    # The wait: paired steps other than tile 0's first, parity (j + t - 1) & 1 on the tile's own barrier.
    assert re.search(r"j < n_pair && j \+ t > 0 &&\s*!ptx::mbar_wait_warp\(turn_mine, \(j \+ t - 1\) & 1", src)
    # The pass: one arrival by lane 0 on the other tile's barrier after each paired step's loops.
    assert re.search(r"if \(j < n_pair && lane == 0\) ptx::mbar_arrive\(turn_next\);", src)
    assert "turn_mine = &bars->turn[t][quarter]" in src and "turn_next = &bars->turn[t ^ 1][quarter]" in src
    assert re.search(r"mbar_init\(&bars->turn\[t\]\[q\], 1\)", src)
