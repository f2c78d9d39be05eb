"""The attention kernel's exponential turn: a model of its named-barrier protocol.

The two query tiles' softmax warpgroups (4 warps each) pass the turn through two hardware named
barriers of 256 threads (8 warps): barrier 1 is tile A's turn, barrier 2 tile B's. A named barrier
has no timeout, so the kernel (attn.cu, the softmax branch of attn_fwd_kernel) makes every warp
run the same sequence of barrier operations on every path:
- per key tile g, tile A syncs on 1 (for g > 0) and arrives on 2; tile B syncs on 2 and arrives
  on 1;
- after its last tile, tile A syncs once more on 1;
- a warp whose bounded mbarrier wait fails (before the turn of tile g: the score wait; after it:
  the PV wait of tile g or the item's final PV wait) stops working but first runs the turn
  operations of the key tiles it has not walked.

This test restates that control flow per warp, injects a failure at every wait site of every
tile in any subset of warps, and simulates bar.sync / bar.arrive: every run must finish with no
warp left waiting and every barrier phase complete.
"""
import itertools

import pytest

BAR_WARPS = 8  # 256 threads


def warp_program(t, n_tiles, fail=None):
    """The barrier operations one softmax warp of tile t (0 = A, 1 = B) executes, in order.

    fail = (g, "before") for a failed score wait at key tile g, (g, "after") for a failed PV
    wait after the turn of tile g, (n_tiles, "end") for a failed final PV wait; None for none."""
    ops = []
    g_turn = 0
    failed = False
    for g in range(n_tiles):
        if fail == (g, "before"):
            failed = True
            break
        if t == 1 or g > 0:
            ops.append(("sync", 1 + t))
        ops.append(("arrive", 2 - t))
        g_turn = g + 1
        if fail == (g, "after"):
            failed = True
            break
    if not failed and fail == (n_tiles, "end"):
        failed = True
    if failed:
        for gg in range(g_turn, n_tiles):
            if t == 1 or gg > 0:
                ops.append(("sync", 1 + t))
            ops.append(("arrive", 2 - t))
    if t == 0:
        ops.append(("sync", 1))
    return ops


def simulate(programs):
    """Run warps' barrier programs to completion under hardware named-barrier semantics (a sync
    blocks until BAR_WARPS warps have arrived or synced on that barrier's current phase; an
    arrive counts and continues). Returns True when every warp finishes and no phase is left
    partial; False on a deadlock."""
    pc = [0] * len(programs)
    count = {1: 0, 2: 0}
    waiting = {1: set(), 2: set()}
    while True:
        progressed = False
        for w, prog in enumerate(programs):
            if pc[w] >= len(prog) or any(w in s for s in waiting.values()):
                continue
            op, bar = prog[pc[w]]
            count[bar] += 1
            if op == "sync":
                waiting[bar].add(w)
            else:
                pc[w] += 1
            if count[bar] == BAR_WARPS:  # the phase completes: release its syncing warps
                for v in waiting[bar]:
                    pc[v] += 1
                waiting[bar].clear()
                count[bar] = 0
            progressed = True
        if not progressed:
            done = all(pc[w] >= len(p) for w, p in enumerate(programs))
            return done and count == {1: 0, 2: 0}


def failure_points(n_tiles):
    pts = [None, (n_tiles, "end")]
    for g in range(n_tiles):
        pts += [(g, "before"), (g, "after")]
    return pts


@pytest.mark.parametrize("n_tiles", [1, 2, 3, 12])
def test_turn_completes_without_failures(n_tiles):
    programs = [warp_program(0, n_tiles) for _ in range(4)] + [warp_program(1, n_tiles) for _ in range(4)]
    assert simulate(programs)


@pytest.mark.parametrize("n_tiles", [1, 2, 3, 5])
def test_turn_completes_whatever_warp_fails_where(n_tiles):
    pts = failure_points(n_tiles)
    # one failing warp of each tile (any point), the others running normally
    for fa, fb in itertools.product(pts, pts):
        programs = ([warp_program(0, n_tiles, fa)] + [warp_program(0, n_tiles) for _ in range(3)] +
                    [warp_program(1, n_tiles, fb)] + [warp_program(1, n_tiles) for _ in range(3)])
        assert simulate(programs), (fa, fb)


def test_turn_completes_with_every_warp_failing_independently():
    n_tiles = 3
    pts = failure_points(n_tiles)
    for combo in itertools.product(pts, repeat=4):  # the four warps of tile A fail anywhere
        programs = [warp_program(0, n_tiles, f) for f in combo] + [warp_program(1, n_tiles, combo[0]) for _ in range(4)]
        assert simulate(programs), combo


def test_model_detects_a_broken_protocol():
    """The simulator is not vacuous: a warp that stops without running its remaining turn
    operations leaves the other tile waiting."""
    n_tiles = 3
    good = [warp_program(0, n_tiles) for _ in range(4)] + [warp_program(1, n_tiles) for _ in range(4)]
    broken = list(good)
    broken[0] = broken[0][:2]  # tile A's first warp leaves after its first turn, skipping the rest
    assert simulate(good)
    assert not simulate(broken)
