"""Host-side checks of the balanced schedule of the K = V = 128 tensor-core forward.

With more (batch, head) pairs than resident thread blocks, the pairs' steps are laid end to
end (pair p owns positions [p T, (p+1) T)) and every block takes an equal stretch.  A pair
cut by a stretch boundary runs its first steps at the start of the later block's stretch
and its last steps at the end of the earlier block's stretch; the state passes between them
through the pair's own y rows, so the earlier block must run at least 129 of its steps.
Rows of H and pairs are independent (the M²RNN notes, Sec. 1.2 and 2.6), so this
reordering leaves every result bit for bit unchanged; these checks cover the arithmetic
of the schedule itself, without a GPU.
"""
import pytest

import __graft_entry__
from matrix_state_nonlinear_gb300 import m2rnn as binding

HANDOFF_ROWS = 129


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return binding.load_library()


def segments(pairs, T, workers):
    """Per block, its (pair, first step, end step, kind) in the order the block runs them."""
    out = []
    for w in range(workers):
        s, e = binding.balanced_stretch(pairs, T, workers, w)
        segs = []
        p = s // T
        while p * T < e:
            lo = max(s, p * T) - p * T
            hi = min(e, (p + 1) * T) - p * T
            if lo > 0:
                segs.append((p, 0, T - lo, "first"))
            elif hi < T:
                segs.append((p, T - hi, T, "last"))
            else:
                segs.append((p, 0, T, "whole"))
            p += 1
        out.append((s, e, segs))
    return out


CASES = [(512, 8192, 304), (360, 300, 304), (305, 1000, 304), (400, 100, 304), (1000, 129, 304),
         (1000, 130, 304), (1000, 258, 304), (7, 500, 3), (304, 8192, 304), (608, 8192, 304),
         (1, 5, 1), (5, 1, 2), (153, 20000, 152)]


@pytest.mark.parametrize("pairs,T,workers", CASES)
def test_stretches_partition_the_line(lib, pairs, T, workers):
    line = -(-pairs * T // workers)
    sched = segments(pairs, T, workers)
    assert sched[0][0] == 0 and sched[-1][1] == pairs * T
    for (s0, e0, _), (s1, _, _) in zip(sched, sched[1:]):
        assert e0 == s1 and s0 <= e0
    for s, e, _ in sched:
        assert e - s <= line + HANDOFF_ROWS - 1     # the schedule's length, up to one handoff


@pytest.mark.parametrize("pairs,T,workers", CASES)
def test_every_step_of_every_pair_runs_once(lib, pairs, T, workers):
    covered = {}
    for _, _, segs in segments(pairs, T, workers):
        kinds = [k for _, _, _, k in segs]
        # a cut pair's first steps open a block's stretch, its last steps close one
        assert kinds.count("first") <= 1 and kinds.count("last") <= 1
        if "first" in kinds:
            assert kinds[0] == "first"
        if "last" in kinds:
            assert kinds[-1] == "last"
        for p, t0, t1, kind in segs:
            assert 0 <= t0 < t1 <= T
            covered.setdefault(p, []).append((t0, t1, kind))
    assert sorted(covered) == list(range(pairs))
    for p, parts in covered.items():
        parts.sort()
        assert parts[0][0] == 0 and parts[-1][1] == T
        for (a0, a1, _), (b0, _, _) in zip(parts, parts[1:]):
            assert a1 == b0
        assert len(parts) <= 2
        if len(parts) == 2:
            assert parts[0][2] == "first" and parts[1][2] == "last"
            assert T - parts[1][0] >= HANDOFF_ROWS  # room for the state and its ready word


@pytest.mark.parametrize("pairs,T,workers", CASES)
def test_handed_off_state_is_ready_before_it_is_needed(lib, pairs, T, workers):
    """At equal step rates, a cut pair's first steps end (the later block's step T - r)
    no later than the earlier block reaches its last steps, so no block waits."""
    sched = segments(pairs, T, workers)
    first_end = {}
    for s, _, segs in sched:
        if segs and segs[0][3] == "first":
            first_end[segs[0][0]] = segs[0][2] - segs[0][1]
    for s, e, segs in sched:
        if segs and segs[-1][3] == "last":
            p, t0, t1, _ = segs[-1]
            start = sum(b - a for _, a, b, _ in segs[:-1])   # steps this block runs before it
            assert start >= first_end[p], (p, start, first_end[p])


def test_no_cut_when_pairs_fit_or_divide(lib):
    for pairs, T, workers in [(304, 8192, 304), (608, 8192, 304), (400, 100, 304)]:
        for _, _, segs in segments(pairs, T, workers):
            assert all(kind == "whole" for *_, kind in segs)


def test_headline_wide_workload_balances(lib):
    """B=16, N=32 (512 pairs), T=8192 on 304 resident blocks: 1.68 pairs of steps per block
    instead of two whole pairs on the busiest block."""
    lengths = [e - s for s, e, _ in segments(512, 8192, 304)]
    assert max(lengths) <= -(-512 * 8192 // 304) + HANDOFF_ROWS - 1
    assert max(lengths) < 2 * 8192 * 0.85


@pytest.mark.parametrize("args", [(0, 5, 1, 0), (3, 0, 1, 0), (3, 5, 0, 0), (3, 5, 2, 2),
                                  (3, 5, 2, -1)])
def test_invalid_schedule_arguments(lib, args):
    with pytest.raises(ValueError):
        binding.balanced_stretch(*args)
