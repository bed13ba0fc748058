"""The wrap-around schedule of srwm_forward_balanced (d = 32), checked on the
host through the library's own schedule functions (no GPU needed).

The schedule lays every stream's T steps end to end and gives each warp slot
an equal range of them, taken last piece first.  These tests check what makes
it correct and fast: every (stream, step) is covered exactly once, a stream
is split at most once, its first part is the first piece of one slot and its
last part the last piece of the next slot, so the second part normally starts
after the first has finished.
"""
import pytest

from self_referential_weight_gb300 import binding

CASES = [
    (2048, 512, 1824, 16),   # rl on a 152-SM GB300: 512 x 4 streams, 12 warp slots per SM
    (1852, 70, 1824, 16),    # ragged T: splits fall inside TMA chunks
    (2049, 33, 2048, 16),
    (5, 1000, 3, 16),
    (100, 7, 30, 16),
    (97, 1, 13, 16),         # one-step streams: never split
    (64, 48, 63, 16),
]


def pieces_of(n, T, C, slots):
    return [binding.srwm_debug_wrap_pieces(n, T, C, k) for k in range(slots)]


@pytest.mark.parametrize("n,T,slots,tau", CASES)
def test_wrap_len(n, T, slots, tau):
    C = binding.srwm_debug_wrap_len(n, T, slots, tau)
    assert C % tau == 0 and C >= T
    assert C * slots >= n * T
    assert (C - tau) * slots < n * T   # no whole chunk more than needed


def test_wrap_len_not_used():
    assert binding.srwm_debug_wrap_len(1824, 512, 1824, 16) == 0   # every stream has a slot
    assert binding.srwm_debug_wrap_len(10, 0, 3, 16) == 0
    assert binding.srwm_debug_wrap_len(10, 5, 0, 16) == 0


@pytest.mark.parametrize("n,T,slots,tau", CASES)
def test_wrap_pieces_cover_every_step_once(n, T, slots, tau):
    C = binding.srwm_debug_wrap_len(n, T, slots, tau)
    seen = [[] for _ in range(n)]
    for k, pcs in enumerate(pieces_of(n, T, C, slots)):
        assert sum(p[3] for p in pcs) <= C
        for (p, seg, t0, ln) in pcs:
            assert 0 <= p < n and ln > 0 and 0 <= t0 and t0 + ln <= T
            seen[p].append((t0, ln, seg, k))
    for p in range(n):
        parts = sorted(seen[p])
        assert parts[0][0] == 0 and len(parts) <= 2
        assert sum(ln for (_, ln, _, _) in parts) == T
        for i, (t0, ln, seg, _) in enumerate(parts):
            assert seg == i
            if i:
                assert t0 == parts[i - 1][0] + parts[i - 1][1]


@pytest.mark.parametrize("n,T,slots,tau", CASES)
def test_wrap_split_streams_run_in_order(n, T, slots, tau):
    """A split stream's first part opens its slot's run order and its last
    part closes the next slot's, so with equal speed per step the last part
    starts no earlier than the first ends (slots with at least T steps)."""
    C = binding.srwm_debug_wrap_len(n, T, slots, tau)
    all_pcs = pieces_of(n, T, C, slots)
    where = {}
    for k, pcs in enumerate(all_pcs):
        start = 0
        for i, (p, seg, t0, ln) in enumerate(pcs):
            where[(p, seg)] = (k, i, start, ln, len(pcs), sum(q[3] for q in pcs))
            start += ln
    for (p, seg), (k, i, start, ln, npc, total) in where.items():
        if seg == 1:
            k0, i0, start0, ln0, _, _ = where[(p, 0)]
            assert k == k0 + 1
            assert i0 == 0 and i == npc - 1
            if total >= T:
                assert start >= start0 + ln0


def test_wrap_pieces_invalid_arguments():
    with pytest.raises(binding.SrwmError):
        binding.srwm_debug_wrap_pieces(10, 5, 4, 0)   # range shorter than a stream
    with pytest.raises(binding.SrwmError):
        binding.srwm_debug_wrap_pieces(0, 5, 8, 0)
    assert binding.srwm_debug_wrap_pieces(10, 5, 8, 7) == []   # past the last position


# ---------------------------------------------------------------- host pipeline chunk plan

def longest_chunk(T, d):
    """Where the recurrence sets the pace (d = 64) chunks grow to 256 steps, or
    T / 8 for longer sequences; where the host copies do (d <= 32), to 64."""
    return 64 if d <= 32 else max(256, T // 8)


@pytest.mark.parametrize("d", [16, 32, 64])
@pytest.mark.parametrize("T", [0, 1, 31, 63, 64, 65, 75, 95, 96, 200, 512, 1024, 1500, 2056, 8192])
def test_chunk_plan_doubling(T, d):
    """chunk_steps <= 0: chunks double from 32 steps up to at most half the
    longest chunk and halve again at the end, the middle split evenly into
    chunks of at most the longest; they cover the T steps in order.  Short
    first and last chunks keep the copies that nothing overlaps short."""
    plan = binding.srwm_debug_chunk_plan(T, d, 0)
    assert sum(plan) == T and all(c > 0 for c in plan)
    if T == 0:
        assert plan == []
        return
    assert max(plan) <= longest_chunk(T, d)
    ramp = 0
    while ramp < len(plan) // 2 and plan[ramp] == 32 << ramp and plan[-1 - ramp] == 32 << ramp:
        ramp += 1
    mid = plan[ramp:len(plan) - ramp]
    assert not mid or max(mid) - min(mid) <= 1   # the middle split evenly
    if T >= 96:   # room for a 32-step chunk at both ends and as much between them
        assert plan[0] == 32 and plan[-1] == 32
    else:         # no ramp: T split evenly into as few chunks as the longest allows
        assert len(plan) == -(-T // longest_chunk(T, d)) and max(plan) - min(plan) <= 1


def test_chunk_plan_by_width():
    assert binding.srwm_debug_chunk_plan(512, 32, 0) == [32] + [64] * 7 + [32]          # rl
    assert binding.srwm_debug_chunk_plan(1024, 64, 0) == [32, 64, 128, 192, 192, 192, 128, 64, 32]   # mid
    assert binding.srwm_debug_chunk_plan(26, 16, 0) == [26]                              # few-shot


@pytest.mark.parametrize("d", [16, 64])
def test_chunk_plan_rises_then_falls(d):
    """chunk_steps <= 0: over every length up to 4,096 steps (and some longer
    ones) the chunks never shrink and then grow again, so a chunk whose copies
    nothing overlaps is never in the middle of the call."""
    for T in list(range(1, 4097)) + [6000, 8192, 10000, 65536]:
        plan = binding.srwm_debug_chunk_plan(T, d, 0)
        assert sum(plan) == T
        top = plan.index(max(plan))
        assert all(a <= b for a, b in zip(plan[:top], plan[1:top + 1])), (T, plan)
        assert all(a >= b for a, b in zip(plan[top:], plan[top + 1:])), (T, plan)


@pytest.mark.parametrize("T,c", [(75, 32), (64, 64), (100, 1), (5, 128)])
def test_chunk_plan_fixed(T, c):
    plan = binding.srwm_debug_chunk_plan(T, 64, c)
    assert sum(plan) == T and all(v == c for v in plan[:-1]) and 0 < plan[-1] <= c
