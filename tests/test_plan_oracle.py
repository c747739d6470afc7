"""Pins for the independent Python planner (test infrastructure).

The plan is checked against a brute-force per-token labelling: every token
gets its sequence and segment by linear search, and the plan's pieces, flags,
continuing rows and chunks must agree with that labelling.  Rules follow
cuLA PR #136 ("feat(kda): add cuDNN concatenated-summary Kimi CP",
§Walkthrough: balanced or custom contiguous shards, validated against
sequence boundaries, rank spans and invalid inputs).
"""
import numpy as np
import pytest

from context_kda_gb300.inputs import workloads
from oracle.plan import (CONT, FIRST, SEG_HAS_RESET, SEG_LAST, SEG_STARTS_SEQ, SEQ_END, PlanError,
                         decode, plan_segments)


def _labels(cu, bounds):
    T = cu[-1]
    seq = np.empty(T, dtype=np.int64)
    seg = np.empty(T, dtype=np.int64)
    for t in range(T):
        seq[t] = next(s for s in range(len(cu) - 1) if cu[s] <= t < cu[s + 1])
        seg[t] = next(j for j in range(len(bounds) - 1) if bounds[j] <= t < bounds[j + 1])
    return seq, seg


def check_plan_against_labels(cu, S, bounds=None):
    words = plan_segments(cu, S, bounds)
    d = decode(words)
    b = d["seg_bounds"]
    if bounds is None:
        T = cu[-1]
        assert b == [(j * T) // S for j in range(S + 1)]
    seq, seg = _labels(cu, b)
    T = cu[-1]
    covered = np.zeros(T, dtype=np.int64)
    starts = set(cu[:-1])
    for i, (st, ln, s, j, fl, ci, row, fi) in enumerate(d["pieces"]):
        assert ln > 0
        covered[st:st + ln] += 1
        assert np.all(seq[st:st + ln] == s) and np.all(seg[st:st + ln] == j)
        # a piece is maximal: the token before it and after it change sequence or segment
        if st > 0:
            assert seq[st - 1] != s or seg[st - 1] != j
        if st + ln < T:
            assert seq[st + ln] != s or seg[st + ln] != j
        assert bool(fl & FIRST) == (st == cu[s])
        assert bool(fl & CONT) == (st != cu[s])
        assert bool(fl & SEG_LAST) == (st + ln == b[j + 1])
        assert bool(fl & SEQ_END) == (st + ln == cu[s + 1])
        if fl & CONT:
            assert st == b[j] and ci >= 0 and d["cont"][ci][0] == i and d["cont"][ci][2] == row
        else:
            assert ci == -1 and row == -1
        assert (fi >= 0) == bool((fl & CONT) and (fl & SEQ_END))
    assert np.all(covered == 1)
    for j, (s0, fl, fp, npc) in enumerate(d["segs"]):
        assert s0 == seq[b[j]]
        assert bool(fl & SEG_STARTS_SEQ) == (b[j] in starts)
        assert bool(fl & SEG_HAS_RESET) == any(b[j] <= c < b[j + 1] for c in starts)
        assert all(d["pieces"][p][3] == j for p in range(fp, fp + npc))
    # continuing rows are the running sum of continuing lengths
    row = 0
    for c in d["cont"]:
        assert c[2] == row
        row += c[3]
    assert d["T_cont"] == row
    # chunks tile each piece in steps of C from its start
    per_piece = {}
    for (p, st, ln, ix) in d["chunks"]:
        assert 0 < ln <= 64
        per_piece.setdefault(p, []).append((ix, st, ln))
    for i, pc in enumerate(d["pieces"]):
        got = sorted(per_piece[i])
        assert [x[0] for x in got] == list(range(len(got)))
        assert got[0][1] == pc[0] and sum(x[2] for x in got) == pc[1]
        assert all(x[2] == 64 for x in got[:-1])
    # items: a state item for every piece, a transition item for every continuing piece
    kinds = sorted((p, k) for p, k in d["items"])
    want = sorted([(i, 0) for i in range(len(d["pieces"]))] +
                  [(i, 1) for i, p in enumerate(d["pieces"]) if p[4] & CONT])
    assert kinds == want
    lens = [d["pieces"][p][1] for p, _ in d["items"]]
    assert lens == sorted(lens, reverse=True)
    return d


@pytest.mark.parametrize("name", ["t1024_h4_s2", "t4096_h8_s4", "t8192_h16_s4", "packed65536_h32_s64"])
def test_workload_plans(name):
    w = workloads()[name]
    cu = [0] + list(np.cumsum(w.seqlens))
    d = check_plan_against_labels([int(x) for x in cu], w.segments)
    if name == "packed65536_h32_s64":
        assert d["T"] == 65536 and len(w.seqlens) == 24


def test_random_varlen_plans():
    rng = np.random.default_rng(0)
    for trial in range(40):
        n = int(rng.integers(1, 8))
        lens = [int(x) for x in rng.integers(1, 200, size=n)]
        cu = [0] + list(np.cumsum(lens))
        T = cu[-1]
        S = int(rng.integers(1, min(T, 12) + 1))
        check_plan_against_labels([int(x) for x in cu], S)
        if T >= 3:
            inner = sorted(set(int(x) for x in rng.integers(1, T, size=int(rng.integers(1, 5)))))
            bounds = [0] + inner + [T]
            check_plan_against_labels([int(x) for x in cu], len(bounds) - 1, bounds)


def test_single_segment_and_one_token_segments():
    check_plan_against_labels([0, 5, 9], 1)
    check_plan_against_labels([0, 5, 9], 9)


@pytest.mark.parametrize("cu,S,bounds,code", [
    ([0], 1, None, "invalid"),
    ([1, 5], 1, None, "invalid"),
    ([0, 5, 5], 1, None, "invalid"),
    ([0, 4], 5, None, "invalid"),
    ([0, 4], 0, None, "invalid"),
    ([0, 8], 2, [0, 4, 7], "invalid"),
    ([0, 8], 2, [0, 9, 8], "invalid"),
    ([0, 8], 2, [0, 4, 4], "invalid"),
    ([0, 8], 3, [0, 4, 8], "invalid"),
])
def test_invalid_inputs(cu, S, bounds, code):
    with pytest.raises(PlanError) as e:
        plan_segments(cu, S, bounds)
    assert e.value.code == code


def test_chunk_other_than_64_is_unsupported():
    with pytest.raises(PlanError) as e:
        plan_segments([0, 128], 2, None, chunk=32)
    assert e.value.code == "unsupported"
