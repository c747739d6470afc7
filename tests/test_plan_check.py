"""Whole-plan validation on the host (no GPU needed): kda_plan_check accepts every
plan the planner makes and rejects any plan whose words differ from what the
planner gives for its own bounds -- a changed word in any section, with or
without its checksum re-stamped, changed counts, offsets or lengths -- and the
entry points refuse such plans before any device work is enqueued.

The checksum word follows the rule stated in include/kda.h; the independent
Python planner computes it too, and the two agree on every workload."""
import ctypes

import numpy as np
import pytest

from context_kda_gb300.inputs import workloads
from oracle.plan import CHECKSUM_WORD, checksum, plan_segments


@pytest.fixture(scope="module")
def kda():
    import __graft_entry__
    __graft_entry__._load_build_module().build()
    from context_kda_gb300 import binding
    return binding


def _cu(seqlens):
    return [0] + [int(x) for x in np.cumsum(seqlens)]


def _restamp(words):
    w = np.array(words, dtype=np.int32)
    w[CHECKSUM_WORD] = checksum(w.tolist())
    return w


@pytest.mark.parametrize("name", list(workloads().keys()))
def test_every_workload_plan_passes(kda, name):
    w = workloads()[name]
    plan = kda.kda_plan_segments(_cu(w.seqlens), w.segments)
    assert kda.kda_plan_check(plan) == kda.KDA_OK
    assert int(plan[CHECKSUM_WORD]) == checksum(plan.tolist())


def test_checksum_ignores_its_own_word_and_sees_every_other():
    words = list(range(40))
    base = checksum(words)
    w2 = list(words)
    w2[CHECKSUM_WORD] = 12345
    assert checksum(w2) == base
    for i in (0, 21, 23, 39):
        w3 = list(words)
        w3[i] += 1
        assert checksum(w3) != base


def _sections(plan):
    off = [int(plan[14 + i]) for i in range(8)] + [int(plan[2])]
    return [(off[i], off[i + 1]) for i in range(8)]


def test_any_changed_word_is_rejected(kda):
    rng = np.random.default_rng(5)
    cases = [([0, 100, 300, 301, 640], 5), ([0, 1000], 3), ([0, 64, 128, 700], 4), ([0, 2048], 1)]
    for cu, S in cases:
        plan = kda.kda_plan_segments(cu, S)
        assert kda.kda_plan_check(plan) == kda.KDA_OK
        for lo, hi in _sections(plan):
            if hi <= lo:
                continue
            for _ in range(6):
                i = int(rng.integers(lo, hi))
                bad = plan.copy()
                bad[i] += int(rng.choice([-2, -1, 1, 3]))
                # the checksum catches the edit; with the checksum re-stamped, re-planning does
                assert kda.kda_plan_check(bad) == kda.KDA_ERR_INVALID_ARG, (cu, S, i)
                assert kda.kda_plan_check(_restamp(bad)) == kda.KDA_ERR_INVALID_ARG, (cu, S, i)
        for i in list(range(0, 14)) + list(range(14, 22)) + [23, 31]:   # header words
            bad = plan.copy()
            bad[i] += 1
            assert kda.kda_plan_check(_restamp(bad)) == kda.KDA_ERR_INVALID_ARG, (cu, S, i)


def test_items_in_another_order_are_rejected(kda):
    plan = kda.kda_plan_segments([0, 100, 300, 301, 640], 5)
    lo, hi = _sections(plan)[4]
    items = plan[lo:hi].reshape(-1, 2)[::-1].copy()
    bad = plan.copy()
    bad[lo:hi] = items.reshape(-1)
    assert kda.kda_plan_check(_restamp(bad)) == kda.KDA_ERR_INVALID_ARG


def test_other_plans_with_restamped_header_are_rejected(kda):
    """A plan of one problem whose header claims another problem's sizes."""
    a = kda.kda_plan_segments([0, 500, 1000], 4)
    b = kda.kda_plan_segments([0, 300, 1000], 4)
    mixed = a.copy()
    mixed[:32] = b[:32]
    assert kda.kda_plan_check(_restamp(mixed)) == kda.KDA_ERR_INVALID_ARG


def test_entry_points_refuse_a_changed_plan_before_device_work(kda):
    lib = kda._lib
    plan = kda.kda_plan_segments([0, 100, 300, 301, 640], 5)
    lo, hi = _sections(plan)[3]          # a piece length
    bad = _restamp(np.concatenate([plan[:lo + 1], [plan[lo + 1] + 1], plan[lo + 2:]]))
    with pytest.raises(kda.KDAError) as e:
        kda.kda_workspace_layout(bad, 2)
    assert e.value.status == kda.KDA_ERR_INVALID_ARG
    assert kda.kda_workspace_bytes(bad, 2) == 0
    pp = bad.ctypes.data_as(ctypes.c_void_p)
    fake = ctypes.c_void_p(1 << 20)      # never dereferenced: validation fails first
    ws = 1 << 40
    assert lib.kda_forward_segmented(pp, fake, 2, fake, fake, fake, fake, fake, None, ctypes.c_float(1.0), fake,
                                     fake, fake, ws, None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_forward_two_pass(pp, fake, 2, fake, fake, fake, fake, fake, None, ctypes.c_float(1.0), fake,
                                    fake, fake, ws, None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_compose_summaries(pp, fake, 2, fake, fake, None, fake, None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_apply_boundary(pp, fake, 2, fake, fake, ws, fake, fake, None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_forward_segmented_noalloc(pp, fake, 2, fake, fake, fake, fake, fake, None, ctypes.c_float(1.0),
                                             fake, fake, None) == kda.KDA_ERR_INVALID_ARG


def test_python_planner_writes_the_same_checksum(kda):
    rng = np.random.default_rng(11)
    for _ in range(50):
        n = int(rng.integers(1, 6))
        lens = rng.integers(1, 400, size=n)
        cu = _cu(lens)
        S = int(rng.integers(1, min(cu[-1], 9) + 1))
        got = kda.kda_plan_segments(cu, S)
        want = np.array(plan_segments(cu, S), dtype=np.int32)
        assert np.array_equal(got, want)
        assert kda.kda_plan_check(got) == kda.KDA_OK


# ---- the chunk-level split within a segment (kda_plan_segments_refined)

@pytest.mark.parametrize("cu,S,H,sms", [([0, 131072], 1, 2, 152), ([0, 8192], 4, 16, 152), ([0, 1024], 2, 4, 152),
                                         ([0, 300, 5000, 9000], 3, 1, 152), ([0, 4000], 2, 1, 8),
                                         ([0, 100], 1, 1, 152)])
def test_refined_plan_refines_on_the_chunk_grid(kda, cu, S, H, sms):
    base = kda.kda_plan_segments(cu, S)
    ref = kda.kda_plan_segments_refined(cu, S, H, sms)
    assert kda.kda_plan_check(ref) == kda.KDA_OK
    Sb, Sr = int(base[5]), int(ref[5])
    bb = [int(x) for x in base[int(base[14]):int(base[14]) + Sb + 1]]
    br = [int(x) for x in ref[int(ref[14]):int(ref[14]) + Sr + 1]]
    assert set(bb) <= set(br)                                  # a refinement of the caller's segments
    chunks = min((bb[j + 1] - bb[j]) // 64 for j in range(Sb))
    m = max(1, min(sms // (2 * H * Sb), chunks // 4))
    assert Sr <= Sb * m and (m == 1) == (Sr == Sb)
    for j in range(Sb):                                        # cuts on the 64-token grid of each segment
        for x in br:
            if bb[j] < x < bb[j + 1]:
                assert (x - bb[j]) % 64 == 0
    # the refined plan is the ordinary plan of its bounds, word for word
    assert np.array_equal(ref, np.array(plan_segments(cu, Sr, br), dtype=np.int32))


def test_refined_plan_rejects_what_the_planner_rejects(kda):
    with pytest.raises(kda.KDAError):
        kda.kda_plan_segments_refined([0, 10, 10], 1, 2, 152)        # zero-length sequence
    with pytest.raises(kda.KDAError):
        kda.kda_plan_segments_refined([0, 100], 1, 0, 152)           # no heads
