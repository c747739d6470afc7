"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle.

Workloads are the seeded synthetic problems of context_kda_gb300.inputs (shapes
of cuLA PR #110, "feat(cp): add opt-in NVSHMEM CP state handoff",
§Correctness / §Performance, and the CP64 packed case of cuLA PR #136,
"feat(kda): add cuDNN concatenated-summary Kimi CP", §Latest cuDNN
compatibility).  Outputs and final states are compared element by element on
every head of the single-sequence workloads, the packed 64-segment workload and
the 32768-token long-context workloads, and A, B and S_in on every (segment,
head) of them; the 131072-token workloads take four heads each (their oracle
run on every head would dominate the suite).  Tolerances are in
tests/harness.py.
"""
import numpy as np
import pytest

from context_kda_gb300.inputs import bf16_to_f32, make_inputs, make_workload, workloads
from harness import (O_TOL, REL_TOL, gpu_forward, oracle_forward, oracle_segment, oracle_summaries, rel_err,
                     to_device)

pytestmark = pytest.mark.gpu


def _check_outputs(res, inp, heads=None, scale=1.0):
    o_ref, f_ref = oracle_forward(inp, heads=heads, scale=scale)
    hs = list(range(inp.heads)) if heads is None else list(heads)
    err = float(np.max(np.abs(res["o"][:, hs] - o_ref[:, hs])))
    frel = rel_err(res["final"][:, hs], f_ref[:, hs])
    assert err <= O_TOL, f"max|o - o_ref| = {err:.3e}"
    assert frel <= REL_TOL, f"final-state rel = {frel:.3e}"
    return err, frel


def _check_segments(res, inp, pairs):
    b = res["bounds"]
    worst = 0.0
    for j, h in pairs:
        A, B, S_in = oracle_segment(inp, b, j, h)
        ea, eb, es = rel_err(res["A"][j, h], A), rel_err(res["B"][j, h], B), rel_err(res["S_in"][j, h], S_in)
        if np.all(A == 0):
            assert np.all(res["A"][j, h] == 0), f"segment {j} head {h}: A must be exactly 0"
        assert max(ea, eb, es) <= REL_TOL, f"segment {j} head {h}: A {ea:.2e} B {eb:.2e} S_in {es:.2e}"
        worst = max(worst, ea, eb, es)
    return worst


@pytest.mark.parametrize("name", ["t1024_h4_s2", "t4096_h8_s4", "t8192_h16_s4"])
def test_single_sequence_workloads_all_heads(name):
    inp = make_workload(workloads()[name])
    res = gpu_forward(inp)
    _check_outputs(res, inp)
    _check_segments(res, inp, [(j, h) for j in range(inp.segments) for h in range(inp.heads)])


def _check_all_segments(res, inp, heads=None):
    """A, B and S_in of every segment of the listed heads (default all) against the oracle."""
    b = res["bounds"]
    A, B, S_in = oracle_summaries(inp, b, heads)
    hs = list(range(inp.heads)) if heads is None else list(heads)
    for h in hs:
        for j in range(len(b) - 1):
            if np.all(A[j, h] == 0):
                assert np.all(res["A"][j, h] == 0), f"segment {j} head {h}: A must be exactly 0"
    worst = max(rel_err(res["A"][:, hs], A[:, hs]), rel_err(res["B"][:, hs], B[:, hs]),
                rel_err(res["S_in"][:, hs], S_in[:, hs]))
    assert worst <= REL_TOL, f"summaries rel = {worst:.3e}"
    return worst


def test_packed_varlen_64_segments_every_head_and_segment():
    inp = make_workload(workloads()["packed65536_h32_s64"])
    res = gpu_forward(inp)
    _check_outputs(res, inp)
    _check_all_segments(res, inp)


@pytest.mark.parametrize("name", ["t32768_h32_s8", "t32768_h32_s64"])
def test_long_context_every_head_and_segment(name):
    inp = make_workload(workloads()[name])
    res = gpu_forward(inp)
    _check_outputs(res, inp)
    _check_all_segments(res, inp)


@pytest.mark.parametrize("name", ["t131072_h32_s8", "t131072_h32_s64"])
def test_long_context_131072_four_heads(name):
    inp = make_workload(workloads()[name])
    res = gpu_forward(inp)
    heads = [0, 5, 17, 31]
    _check_outputs(res, inp, heads=heads)
    _check_all_segments(res, inp, heads=heads)


def test_three_call_path_matches_fused_bitwise():
    inp = make_workload(workloads()["t4096_h8_s4"])
    dev = to_device(inp)
    a = gpu_forward(inp, path="fused", dev=dev)
    b = gpu_forward(inp, path="split", dev=dev)
    for key in ("o_bits", "final", "A", "B", "S_in"):
        assert np.array_equal(a[key], b[key]), key


def test_fresh_launches_are_bitwise_identical():
    """Repeated launches agree exactly (cuLA PR #110 §Correctness: 3/3 fresh launches,
    maximum absolute difference 0.0; fixture tests/golden/pages_correctness_shapes.txt)."""
    inp = make_workload(workloads()["t4096_h8_s4"])
    dev = to_device(inp)
    runs = [gpu_forward(inp, dev=dev) for _ in range(3)]
    for r in runs[1:]:
        for key in ("o_bits", "final", "A", "B", "S_in"):
            assert np.array_equal(r[key], runs[0][key]), key


def test_one_segment_equals_many():
    """The single-rank path (cuLA PR #136 §Summary by CodeRabbit: single-rank execution)
    and the segmented path both match the oracle, and each other within tolerance."""
    inp1 = make_inputs([1000], heads=3, segments=1, h0_std=0.2, seed=3)
    inp7 = make_inputs([1000], heads=3, segments=7, h0_std=0.2, seed=3)
    r1, r7 = gpu_forward(inp1), gpu_forward(inp7)
    _check_outputs(r1, inp1)
    _check_outputs(r7, inp7)
    assert float(np.max(np.abs(r1["o"] - r7["o"]))) <= O_TOL
    assert rel_err(r7["final"], r1["final"]) <= REL_TOL


@pytest.mark.parametrize("seqlens,S,h0_std,scale", [
    ([1], 1, 0.0, 1.0),                        # one token
    ([63, 1, 65, 130], 3, 0.1, 1.0),          # ragged tails, a one-token sequence
    ([200, 201, 50, 9, 300], 5, 0.3, 0.5),    # resets inside segments, continuing pieces ending mid-segment
    ([700], 11, 0.0, 1.0),                     # non-64-aligned cuts
    ([5, 5, 5, 5], 20, 0.1, 1.0),              # one-token segments crossing sequence starts
])
def test_edge_cases_all_heads(seqlens, S, h0_std, scale):
    inp = make_inputs(seqlens, heads=2, segments=S, h0_std=h0_std, seed=11, g_lo=-0.2)
    res = gpu_forward(inp, scale=scale)
    _check_outputs(res, inp, scale=scale)
    _check_segments(res, inp, [(j, h) for j in range(S) for h in range(2)])


def test_long_ragged_pieces_with_few_chains():
    """Few, long pieces of unequal length (ragged last chunks, a one-chunk sequence, continuing
    pieces, chains of very different lengths side by side), every head and segment; a second
    launch gives the same bits."""
    inp = make_inputs([1800, 2300, 63, 1400], heads=4, segments=4, h0_std=0.1, seed=15, g_lo=-0.2)
    res = gpu_forward(inp)
    _check_outputs(res, inp)
    _check_segments(res, inp, [(j, h) for j in range(4) for h in range(4)])
    again = gpu_forward(inp)
    assert np.array_equal(res["o"], again["o"]) and np.array_equal(res["final"], again["final"])


# ---- the forward from preceding summaries (cuLA PR #136 §Summary: the cuDNN KDA forward takes the
# preceding state update and transition as inputs): same results, reached without a fix-up

@pytest.mark.parametrize("name", ["t1024_h4_s2", "t4096_h8_s4"])
def test_two_pass_single_sequence_all_heads(name):
    inp = make_workload(workloads()[name])
    res = gpu_forward(inp, path="two_pass")
    _check_outputs(res, inp)
    _check_segments(res, inp, [(j, h) for j in range(inp.segments) for h in range(inp.heads)])


@pytest.mark.parametrize("seqlens,S,h0_std,scale", [
    ([1], 1, 0.0, 1.0),                        # one token
    ([300, 1, 77], 1, 0.2, 1.0),               # one segment: no continuing piece at all
    ([63, 1, 65, 130], 3, 0.1, 1.0),
    ([200, 201, 50, 9, 300], 5, 0.3, 0.5),
    ([700], 11, 0.0, 1.0),
    ([5, 5, 5, 5], 20, 0.1, 1.0),
    ([1800, 2300, 63, 1400], 4, 0.1, 1.0),
])
def test_two_pass_edge_cases_all_heads(seqlens, S, h0_std, scale):
    inp = make_inputs(seqlens, heads=2, segments=S, h0_std=h0_std, seed=16, g_lo=-0.2)
    res = gpu_forward(inp, scale=scale, path="two_pass")
    _check_outputs(res, inp, scale=scale)
    _check_segments(res, inp, [(j, h) for j in range(S) for h in range(2)])


def test_two_pass_packed_sampled_heads():
    inp = make_workload(workloads()["packed65536_h32_s64"])
    res = gpu_forward(inp, path="two_pass")
    _check_outputs(res, inp, heads=[0, 31])
    _check_segments(res, inp, [(j, h) for j in (0, 1, 17, 40, 63) for h in (0, 31)])


def test_two_pass_summaries_equal_the_fix_up_paths():
    """The summaries and incoming states come from the same arithmetic in both paths (bit-equal);
    outputs and final states differ only by rounding (the fix-up adds S_in^T qhat afterwards)."""
    inp = make_workload(workloads()["t4096_h8_s4"])
    dev = to_device(inp)
    a = gpu_forward(inp, path="fused", dev=dev)
    b = gpu_forward(inp, path="two_pass", dev=dev)
    for key in ("A", "B", "S_in"):
        assert np.array_equal(a[key], b[key]), key
    assert float(np.max(np.abs(a["o"] - b["o"]))) <= O_TOL
    assert rel_err(b["final"], a["final"]) <= REL_TOL


def test_custom_segment_bounds():
    inp = make_inputs([130, 70, 300], heads=2, segments=4, h0_std=0.1, seed=12)
    bounds = [0, 1, 129, 333, 500]
    res = gpu_forward(inp, seg_bounds=bounds)
    assert res["bounds"] == bounds
    _check_outputs(res, inp)
    _check_segments(res, inp, [(j, h) for j in range(4) for h in range(2)])


def test_closed_form_static_state_on_gpu():
    """beta = 0 and g = 0: the state stays h0, so o_t = h0^T q_t and final = h0."""
    inp = make_inputs([257, 100], heads=2, segments=3, h0_std=0.5, seed=13)
    inp.beta[:] = 0
    inp.g[:] = 0
    res = gpu_forward(inp)
    q = bf16_to_f32(inp.q).astype(np.float64)
    cu = inp.cu_seqlens
    for s in range(inp.num_seqs):
        for h in range(2):
            want = q[cu[s]:cu[s + 1], h] @ inp.h0[s, h].astype(np.float64)
            assert float(np.max(np.abs(res["o"][cu[s]:cu[s + 1], h] - want))) <= O_TOL
            assert rel_err(res["final"][s, h], inp.h0[s, h]) <= REL_TOL


def test_wide_head_count_every_segment():
    """More heads than one wave of 16-column composition slices holds (the 32-column
    slices), with resets, continuing pieces and a random initial state: every head
    and segment against the oracle."""
    inp = make_inputs([300, 500, 77, 900], heads=24, segments=9, h0_std=0.1, seed=14)
    res = gpu_forward(inp)
    _check_outputs(res, inp)
    _check_segments(res, inp, [(j, h) for j in range(9) for h in range(24)])


def test_device_status_is_clear_after_every_kernel():
    """No bounded device-side wait expired in the runs above and in a fresh one (kda_device_status
    synchronises, reads and clears the kernels' status words)."""
    from context_kda_gb300 import binding as kda
    inp = make_workload(workloads()["t4096_h8_s4"])
    gpu_forward(inp)
    assert kda.kda_device_status() == kda.KDA_OK
    assert kda.kda_device_status() == kda.KDA_OK


def test_expired_wait_is_reported_and_the_context_survives():
    """A kernel whose bounded wait runs out (nothing arrives on its barrier) records KDA_ERR_TIMEOUT;
    kda_device_status reports it once, and the library keeps working afterwards."""
    from context_kda_gb300 import binding as kda
    assert kda.kda_device_status() == kda.KDA_OK
    kda.kda_selftest_wait_expiry()
    assert kda.kda_device_status() == kda.KDA_ERR_TIMEOUT
    assert kda.kda_device_status() == kda.KDA_OK
    inp = make_workload(workloads()["t1024_h4_s2"])
    res = gpu_forward(inp)
    _check_outputs(res, inp)
    assert kda.kda_device_status() == kda.KDA_OK


# ---- the two-level (blocked, log-depth across groups) scan: the same S_in as the chain

def _check_blocked(inp, heads=None, seg_bounds=None):
    from harness import gpu_scan_both
    res = gpu_scan_both(inp, seg_bounds)
    assert np.all(np.isfinite(res["S_in_blocked"]))
    hs = list(range(inp.heads)) if heads is None else list(heads)
    _, _, S_ref = oracle_summaries(inp, res["bounds"], hs)
    e_blocked = rel_err(res["S_in_blocked"][:, hs], S_ref[:, hs])
    e_chain = rel_err(res["S_in_chain"][:, hs], S_ref[:, hs])
    assert e_blocked <= REL_TOL, f"blocked scan S_in rel = {e_blocked:.3e}"
    assert e_chain <= REL_TOL, f"chain S_in rel = {e_chain:.3e}"
    assert rel_err(res["S_in_blocked"], res["S_in_chain"]) <= REL_TOL
    return e_blocked


def test_blocked_scan_packed_every_head_and_segment():
    _check_blocked(make_workload(workloads()["packed65536_h32_s64"]))


def test_blocked_scan_long_context_64_segments():
    _check_blocked(make_workload(workloads()["t32768_h32_s64"]), heads=[0, 7, 31])


@pytest.mark.parametrize("seqlens,S,h0_std", [
    ([1], 1, 0.0),                              # one segment, one group
    ([700], 2, 0.2),                            # two segments: groups of two
    ([900, 40, 300], 5, 0.1),                   # groups of 3, the last one short
    ([5, 5, 5, 5, 80], 20, 0.1),                # seeds and updates inside and at group starts
    ([2000], 17, 0.0),                          # S just above a square: a one-segment last group
    ([600, 1, 900], 50, 0.3),                   # a sequence starting exactly at a segment start
])
def test_blocked_scan_edge_cases(seqlens, S, h0_std):
    inp = make_inputs(seqlens, heads=2, segments=S, h0_std=h0_std, seed=41, g_lo=-0.2)
    _check_blocked(inp)


def test_fused_path_with_the_blocked_scan_every_head_and_segment():
    """Few heads and many segments: kda_forward_segmented composes by the two-level scan there (its
    depth model picks it on this device); outputs, final states and every summary against the
    oracle."""
    inp = make_workload(workloads()["t32768_h2_s64"])
    res = gpu_forward(inp)
    _check_outputs(res, inp)
    _check_all_segments(res, inp)


# ---- the chunk-level split within a segment: refined plans give the same results

def _refined(inp, sms=152):
    from context_kda_gb300 import binding as kda
    plan = kda.kda_plan_segments_refined(inp.cu_seqlens, inp.segments, inp.heads, sms)
    S = int(plan[5])
    return [int(x) for x in plan[int(plan[14]):int(plan[14]) + S + 1]]


@pytest.mark.parametrize("seqlens,H,S,h0_std", [
    ([16384], 2, 1, 0.1),               # one long sequence, two heads: 38 sub-segments
    ([3000, 5000, 900], 1, 2, 0.2),     # packed, one head, resets inside the refined segments
])
def test_refined_plan_matches_the_oracle(seqlens, H, S, h0_std):
    inp = make_inputs(seqlens, heads=H, segments=S, h0_std=h0_std, seed=61, g_lo=-0.1)
    bounds = _refined(inp)
    assert len(bounds) - 1 > S
    res = gpu_forward(inp, seg_bounds=bounds)
    _check_outputs(res, inp)
    _check_all_segments(res, inp)


def test_refined_summaries_compose_to_the_callers():
    """Within each caller segment the sub-segment summaries compose, (A2,B2) o (A1,B1) =
    (A2 A1, A2 B1 + B2), to that segment's summary from the unrefined plan."""
    inp = make_inputs([6000], heads=2, segments=2, h0_std=0.1, seed=62, g_lo=-0.05)
    coarse = gpu_forward(inp)
    bounds = _refined(inp)
    fine = gpu_forward(inp, seg_bounds=bounds)
    assert float(np.max(np.abs(fine["o"] - coarse["o"]))) <= O_TOL
    assert rel_err(fine["final"], coarse["final"]) <= REL_TOL
    cb = coarse["bounds"]
    for j in range(len(cb) - 1):
        subs = [i for i in range(len(bounds) - 1) if cb[j] <= bounds[i] < cb[j + 1]]
        for h in range(2):
            A = np.eye(128)
            B = np.zeros((128, 128))
            for i in subs:
                A2, B2 = fine["A"][i, h].astype(np.float64), fine["B"][i, h].astype(np.float64)
                A, B = A2 @ A, A2 @ B + B2
            assert rel_err(A, coarse["A"][j, h]) <= REL_TOL
            assert rel_err(B, coarse["B"][j, h]) <= REL_TOL
