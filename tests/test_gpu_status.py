"""GPU tests of the device-side status words beyond the bounded waits:

* a device plan that is not the copy of the host plan the launch was sized from
  (another problem's plan uploaded in its place): every kernel compares the
  plan's length and checksum words before reading anything else, does nothing,
  and kda_device_status() reports KDA_ERR_INVALID_ARG once;
* a decay whose per-chunk sum leaves the range the chunkwise form computes in
  fp32 (g ~ U(-3, -0.5), about -112 per 64-token chunk): the preparation
  records KDA_ERR_RANGE;
* a decay just inside that range (g ~ U(-1.15, -1.0), about -69 per chunk)
  matches the oracle and records nothing;
* the state pass's own bounded waits running out (its package copies
  withheld by the abort self-test): KDA_ERR_TIMEOUT, and the context stays
  usable.

Both error cases compute only finite or NaN/inf values without any
value-dependent control flow in the kernels, and leave the context usable: a
checked forward follows each of them.
"""
import numpy as np
import pytest

from context_kda_gb300.inputs import make_inputs
from harness import K, O_TOL, REL_TOL, V, gpu_forward, oracle_forward, rel_err, to_device

pytestmark = pytest.mark.gpu


def _checked_forward(inp):
    res = gpu_forward(inp)
    o_ref, f_ref = oracle_forward(inp)
    assert float(np.max(np.abs(res["o"] - o_ref))) <= O_TOL
    assert rel_err(res["final"], f_ref) <= REL_TOL
    return res


def test_device_plan_of_another_problem_is_refused_on_the_device():
    import torch
    from context_kda_gb300 import binding as kda
    assert kda.kda_device_status() == kda.KDA_OK
    inp = make_inputs([300, 200], heads=2, segments=3, h0_std=0.1, seed=31)
    other = kda.kda_plan_segments([0, 100, 500], 3)          # same T, another split
    plan = kda.kda_plan_segments(inp.cu_seqlens, inp.segments)
    assert not np.array_equal(plan, other)
    dev = to_device(inp)
    ws = torch.empty(kda.kda_workspace_bytes(plan, inp.heads), dtype=torch.uint8, device="cuda")
    o = torch.full((inp.tokens, inp.heads, V), 7.0, dtype=torch.bfloat16, device="cuda")
    fin = torch.full((inp.num_seqs, inp.heads, K, V), 7.0, dtype=torch.float32, device="cuda")
    kda.kda_forward_segmented(plan, kda.upload_plan(other), inp.heads, dev["q"], dev["k"], dev["v"], dev["g"],
                              dev["beta"], dev["h0"], 1.0, o, fin, ws)
    assert kda.kda_device_status() == kda.KDA_ERR_INVALID_ARG
    assert kda.kda_device_status() == kda.KDA_OK
    assert bool(torch.all(o == 7.0)) and bool(torch.all(fin == 7.0))   # nothing was written
    _checked_forward(inp)
    assert kda.kda_device_status() == kda.KDA_OK


def test_decay_beyond_the_chunkwise_range_is_reported():
    from context_kda_gb300 import binding as kda
    assert kda.kda_device_status() == kda.KDA_OK
    inp = make_inputs([256, 190], heads=2, segments=2, seed=32, g_lo=-3.0, g_hi=-0.5)
    gpu_forward(inp)
    assert kda.kda_device_status() == kda.KDA_ERR_RANGE
    assert kda.kda_device_status() == kda.KDA_OK
    _checked_forward(make_inputs([256, 190], heads=2, segments=2, seed=33))
    assert kda.kda_device_status() == kda.KDA_OK


def test_decay_just_inside_the_range_matches_the_oracle():
    from context_kda_gb300 import binding as kda
    assert kda.kda_device_status() == kda.KDA_OK
    inp = make_inputs([300, 70, 200], heads=2, segments=4, h0_std=0.1, seed=34, g_lo=-1.15, g_hi=-1.0)
    _checked_forward(inp)
    assert kda.kda_device_status() == kda.KDA_OK


def test_state_pass_abort_path_reports_and_the_context_survives():
    """A real kernel's waits run out: the state pass with the package copies of every piece's second
    chunk withheld waits about two seconds for them, then lets its issued copies and products land,
    frees its tensor memory and returns; kda_device_status reports KDA_ERR_TIMEOUT once, and a checked
    forward follows."""
    import torch
    from context_kda_gb300 import binding as kda
    assert kda.kda_device_status() == kda.KDA_OK
    inp = make_inputs([300, 200], heads=2, segments=3, h0_std=0.1, seed=35)
    plan = kda.kda_plan_segments(inp.cu_seqlens, inp.segments)
    plan_dev = kda.upload_plan(plan)
    dev = to_device(inp)
    T, H, N, S = inp.tokens, inp.heads, inp.num_seqs, inp.segments
    off = kda.kda_workspace_layout(plan, H)
    ws = torch.empty(off[3], dtype=torch.uint8, device="cuda")
    o = torch.empty((T, H, V), dtype=torch.bfloat16, device="cuda")
    A = torch.empty((S, H, K, K), dtype=torch.float32, device="cuda")
    B = torch.empty((S, H, K, V), dtype=torch.float32, device="cuda")
    fin = torch.empty((N, H, K, V), dtype=torch.float32, device="cuda")
    kda.kda_selftest_state_abort(plan, plan_dev, H, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["h0"],
                                 1.0, o, A, B, fin, ws)
    assert kda.kda_device_status() == kda.KDA_ERR_TIMEOUT
    assert kda.kda_device_status() == kda.KDA_OK
    _checked_forward(inp)
    assert kda.kda_device_status() == kda.KDA_OK
