"""GPU test of kda_forward_segmented_noalloc, the entry point for callers that
cannot allocate device memory (a plugin handed only its input and output
buffers by a framework that owns every allocation, or a loop that must not
call cudaMalloc because an allocation can synchronise the device).  It uses the
library's fixed 32 MiB device workspace instead of a caller buffer.

The test calls it through the C ABI twice in a row, on two different problems
and then on the first again.  The forward is deterministic, so every result
must equal, bit for bit, that of kda_forward_segmented with a caller-allocated
workspace; both problems are also checked against the fp64 oracle with the
tolerances of the other GPU tests.  This file is collected last on purpose, and
it passes both on its own in a fresh process and after the rest of the suite.
"""
import numpy as np
import pytest

from context_kda_gb300.inputs import make_inputs, make_workload, workloads
from harness import O_TOL, REL_TOL, K, V, oracle_forward, rel_err, to_device

pytestmark = pytest.mark.gpu


def _run(inp, noalloc):
    import torch
    from context_kda_gb300 import binding as kda
    dev = to_device(inp)
    plan = kda.kda_plan_segments(inp.cu_seqlens, inp.segments)
    plan_dev = kda.upload_plan(plan)
    o = torch.full((inp.tokens, inp.heads, V), float("nan"), dtype=torch.bfloat16, device="cuda")
    fin = torch.full((inp.num_seqs, inp.heads, K, V), float("nan"), dtype=torch.float32, device="cuda")
    args = (plan, plan_dev, inp.heads, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["h0"], 1.0, o, fin)
    if noalloc:
        kda.kda_forward_segmented_noalloc(*args)
    else:
        ws = torch.empty(kda.kda_workspace_bytes(plan, inp.heads), dtype=torch.uint8, device="cuda")
        kda.kda_forward_segmented(*args, ws)
    torch.cuda.synchronize()
    return o.view(torch.int16).cpu().numpy(), o.float().cpu().numpy(), fin.cpu().numpy()


def _compare(inp):
    bits_ref, _, f_ref = _run(inp, noalloc=False)
    bits_na, o_na, f_na = _run(inp, noalloc=True)
    assert np.all(np.isfinite(o_na)) and np.all(np.isfinite(f_na))
    assert np.array_equal(bits_na, bits_ref)
    assert np.array_equal(f_na.view(np.int32), f_ref.view(np.int32))
    o_or, f_or = oracle_forward(inp)
    assert float(np.max(np.abs(o_na - o_or))) <= O_TOL
    assert rel_err(f_na, f_or) <= REL_TOL


def test_noalloc_matches_caller_workspace_on_consecutive_calls():
    first = make_workload(workloads()["t1024_h4_s2"])
    second = make_inputs([300, 500, 224], heads=4, segments=5, h0_std=0.1, seed=21, g_lo=-0.2)
    _compare(first)
    _compare(second)
    _compare(first)      # the array still holds the second call's contents


def test_noalloc_rejects_problems_beyond_its_scratch():
    from context_kda_gb300 import binding as kda
    inp = make_workload(workloads()["t8192_h16_s4"])   # needs 278 MiB of workspace
    plan = kda.kda_plan_segments(inp.cu_seqlens, inp.segments)
    assert kda.kda_workspace_bytes(plan, inp.heads) > kda.NOALLOC_SCRATCH_BYTES
    import torch
    plan_dev = kda.upload_plan(plan)
    dev = to_device(inp)
    o = torch.empty((inp.tokens, inp.heads, V), dtype=torch.bfloat16, device="cuda")
    fin = torch.empty((inp.num_seqs, inp.heads, K, V), dtype=torch.float32, device="cuda")
    with pytest.raises(kda.KDAError) as e:
        kda.kda_forward_segmented_noalloc(plan, plan_dev, inp.heads, dev["q"], dev["k"], dev["v"], dev["g"],
                                          dev["beta"], dev["h0"], 1.0, o, fin)
    assert e.value.status == kda.KDA_ERR_WORKSPACE
