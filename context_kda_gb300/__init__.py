"""Segment-parallel Kimi Delta Attention (KDA) forward on GB300 (sm_103a).

The compute lives in ``libkda.so`` (hand-written CUDA for sm_103a behind the C
ABI of ``include/kda.h``); ``binding`` is its thin ctypes binding, whose
functions carry the C entry points' names and are re-exported here on first
use.  Accessing any of them raises ImportError when libkda.so has not been
built: there is no fallback.  ``inputs`` draws the seeded synthetic
workloads and can be used without the library.
"""
from __future__ import annotations

import importlib

_BINDING_NAMES = ("kda_status_string", "kda_plan_segments", "kda_plan_check", "kda_plan_segments_refined", "kda_workspace_layout",
                  "kda_workspace_bytes", "kda_segment_forward", "kda_compose_summaries", "kda_apply_boundary",
                  "kda_forward_segmented", "kda_forward_two_pass", "kda_forward_segmented_noalloc",
                  "kda_device_status", "kda_selftest_wait_expiry", "kda_compose_summaries_blocked",
                  "kda_scan_workspace_bytes", "kda_backward_segmented", "kda_backward_workspace_bytes", "upload_plan", "KDAError", "LIB_PATH")


def __getattr__(name):
    if name in _BINDING_NAMES:
        return getattr(importlib.import_module(".binding", __name__), name)
    raise AttributeError(name)
