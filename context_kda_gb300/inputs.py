"""Seeded synthetic inputs for segmented KDA forward workloads.

This module only draws random numbers and lays them out; it performs none of
the KDA arithmetic.  Both the CUDA path and the CPU oracle consume exactly the
arrays produced here, so the two sides see identical bf16 bit patterns and
fp32 values.

Workload shapes follow the correctness/performance tables of cuLA PR #110
("feat(cp): add opt-in NVSHMEM CP state handoff", §Correctness and
§Performance: 1024x4 at CP 2 and 4, 4096x8 and 8192x16 at CP 4) and the
summary-workspace example of cuLA PR #136 ("feat(kda): add cuDNN
concatenated-summary Kimi CP", §Latest cuDNN compatibility: CP64, H=32,
K=V=128).  The pages publish no dataset; everything is drawn here.

Recipe (seed 0).  Every tensor has its own generator family, PCG64 seeded by
``SeedSequence(seed, spawn_key=(tensor id, block))``; large tensors are drawn in
blocks of 2^16 (token, head) rows, one generator per block, so the blocks can be
drawn in parallel and the values do not depend on the thread count:
  lengths (id 0; packed variable-length workload only): l_i = exp(U(ln 256, ln 8192)),
      rescaled to the requested total (floor, deficit given +1 each to the
      largest fractional parts, ties to the lower index);
  q, k (ids 1, 2): N(0,1) fp32, L2-normalised per (token, head) over K (squared
         norm accumulated in fp64, no epsilon; row times the fp32 reciprocal
         norm), rounded to bf16 (round-to-nearest-even);
  v (id 3): N(0,1) fp32 rounded to bf16;
  g (id 4): fp32 log-decay per key channel, lo + (hi - lo) U(0,1);
  beta (id 5): sigmoid(N(0,1)) in fp64, stored as fp32, one per (token, head);
  h0 (id 6): optional fp32 N(0, std^2) initial state per sequence, [N,H,K,V].

bf16 tensors are returned as ``uint16`` bit patterns; ``bf16_to_f32`` gives
their exact fp32 values.
"""
from __future__ import annotations

import concurrent.futures as cf
import math
import os
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np

K_DIM = 128
V_DIM = 128
CHUNK = 64
_ROWS_PER_BLOCK = 1 << 16   # (token, head) rows drawn per independent block


@dataclass(frozen=True)
class Workload:
    """Shape and distribution of one synthetic segmented-KDA workload."""

    name: str
    seqlens: tuple            # lengths of the packed sequences (sum = T)
    heads: int
    segments: int
    g_lo: float = -0.05
    g_hi: float = -0.001
    h0_std: float = 0.0       # 0 => zero initial state (h0 = None)
    seed: int = 0
    lognormal_lengths: Optional[tuple] = None   # (count, lo, hi, total) when drawn
    note: str = ""

    @property
    def tokens(self) -> int:
        return int(sum(self.seqlens))


def _block_rng(seed: int, tensor_id: int, block: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=(tensor_id, block))))


def draw_lengths(rng: np.random.Generator, count: int, lo: float, hi: float, total: int) -> List[int]:
    """Log-uniform lengths rescaled to sum exactly to ``total``."""
    raw = np.exp(rng.uniform(math.log(lo), math.log(hi), size=count))
    scaled = raw * (float(total) / float(raw.sum()))
    base = np.floor(scaled).astype(np.int64)
    deficit = int(total - int(base.sum()))
    frac = scaled - base
    # largest fractional parts first; ties resolved toward the lower index
    order = sorted(range(count), key=lambda i: (-frac[i], i))
    for i in order[:deficit]:
        base[i] += 1
    return [int(x) for x in base]


def _packed_lengths() -> tuple:
    return tuple(draw_lengths(_block_rng(0, 0, 0), 24, 256.0, 8192.0, 65536))


def workloads() -> Dict[str, Workload]:
    """The named workloads.  ``t8192_h16_s4`` is the throughput headline."""
    packed = _packed_lengths()
    w = [
        Workload("t1024_h4_s2", (1024,), 4, 2, note="1 sequence, 2 segments, zero h0"),
        Workload("t4096_h8_s4", (4096,), 8, 4, h0_std=0.1, note="1 sequence, 4 segments, h0 ~ N(0, 0.1^2)"),
        Workload("t8192_h16_s4", (8192,), 16, 4, g_lo=-0.2, g_hi=-0.001,
                 note="1 sequence, 4 segments, strong decay g ~ U(-0.2,-0.001)"),
        Workload("packed65536_h32_s64", packed, 32, 64, lognormal_lengths=(24, 256, 8192, 65536),
                 note="24 packed sequences, 64 balanced segments crossing sequence boundaries"),
        Workload("t32768_h32_s8", (32768,), 32, 8, note="long context"),
        Workload("t32768_h32_s64", (32768,), 32, 64, note="long context"),
        Workload("t131072_h32_s8", (131072,), 32, 8, note="long context"),
        Workload("t131072_h32_s64", (131072,), 32, 64, note="long context"),
        Workload("t32768_h2_s64", (32768,), 2, 64,
                 note="few heads, many segments: the composition chain leaves most SMs idle"),
        Workload("t131072_h2_s1", (131072,), 2, 1,
                 note="few heads, one long segment: two serial chains of 2048 chunks (the chunk-level split)"),
    ]
    return {x.name: x for x in w}


HEADLINE = "t8192_h16_s4"


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (round-to-nearest-even); returns uint16 bit patterns.

    Inputs here are finite, so no NaN handling is needed."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact fp32 values of bf16 bit patterns."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _l2_normalised_bf16(x: np.ndarray) -> np.ndarray:
    """Per-row L2 normalisation over the last axis (squared norm accumulated in fp64, the row
    scaled by the fp32 reciprocal of the norm), then bf16."""
    nrm = np.sqrt(np.einsum("ij,ij->i", x, x, dtype=np.float64))
    return f32_to_bf16_bits(x * (1.0 / nrm).astype(np.float32)[:, None])


def _draw_rows(seed: int, tensor_id: int, rows: int, width: int, kind: str) -> np.ndarray:
    """rows x width array filled block by block; block b of 2^16 rows comes from its own
    generator (seed, spawn key (tensor_id, b))."""
    out = np.empty((rows, width), dtype=np.float32 if kind == "u01" else np.uint16)
    nblk = (rows + _ROWS_PER_BLOCK - 1) // _ROWS_PER_BLOCK

    def one(b):
        lo, hi = b * _ROWS_PER_BLOCK, min(rows, (b + 1) * _ROWS_PER_BLOCK)
        rng = _block_rng(seed, tensor_id, b)
        if kind == "bf16n":      # N(0,1), L2-normalised per row, bf16
            out[lo:hi] = _l2_normalised_bf16(rng.standard_normal((hi - lo, width), dtype=np.float32))
        elif kind == "bf16":     # N(0,1), bf16
            out[lo:hi] = f32_to_bf16_bits(rng.standard_normal((hi - lo, width), dtype=np.float32))
        else:                    # U(0,1) fp32
            out[lo:hi] = rng.random((hi - lo, width), dtype=np.float32)

    workers = min(16, max(1, os.cpu_count() or 1), max(1, nblk))
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        list(ex.map(one, range(nblk)))
    return out


@dataclass
class Inputs:
    """One drawn problem.  bf16 tensors are uint16 bit patterns."""

    cu_seqlens: np.ndarray    # int32 [N+1]
    q: np.ndarray             # uint16 [T,H,K]
    k: np.ndarray             # uint16 [T,H,K]
    v: np.ndarray             # uint16 [T,H,V]
    g: np.ndarray             # float32 [T,H,K]
    beta: np.ndarray          # float32 [T,H]
    h0: Optional[np.ndarray]  # float32 [N,H,K,V] or None
    segments: int
    heads: int
    extra: dict = field(default_factory=dict)

    @property
    def tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def num_seqs(self) -> int:
        return int(self.cu_seqlens.shape[0] - 1)


def make_inputs(seqlens, heads: int, segments: int, g_lo: float = -0.05, g_hi: float = -0.001,
                h0_std: float = 0.0, seed: int = 0, K: int = K_DIM, V: int = V_DIM,
                draw_lengths_spec: Optional[tuple] = None) -> Inputs:
    """Draw lengths (when asked), q, k, v, g, beta and h0 from ``seed`` (recipe above)."""
    if draw_lengths_spec is not None:
        count, lo, hi, total = draw_lengths_spec
        seqlens = draw_lengths(_block_rng(seed, 0, 0), count, lo, hi, total)
    seqlens = [int(x) for x in seqlens]
    T = int(sum(seqlens))
    H = int(heads)
    cu = np.zeros(len(seqlens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(seqlens)
    q = _draw_rows(seed, 1, T * H, K, "bf16n").reshape(T, H, K)
    k = _draw_rows(seed, 2, T * H, K, "bf16n").reshape(T, H, K)
    v = _draw_rows(seed, 3, T * H, V, "bf16").reshape(T, H, V)
    u = _draw_rows(seed, 4, T * H, K, "u01").reshape(T, H, K)
    g = (np.float32(g_lo) + np.float32(g_hi - g_lo) * u).astype(np.float32)
    del u
    logits = _block_rng(seed, 5, 0).standard_normal((T, H), dtype=np.float32).astype(np.float64)
    beta = (1.0 / (1.0 + np.exp(-logits))).astype(np.float32)
    h0 = None
    if h0_std > 0.0:
        h0 = (_block_rng(seed, 6, 0).standard_normal((len(seqlens), H, K, V), dtype=np.float32)
              * np.float32(h0_std)).astype(np.float32)
    return Inputs(cu, q, k, v, g, beta, h0, int(segments), H)


def make_workload(w: Workload, seed: Optional[int] = None) -> Inputs:
    return make_inputs(w.seqlens if w.lognormal_lengths is None else None, w.heads, w.segments,
                       w.g_lo, w.g_hi, w.h0_std, w.seed if seed is None else seed,
                       draw_lengths_spec=w.lognormal_lengths)


def draw_output_grads(inp: Inputs, seed: int = 0, with_dfinal: bool = True):
    """Seeded gradients of a problem's outputs for the backward: do ~ N(0,1) rounded to bf16
    [T,H,V] (tensor id 7) and, when asked, dfinal ~ N(0,1) fp32 [N,H,K,V] (tensor id 8)."""
    T, H, N = inp.tokens, inp.heads, inp.num_seqs
    V, K = inp.v.shape[2], inp.q.shape[2]
    do = _draw_rows(seed, 7, T * H, V, "bf16").reshape(T, H, V)
    dfinal = None
    if with_dfinal:
        dfinal = _block_rng(seed, 8, 0).standard_normal((N, H, K, V), dtype=np.float32)
    return do, dfinal
