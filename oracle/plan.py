"""Independent Python planner for packed-THD segment plans -- test infrastructure.

Re-implements, from the written format rules only, the plan that the C-ABI
``kda_plan_segments`` produces, so the two can be compared word for word.
The rules follow cuLA PR #136 ("feat(kda): add cuDNN concatenated-summary
Kimi CP", §Walkthrough, packed-shard planning): balanced or custom contiguous
shards over a packed token stream, validated against sequence boundaries.

Plan format v2 (int32 words)
  header (32 words):
     0 magic 0x4B444131        1 version 2            2 total words
     3 T tokens                4 N sequences          5 S segments
     6 C chunk                 7 n_pieces             8 n_cont
     9 T_cont                 10 n_fin               11 n_chunks
    12 n_items                13 max piece length
    14..21 word offsets of: seg_bounds, cu_seqlens, segs, pieces, items,
           chunks, cont, fin
    22 checksum: FNV-1a over the 32-bit words of the whole plan (this word
       taken as 0): h = 2166136261, then h = (h ^ w) * 16777619 mod 2^32 per
       word, stored as a signed 32-bit value;   23..31 zero
  seg_bounds [S+1]; cu_seqlens [N+1]
  segs    [S][4]  (sequence containing the segment's first token, flags,
                   first piece, piece count); flags: 1 = segment starts a
                   sequence, 2 = some sequence starts inside the segment
  pieces  [n][8]  (start, len, sequence, segment, flags, cont index or -1,
                   qhat row or -1, fin index or -1) in (segment, start) order;
                   flags: 1 FIRST (starts its sequence), 2 CONT (continues a
                   sequence begun in an earlier segment), 4 SEG_LAST,
                   8 SEQ_END
  items   [m][2]  (piece, kind) kind 0 = state columns (every piece),
                   kind 1 = transition columns (CONT pieces); sorted by
                   (-piece length, piece, kind)
  chunks  [c][4]  (piece, start, len, index in piece), pieces cut every C
                   tokens from the piece start
  cont    [n_cont][4] (piece, segment, qhat row, len); qhat rows are the running
                   sum of CONT piece lengths in piece order
  fin     [n_fin][4]  (piece, sequence, segment, cont index) for CONT pieces
                   that end their sequence
"""
from __future__ import annotations

MAGIC = 0x4B444131
VERSION = 2
CHECKSUM_WORD = 22
HEADER_WORDS = 32

FIRST, CONT, SEG_LAST, SEQ_END = 1, 2, 4, 8
SEG_STARTS_SEQ, SEG_HAS_RESET = 1, 2


class PlanError(ValueError):
    def __init__(self, code: str, msg: str):
        super().__init__(f"{code}: {msg}")
        self.code = code


def plan_segments(cu_seqlens, num_segments, seg_bounds=None, chunk=64):
    cu = [int(x) for x in cu_seqlens]
    if chunk != 64:
        raise PlanError("unsupported", "chunk must be 64")
    if len(cu) < 2:
        raise PlanError("invalid", "need at least one sequence")
    if cu[0] != 0:
        raise PlanError("invalid", "cu_seqlens[0] must be 0")
    for a, b in zip(cu, cu[1:]):
        if b <= a:
            raise PlanError("invalid", "sequence lengths must be positive")
    T = cu[-1]
    N = len(cu) - 1
    S = int(num_segments)
    if S < 1:
        raise PlanError("invalid", "need at least one segment")
    if seg_bounds is None:
        if S > T:
            raise PlanError("invalid", "more segments than tokens")
        bounds = [(j * T) // S for j in range(S + 1)]
    else:
        bounds = [int(x) for x in seg_bounds]
        if len(bounds) != S + 1 or bounds[0] != 0 or bounds[-1] != T:
            raise PlanError("invalid", "custom bounds must run from 0 to T")
        for a, b in zip(bounds, bounds[1:]):
            if b <= a:
                raise PlanError("invalid", "custom bounds must be strictly increasing")

    def seq_of(t):
        # the sequence whose token range holds t (linear search; plain by design)
        for s in range(N):
            if cu[s] <= t < cu[s + 1]:
                return s
        raise AssertionError

    starts = set(cu[:-1])
    segs, pieces = [], []
    for j in range(S):
        a, b = bounds[j], bounds[j + 1]
        flags = 0
        if a in starts:
            flags |= SEG_STARTS_SEQ
        if any(a <= c < b for c in cu[:-1]):
            flags |= SEG_HAS_RESET
        first_piece = len(pieces)
        for s in range(N):
            lo, hi = max(a, cu[s]), min(b, cu[s + 1])
            if lo >= hi:
                continue
            pf = FIRST if lo == cu[s] else CONT
            if hi == b:
                pf |= SEG_LAST
            if hi == cu[s + 1]:
                pf |= SEQ_END
            pieces.append([lo, hi - lo, s, j, pf, -1, -1, -1])
        segs.append([seq_of(a), flags, first_piece, len(pieces) - first_piece])

    cont, fin = [], []
    row = 0
    for i, p in enumerate(pieces):
        if p[4] & CONT:
            p[5] = len(cont)
            p[6] = row
            cont.append([i, p[3], row, p[1]])
            row += p[1]
            if p[4] & SEQ_END:
                p[7] = len(fin)
                fin.append([i, p[2], p[3], p[5]])

    items = [(i, 0) for i in range(len(pieces))] + [(i, 1) for i, p in enumerate(pieces) if p[4] & CONT]
    items.sort(key=lambda it: (-pieces[it[0]][1], it[0], it[1]))

    chunks = []
    for i, p in enumerate(pieces):
        n = (p[1] + chunk - 1) // chunk
        for c in range(n):
            chunks.append([i, p[0] + c * chunk, min(chunk, p[1] - c * chunk), c])

    sections = [bounds, cu, [w for s_ in segs for w in s_], [w for p in pieces for w in p],
                [w for it in items for w in it], [w for c in chunks for w in c],
                [w for c in cont for w in c], [w for f in fin for w in f]]
    offsets = []
    pos = HEADER_WORDS
    for sec in sections:
        offsets.append(pos)
        pos += len(sec)
    header = [MAGIC, VERSION, pos, T, N, S, chunk, len(pieces), len(cont), row, len(fin), len(chunks),
              len(items), max(p[1] for p in pieces)] + offsets
    header += [0] * (HEADER_WORDS - len(header))
    words = header
    for sec in sections:
        words = words + list(sec)
    assert len(words) == pos
    words[CHECKSUM_WORD] = checksum(words)
    return words


def checksum(words):
    """FNV-1a over 32-bit words with the checksum word taken as 0, as a signed 32-bit value."""
    h = 2166136261
    for i, w in enumerate(words):
        x = 0 if i == CHECKSUM_WORD else (int(w) & 0xFFFFFFFF)
        h = ((h ^ x) * 16777619) & 0xFFFFFFFF
    return h - (1 << 32) if h >= (1 << 31) else h


def decode(words):
    """Split a v2 plan into named Python lists (for tests)."""
    h = list(words[:HEADER_WORDS])
    T, N, S = h[3], h[4], h[5]
    n_p, n_c, n_f, n_ch, n_it = h[7], h[8], h[10], h[11], h[12]

    def sec(i, n, w):
        off = h[14 + i]
        flat = list(words[off:off + n * w])
        return [flat[r * w:(r + 1) * w] for r in range(n)] if w > 1 else flat

    return {
        "T": T, "N": N, "S": S, "C": h[6], "T_cont": h[9], "max_piece_len": h[13],
        "seg_bounds": sec(0, S + 1, 1), "cu_seqlens": sec(1, N + 1, 1), "segs": sec(2, S, 4),
        "pieces": sec(3, n_p, 8), "items": sec(4, n_it, 2), "chunks": sec(5, n_ch, 4),
        "cont": sec(6, n_c, 4), "fin": sec(7, n_f, 4),
    }
