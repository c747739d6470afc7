// Host planner for packed-THD segment plans (integer work only).
//
// cuLA PR #136, "feat(kda): add cuDNN concatenated-summary Kimi CP",
// §Walkthrough: CPU-only plan construction and validation for balanced or
// custom contiguous shards, checked against sequence boundaries, rank spans and
// invalid inputs.  The word layout is documented in include/kda.h.
//
// One merge-style walk over the segment bounds and the sequence boundaries
// yields the pieces (segment x sequence intersections) in (segment, start)
// order; everything else is derived from the piece list.
#include <algorithm>
#include <climits>
#include <cstdint>
#include <cstring>
#include <vector>

#include "../../include/kda.h"

namespace {

struct Piece {
    int32_t start, len, seq, seg, flags, cont, row, fin;
};

// FNV-1a over the plan's 32-bit words, the checksum word taken as 0 (the rule stated in kda.h).
uint32_t checksum_words(const int32_t *plan, size_t total)
{
    uint32_t h = 2166136261u;
    for (size_t i = 0; i < total; ++i) {
        const uint32_t w = i == KDA_PH_CHECKSUM ? 0u : static_cast<uint32_t>(plan[i]);
        h = (h ^ w) * 16777619u;
    }
    return h;
}

}  // namespace

// Checksum of a plan of 'total' words, for the other translation units of the library.
namespace kda {
uint32_t plan_checksum_words(const int32_t *plan, size_t total) { return checksum_words(plan, total); }
}  // namespace kda

extern "C" int kda_plan_segments(const int32_t *cu, int32_t num_seqs, int32_t num_segments,
                                 const int32_t *seg_bounds, int32_t chunk, int32_t *plan,
                                 size_t *plan_len)
{
    if (!plan_len || !cu || num_seqs < 1 || num_segments < 1) return KDA_ERR_INVALID_ARG;
    if (cu[0] != 0) return KDA_ERR_INVALID_ARG;
    for (int32_t n = 0; n < num_seqs; ++n)
        if (cu[n + 1] <= cu[n]) return KDA_ERR_INVALID_ARG;
    if (chunk != KDA_CHUNK) return KDA_ERR_UNSUPPORTED;
    const int64_t T = cu[num_seqs];
    const int32_t N = num_seqs, S = num_segments;

    std::vector<int32_t> bounds(static_cast<size_t>(S) + 1);
    if (seg_bounds) {
        if (seg_bounds[0] != 0 || seg_bounds[S] != T) return KDA_ERR_INVALID_ARG;
        for (int32_t j = 0; j < S; ++j)
            if (seg_bounds[j + 1] <= seg_bounds[j]) return KDA_ERR_INVALID_ARG;
        std::memcpy(bounds.data(), seg_bounds, sizeof(int32_t) * bounds.size());
    } else {
        if (S > T) return KDA_ERR_INVALID_ARG;
        for (int32_t j = 0; j <= S; ++j) bounds[j] = static_cast<int32_t>((int64_t)j * T / S);
    }

    // Walk segments and sequences together.
    std::vector<Piece> pieces;
    std::vector<int32_t> segs(static_cast<size_t>(S) * 4);
    int32_t s = 0;  // sequence holding the current segment start
    for (int32_t j = 0; j < S; ++j) {
        const int32_t a = bounds[j], b = bounds[j + 1];
        while (cu[s + 1] <= a) ++s;
        int32_t flags = 0;
        if (cu[s] == a) flags |= KDA_SEG_STARTS_SEQ | KDA_SEG_HAS_RESET;
        const int32_t first = static_cast<int32_t>(pieces.size());
        int32_t pos = a, t = s;
        while (pos < b) {
            const int32_t end = std::min(b, cu[t + 1]);
            Piece p{pos, end - pos, t, j, 0, -1, -1, -1};
            p.flags = (pos == cu[t]) ? KDA_PIECE_FIRST : KDA_PIECE_CONT;
            if (pos == cu[t]) flags |= KDA_SEG_HAS_RESET;
            if (end == b) p.flags |= KDA_PIECE_SEG_LAST;
            if (end == cu[t + 1]) p.flags |= KDA_PIECE_SEQ_END;
            pieces.push_back(p);
            pos = end;
            if (pos == cu[t + 1]) ++t;
        }
        segs[4 * j + 0] = s;
        segs[4 * j + 1] = flags;
        segs[4 * j + 2] = first;
        segs[4 * j + 3] = static_cast<int32_t>(pieces.size()) - first;
    }

    const int32_t n_pieces = static_cast<int32_t>(pieces.size());
    std::vector<int32_t> cont, fin, chunks;
    int64_t row = 0;
    int32_t max_len = 0, n_chunks = 0;
    for (int32_t i = 0; i < n_pieces; ++i) {
        Piece &p = pieces[i];
        max_len = std::max(max_len, p.len);
        if (p.flags & KDA_PIECE_CONT) {
            p.cont = static_cast<int32_t>(cont.size() / 4);
            p.row = static_cast<int32_t>(row);
            cont.insert(cont.end(), {i, p.seg, p.row, p.len});
            row += p.len;
            if (p.flags & KDA_PIECE_SEQ_END) {
                p.fin = static_cast<int32_t>(fin.size() / 4);
                fin.insert(fin.end(), {i, p.seq, p.seg, p.cont});
            }
        }
        for (int32_t c = 0, st = 0; st < p.len; ++c, st += chunk) {
            chunks.insert(chunks.end(), {i, p.start + st, std::min(chunk, p.len - st), c});
            ++n_chunks;
        }
    }

    // Work items: longest pieces first so the longest serial chains start earliest.
    std::vector<std::pair<int32_t, int32_t>> items;
    items.reserve(static_cast<size_t>(n_pieces) * 2);
    for (int32_t i = 0; i < n_pieces; ++i) {
        items.emplace_back(i, 0);
        if (pieces[i].flags & KDA_PIECE_CONT) items.emplace_back(i, 1);
    }
    std::sort(items.begin(), items.end(), [&](const auto &x, const auto &y) {
        if (pieces[x.first].len != pieces[y.first].len) return pieces[x.first].len > pieces[y.first].len;
        if (x.first != y.first) return x.first < y.first;
        return x.second < y.second;
    });

    const int32_t n_cont = static_cast<int32_t>(cont.size() / 4);
    const int32_t n_fin = static_cast<int32_t>(fin.size() / 4);
    const int32_t n_items = static_cast<int32_t>(items.size());
    const size_t sizes[8] = {static_cast<size_t>(S) + 1, static_cast<size_t>(N) + 1, segs.size(),
                             static_cast<size_t>(n_pieces) * 8, static_cast<size_t>(n_items) * 2,
                             chunks.size(), cont.size(), fin.size()};
    size_t total = KDA_PLAN_HEADER_WORDS;
    size_t offs[8];
    for (int i = 0; i < 8; ++i) {
        offs[i] = total;
        total += sizes[i];
    }
    if (total > 0x7fffffffu) return KDA_ERR_UNSUPPORTED;
    const size_t cap = *plan_len;
    *plan_len = total;
    if (!plan) return KDA_OK;
    if (cap < total) return KDA_ERR_WORKSPACE;

    std::memset(plan, 0, sizeof(int32_t) * KDA_PLAN_HEADER_WORDS);
    plan[KDA_PH_MAGIC] = KDA_PLAN_MAGIC;
    plan[KDA_PH_VERSION] = KDA_PLAN_VERSION;
    plan[KDA_PH_TOTAL] = static_cast<int32_t>(total);
    plan[KDA_PH_T] = static_cast<int32_t>(T);
    plan[KDA_PH_N] = N;
    plan[KDA_PH_S] = S;
    plan[KDA_PH_C] = chunk;
    plan[KDA_PH_NPIECES] = n_pieces;
    plan[KDA_PH_NCONT] = n_cont;
    plan[KDA_PH_TCONT] = static_cast<int32_t>(row);
    plan[KDA_PH_NFIN] = n_fin;
    plan[KDA_PH_NCHUNKS] = n_chunks;
    plan[KDA_PH_NITEMS] = n_items;
    plan[KDA_PH_MAXPIECE] = max_len;
    for (int i = 0; i < 8; ++i) plan[KDA_PH_OFF_BOUNDS + i] = static_cast<int32_t>(offs[i]);

    std::memcpy(plan + offs[0], bounds.data(), sizeof(int32_t) * sizes[0]);
    std::memcpy(plan + offs[1], cu, sizeof(int32_t) * sizes[1]);
    std::memcpy(plan + offs[2], segs.data(), sizeof(int32_t) * sizes[2]);
    int32_t *pp = plan + offs[3];
    for (const Piece &p : pieces) {
        const int32_t w[8] = {p.start, p.len, p.seq, p.seg, p.flags, p.cont, p.row, p.fin};
        std::memcpy(pp, w, sizeof(w));
        pp += 8;
    }
    int32_t *ip = plan + offs[4];
    for (const auto &it : items) {
        *ip++ = it.first;
        *ip++ = it.second;
    }
    if (!chunks.empty()) std::memcpy(plan + offs[5], chunks.data(), sizeof(int32_t) * sizes[5]);
    if (!cont.empty()) std::memcpy(plan + offs[6], cont.data(), sizeof(int32_t) * sizes[6]);
    if (!fin.empty()) std::memcpy(plan + offs[7], fin.data(), sizeof(int32_t) * sizes[7]);
    plan[KDA_PH_CHECKSUM] = static_cast<int32_t>(checksum_words(plan, total));
    return KDA_OK;
}

// Whole-plan validation: the header must be self-consistent (sizes, section offsets in order and
// of the sizes the counts imply), and every word must be what the planner gives for the plan's own
// segment bounds and cu_seqlens.  Re-planning is the plainest complete check: the kernels index
// pieces, chunks, items and records from these words, so any other content is rejected.
extern "C" int kda_plan_check(const int32_t *plan)
{
    if (!plan) return KDA_ERR_INVALID_ARG;
    if (plan[KDA_PH_MAGIC] != KDA_PLAN_MAGIC || plan[KDA_PH_VERSION] != KDA_PLAN_VERSION ||
        plan[KDA_PH_C] != KDA_CHUNK)
        return KDA_ERR_INVALID_ARG;
    const int64_t total = plan[KDA_PH_TOTAL], T = plan[KDA_PH_T], N = plan[KDA_PH_N], S = plan[KDA_PH_S];
    if (total < KDA_PLAN_HEADER_WORDS || T < 1 || N < 1 || S < 1 || S > T || N > T) return KDA_ERR_INVALID_ARG;
    const int64_t counts[8] = {S + 1, N + 1, 4 * S, 8 * static_cast<int64_t>(plan[KDA_PH_NPIECES]),
                               2 * static_cast<int64_t>(plan[KDA_PH_NITEMS]),
                               4 * static_cast<int64_t>(plan[KDA_PH_NCHUNKS]),
                               4 * static_cast<int64_t>(plan[KDA_PH_NCONT]),
                               4 * static_cast<int64_t>(plan[KDA_PH_NFIN])};
    int64_t pos = KDA_PLAN_HEADER_WORDS;
    for (int i = 0; i < 8; ++i) {
        if (counts[i] < 0 || plan[KDA_PH_OFF_BOUNDS + i] != pos) return KDA_ERR_INVALID_ARG;
        pos += counts[i];
    }
    if (pos != total) return KDA_ERR_INVALID_ARG;
    if (static_cast<uint32_t>(plan[KDA_PH_CHECKSUM]) != checksum_words(plan, static_cast<size_t>(total)))
        return KDA_ERR_INVALID_ARG;
    // the bounds and sequence sections as the planner's inputs (it checks them itself)
    const int32_t *bounds = plan + plan[KDA_PH_OFF_BOUNDS];
    const int32_t *cu = plan + plan[KDA_PH_OFF_CU];
    if (cu[N] != T) return KDA_ERR_INVALID_ARG;
    size_t len = 0;
    if (kda_plan_segments(cu, static_cast<int32_t>(N), static_cast<int32_t>(S), bounds, KDA_CHUNK, nullptr, &len) !=
            KDA_OK ||
        len != static_cast<size_t>(total))
        return KDA_ERR_INVALID_ARG;
    std::vector<int32_t> again(len);
    if (kda_plan_segments(cu, static_cast<int32_t>(N), static_cast<int32_t>(S), bounds, KDA_CHUNK, again.data(),
                          &len) != KDA_OK)
        return KDA_ERR_INVALID_ARG;
    return std::memcmp(again.data(), plan, sizeof(int32_t) * len) == 0 ? KDA_OK : KDA_ERR_INVALID_ARG;
}

// Refined plan for latency-bound problems: every segment cut into m chunk-aligned sub-segments so
// that the serial chains are about m times shorter while the state pass still fits one wave of
// chains on the device: m = min(floor(num_sms / (2 heads S)), floor(chunks per segment / 4)), at
// least 1 (a piece that continues a sequence adds a transition chain to its state chain, hence the
// 2).  Cuts fall on multiples of 64 tokens from the segment start, the chunk grid of the segment's
// first piece.  The result is an ordinary plan of S m segments (custom bounds).
extern "C" int kda_plan_segments_refined(const int32_t *cu, int32_t num_seqs, int32_t num_segments,
                                         const int32_t *seg_bounds, int32_t chunk, int32_t heads, int32_t num_sms,
                                         int32_t *plan, size_t *plan_len)
{
    if (!plan_len || !cu || num_seqs < 1 || num_segments < 1 || heads < 1 || num_sms < 1)
        return KDA_ERR_INVALID_ARG;
    if (chunk != KDA_CHUNK) return KDA_ERR_UNSUPPORTED;
    // the caller's segmentation, validated by planning it once
    size_t len0 = 0;
    int rc = kda_plan_segments(cu, num_seqs, num_segments, seg_bounds, chunk, nullptr, &len0);
    if (rc != KDA_OK) return rc;
    const int64_t T = cu[num_seqs];
    const int32_t S = num_segments;
    std::vector<int64_t> b(static_cast<size_t>(S) + 1);
    for (int32_t j = 0; j <= S; ++j) b[j] = seg_bounds ? seg_bounds[j] : (int64_t)j * T / S;
    int64_t min_chunks = INT64_MAX;
    for (int32_t j = 0; j < S; ++j) min_chunks = std::min(min_chunks, (b[j + 1] - b[j]) / chunk);
    const int64_t by_sms = num_sms / (2LL * heads * S);
    const int64_t m = std::max<int64_t>(1, std::min(by_sms, min_chunks / 4));
    std::vector<int32_t> nb;
    nb.push_back(0);
    for (int32_t j = 0; j < S; ++j) {
        const int64_t a = b[j], e = b[j + 1], nch = (e - a + chunk - 1) / chunk;
        for (int64_t i = 1; i < m; ++i) {
            const int64_t cut = a + (nch * i / m) * chunk;
            if (cut > nb.back() && cut < e) nb.push_back(static_cast<int32_t>(cut));
        }
        nb.push_back(static_cast<int32_t>(e));
    }
    return kda_plan_segments(cu, num_seqs, static_cast<int32_t>(nb.size()) - 1, nb.data(), chunk, plan, plan_len);
}
