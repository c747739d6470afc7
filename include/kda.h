/*
 * kda.h -- C ABI of libkda: segment-parallel Kimi Delta Attention (KDA) forward
 * on one GB300 (sm_103a).
 *
 * KDA is a gated delta-rule linear attention with a K x V recurrent state per
 * (sequence, head):
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T,
 *     o_t = scale * S_t^T q_t,
 * with BF16 q/k/v and an FP32 state (cuLA PR #110, "feat(cp): add opt-in
 * NVSHMEM CP state handoff", §Supported configuration), g a per-token,
 * per-key-channel natural-log decay and beta a per-token scalar.
 *
 * Context parallelism on one GPU.  A packed token stream is cut into
 * contiguous segments that play the role of context-parallel ranks.  Each
 * segment runs the recurrence locally and publishes an FP32 affine boundary
 * summary of the state crossing its end, S_end = A S_start + B, with a
 * transition A (K x K) and a state update B (K x V) (PR #110 §Motivation:
 * affine recurrence state per producer; cuLA PR #136, "feat(kda): add cuDNN
 * concatenated-summary Kimi CP", §Summary: preceding_transition /
 * preceding_state_update).  Summaries compose in FP32 as
 * (A2,B2) o (A1,B1) = (A2 A1, A2 B1 + B2) (PR #136 §Summary) to give each
 * segment its true incoming state S_in, and the outputs of the piece that
 * continues a sequence from an earlier segment are fixed up with
 * o_t += S_in^T qhat_t, where qhat_t = scale P_t^T q_t and P_t is the
 * transition from the segment start through token t.
 *
 * Call sequence (PR #136 §Walkthrough, sequence diagram: plan, then run):
 *   kda_plan_segments          host, integer only, reusable across calls
 *   kda_segment_forward        local chunkwise recurrence + summaries + qhat
 *   kda_compose_summaries      scan of the summaries -> S_in per segment
 *   kda_apply_boundary         fix-up of continuing outputs and final states
 *   kda_forward_segmented      the three device steps above, in order
 *   kda_forward_two_pass       the same results from the preceding summaries:
 *                              summaries, composition, then the forward from
 *                              each segment's true incoming state (no fix-up)
 *
 * Conventions shared by every entry point
 *   - Fixed sizes: K = V = 128 (key and value head dimensions), chunk C = 64.
 *   - Tensors are contiguous, packed-THD, row-major:
 *       q, k  [T][H][K] bf16      v [T][H][V] bf16      o [T][H][V] bf16
 *       g     [T][H][K] fp32      beta [T][H] fp32
 *       h0, final_state [N][H][K][V] fp32 (state layout K x V, "non-transposed",
 *           PR #110 §Supported configuration); h0 == NULL means zeros
 *       A [S][H][K][K] fp32, B / S_in [S][H][K][V] fp32 (separate typed
 *           tensors, PR #136 §Latest cuDNN compatibility)
 *     bf16 is passed as its 16-bit pattern (kda_bf16).
 *   - The chunkwise form takes exp(+-Gamma), Gamma being the decay summed
 *     within a 64-token chunk.  g is a log-decay (g <= 0); each channel's
 *     per-chunk sum must stay above -77 (2^-112 in fp32: e^{+-Gamma} and the
 *     bf16 low parts of the split operands stay normal numbers), e.g.
 *     g >= -1.2 per token.  The preparation checks every (chunk, head, channel)
 *     and records KDA_ERR_RANGE for kda_device_status() when a sum falls
 *     below; the outputs of that call are then not valid.
 *   - Device pointers must be 16-byte aligned.  The library never allocates
 *     or frees memory, never synchronises, and enqueues all device work on
 *     the caller's CUDA stream ('stream' is a cudaStream_t; NULL = legacy
 *     default stream).
 *   - Arguments are validated on the host before anything is enqueued; a
 *     rejected call enqueues nothing.  There is no fallback path: an
 *     unsupported request returns KDA_ERR_UNSUPPORTED (PR #110 §Supported
 *     configuration: request an error instead of fallback; PR #136 §Latest
 *     cuDNN compatibility: fail early).
 *   - Launch failures return KDA_ERR_CUDA; kda_last_cuda_error() gives the
 *     underlying cudaError_t value.
 *   - Each call takes the host plan (to size its grids without reading device
 *     memory) and a device copy of the same words (plan_dev), which the caller
 *     uploads once.  Every call validates the whole host plan (kda_plan_check:
 *     each word must be what kda_plan_segments gives for its bounds; a plan
 *     seen before is recognised by its checksum) and rejects any other with
 *     KDA_ERR_INVALID_ARG.  Each kernel compares the device copy's length and
 *     checksum words with the host plan's before it reads anything else; on a
 *     mismatch it does nothing and records KDA_ERR_INVALID_ARG for
 *     kda_device_status().
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t kda_bf16;

enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = -1,   /* bad pointer, size, alignment or plan */
    KDA_ERR_UNSUPPORTED = -2,   /* valid request outside what is built (e.g. chunk != 64) */
    KDA_ERR_WORKSPACE = -3,     /* caller buffer too small */
    KDA_ERR_CUDA = -4,          /* a CUDA launch or API call failed */
    KDA_ERR_TIMEOUT = -5,       /* a bounded device-side wait expired */
    KDA_ERR_RANGE = -6          /* a chunk's summed decay is outside the range the chunkwise
                                   form computes in fp32 (see the conventions above) */
};

enum { KDA_HEAD_DIM_K = 128, KDA_HEAD_DIM_V = 128, KDA_CHUNK = 64 };

/* Plan format v2 (int32 words).  Header words: */
enum {
    KDA_PLAN_MAGIC = 0x4B444131,
    KDA_PLAN_VERSION = 2,
    KDA_PLAN_HEADER_WORDS = 32,
    KDA_PH_MAGIC = 0, KDA_PH_VERSION = 1, KDA_PH_TOTAL = 2, KDA_PH_T = 3, KDA_PH_N = 4,
    KDA_PH_S = 5, KDA_PH_C = 6, KDA_PH_NPIECES = 7, KDA_PH_NCONT = 8, KDA_PH_TCONT = 9,
    KDA_PH_NFIN = 10, KDA_PH_NCHUNKS = 11, KDA_PH_NITEMS = 12, KDA_PH_MAXPIECE = 13,
    KDA_PH_OFF_BOUNDS = 14, KDA_PH_OFF_CU = 15, KDA_PH_OFF_SEGS = 16, KDA_PH_OFF_PIECES = 17,
    KDA_PH_OFF_ITEMS = 18, KDA_PH_OFF_CHUNKS = 19, KDA_PH_OFF_CONT = 20, KDA_PH_OFF_FIN = 21,
    KDA_PH_CHECKSUM = 22
};
/* Word 22 is a checksum of the whole plan: FNV-1a over 32-bit words,
 *     h = 2166136261; for every word w (word 22 taken as 0): h = (h ^ w) * 16777619 (mod 2^32),
 * stored as its bit pattern.  Words 23..31 are zero. */
/* Sections (in this order after the header):
 *   seg_bounds [S+1]; cu_seqlens [N+1];
 *   segs   [S][4]: sequence holding the segment's first token, flags
 *                  (1 = segment starts a sequence, 2 = a sequence starts inside
 *                  the segment, so its transition A is exactly 0), first piece,
 *                  piece count;
 *   pieces [n][8]: start, len, sequence, segment, flags (1 FIRST: starts its
 *                  sequence; 2 CONT: continues a sequence from an earlier
 *                  segment; 4 SEG_LAST; 8 SEQ_END), cont index or -1, qhat row
 *                  or -1, fin index or -1; in (segment, start) order;
 *   items  [m][2]: piece, kind (0 state columns for every piece, 1 transition
 *                  columns for CONT pieces), sorted by (-len, piece, kind);
 *   chunks [c][4]: piece, start, len, index in piece (every C tokens from the
 *                  piece start);
 *   cont   [n_cont][4]: piece, segment, qhat row (running sum of CONT lengths),
 *                  len;
 *   fin    [n_fin][4]:  piece, sequence, segment, cont index, for CONT pieces
 *                  that end their sequence. */
enum { KDA_SEG_STARTS_SEQ = 1, KDA_SEG_HAS_RESET = 2 };
enum { KDA_PIECE_FIRST = 1, KDA_PIECE_CONT = 2, KDA_PIECE_SEG_LAST = 4, KDA_PIECE_SEQ_END = 8 };

/* Human-readable name of a status code (static string, never NULL). */
const char *kda_status_string(int status);

/* cudaError_t value behind the most recent KDA_ERR_CUDA on this thread (0 if none). */
int kda_last_cuda_error(void);

/* Device-side status of the kernels run so far on the current device.  A kernel
 * records, in its status word (the first error kept):
 *   KDA_ERR_TIMEOUT      a wait inside it (for a copy, a product or another
 *                        thread's handoff) gave up after about two seconds; it
 *                        let its copies land, freed its tensor memory and
 *                        returned, so the context stays usable;
 *   KDA_ERR_RANGE        a chunk's summed decay was out of range (conventions);
 *   KDA_ERR_INVALID_ARG  its device plan was not the host plan's copy, so it
 *                        returned without touching memory.
 * The results of such a call are invalid.  This call synchronises the current
 * device (the only entry point that does), reads every status word, clears them
 * and returns KDA_OK, the first error found, or KDA_ERR_CUDA if the
 * synchronisation or the read failed. */
int kda_device_status(void);

/* Self-test of that path: enqueues a one-warp kernel whose bounded wait expires
 * (nothing arrives on its barrier), about two seconds later; the next
 * kda_device_status() then returns KDA_ERR_TIMEOUT and clears it.  Returns
 * KDA_OK or KDA_ERR_CUDA (launch failure). */
int kda_selftest_wait_expiry(void *stream);

/* Self-test of a real kernel's abort path: kda_segment_forward's two kernels
 * with the package copies of every piece's second chunk withheld inside the
 * state pass, so that its waits for them (and for the products that need
 * them) run out after about two seconds; the kernel then lets its issued
 * copies and products land, frees its tensor memory and returns.  The next
 * kda_device_status() returns KDA_ERR_TIMEOUT; the results of this call are
 * invalid and the context stays usable.  Arguments as kda_segment_forward
 * (the plan must have a piece of more than one chunk).  Returns KDA_OK,
 * KDA_ERR_INVALID_ARG, KDA_ERR_WORKSPACE or KDA_ERR_CUDA. */
int kda_selftest_state_abort(const int32_t *plan, const int32_t *plan_dev, int32_t H,
                             const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                             const float *g, const float *beta, const float *h0, float scale,
                             kda_bf16 *o, float *A, float *B, float *final_state,
                             void *ws, size_t ws_bytes, void *stream);

/*
 * kda_plan_segments -- packed-THD segment plan (host, integer work only).
 * PR #136 §Walkthrough: CPU-only plan construction and validation for balanced
 * or custom contiguous shards, checked against sequence boundaries and
 * invalid inputs; the plan is reusable (PR #136 §Summary).
 *
 *   cu_seqlens   host int32 [num_seqs+1]: 0 = cu[0] < cu[1] < ... (zero-length
 *                sequences are rejected); T = cu[num_seqs].
 *   num_segments S >= 1.
 *   seg_bounds   host int32 [S+1] strictly increasing from 0 to T, or NULL for
 *                balanced segments b_j = floor(j T / S) (then S <= T).
 *   chunk        must be 64 (else KDA_ERR_UNSUPPORTED).
 *   plan         host int32 buffer of *plan_len words, caller-owned; NULL to
 *                query the size only.
 *   plan_len     in: capacity in words; out: words the plan needs.
 * Returns KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, or
 * KDA_ERR_WORKSPACE (capacity too small; *plan_len holds the size needed).
 * Deterministic: the same arguments give the same words.
 */
int kda_plan_segments(const int32_t *cu_seqlens, int32_t num_seqs, int32_t num_segments,
                      const int32_t *seg_bounds, int32_t chunk, int32_t *plan, size_t *plan_len);

/*
 * kda_plan_check -- validates a host plan word by word: the header's sizes and
 * section offsets, then every section, by planning its segment bounds and
 * cu_seqlens again and comparing all words (the checksum included).  The
 * buffer must hold plan[KDA_PH_TOTAL] words.  Returns KDA_OK or
 * KDA_ERR_INVALID_ARG.  Every entry point that takes a plan runs this check
 * (a plan already accepted is recognised by its checksum and not re-planned).
 */
int kda_plan_check(const int32_t *plan);

/*
 * kda_plan_segments_refined -- the chunk-level split within a segment: a plan
 * whose segments refine the caller's, each cut into m sub-segments of whole
 * 64-token chunks (cuts on multiples of 64 from the segment start), so that
 * the serial chunk chains are m times shorter.  The same affine summaries
 * carry the state across the new cuts (PR #110 §Motivation: affine recurrence
 * state; PR #136 §Summary: summary composition), so kda_forward_segmented on
 * this plan gives the outputs and final states of the caller's segmentation
 * (within rounding); its summaries are those of the sub-segments, which
 * compose within each caller segment to that segment's summary.
 *   m = max(1, min(floor(num_sms / (2 heads S)), floor(chunks per segment / 4))):
 *   about one wave of state and transition chains on the device, and at least
 *   four chunks per sub-segment.  It pays where few heads and long segments
 *   leave most SMs idle (a single long sequence with a few heads); with
 *   2 heads S >= num_sms it changes nothing.
 *   heads, num_sms  the H the plan will run with and the device's SM count.
 * Other arguments, results and errors as kda_plan_segments.
 */
int kda_plan_segments_refined(const int32_t *cu_seqlens, int32_t num_seqs, int32_t num_segments,
                              const int32_t *seg_bounds, int32_t chunk, int32_t heads, int32_t num_sms,
                              int32_t *plan, size_t *plan_len);

/* Bytes of one chunk package: the per-chunk operands that the chunk-parallel
 * preparation hands to the serial state pass (see kda_segment_forward). */
enum { KDA_PACKAGE_BYTES = 123392 };

/*
 * kda_workspace_layout -- byte offsets of the regions of the device workspace
 * for a plan and head count.  off[0..6] = qhat, fin transitions, packages, A,
 * B, S_in, total.  Each region starts on a 256-byte boundary.
 *   qhat   bf16, H*T_cont*K       transition-seen queries of continuing tokens
 *                                  (they only complete bf16 outputs); per head and
 *                                  continuing piece, its rows (from the piece's qhat
 *                                  row) in tiles of 128, the last one R rows: box b
 *                                  (k in [64b, 64b+64)) of a tile holds row r at
 *                                  byte (b*R + r)*128 from the tile's start, the
 *                                  row's 16-byte groups j at ((j ^ (r & 7)) * 16)
 *   fin    fp32 [n_fin][H][K][K]  transitions of continuing pieces that end a sequence
 *   pkg    [H][n_chunks][KDA_PACKAGE_BYTES]  per-chunk operands (scratch)
 *   A      fp32 [S][H][K][K]      (used by kda_forward_segmented)
 *   B      fp32 [S][H][K][V]      (used by kda_forward_segmented)
 *   S_in   fp32 [S][H][K][V]      (used by kda_forward_segmented)
 *   then, when S >= 16, kda_scan_workspace_bytes(plan, H) bytes of scratch for
 *   the two-level scan (256-byte aligned, included in off[6]).
 * The three-call path uses the first off[3] bytes (qhat, fin, packages); A, B
 * and S_in are then caller tensors.  kda_apply_boundary reads only qhat and fin
 * (the first off[2] bytes).  Returns KDA_OK or KDA_ERR_INVALID_ARG.
 */
int kda_workspace_layout(const int32_t *plan, int32_t H, size_t off[7]);

/* kda_workspace_bytes -- total device workspace bytes (off[6] above); 0 if the
 * plan or H is invalid.  The summary part, A + B, is S*H*(K*K + K*V)*4 bytes:
 * 256 MiB at S = 64, H = 32, K = V = 128 (PR #136 §Latest cuDNN compatibility). */
size_t kda_workspace_bytes(const int32_t *plan, int32_t H);

/*
 * kda_segment_forward -- local chunkwise forward of every piece of every
 * segment, plus the segment summaries (PR #110 §Motivation; PR #136 §Summary).
 *   q, k, v, g, beta   inputs as above (device).
 *   h0                 device fp32 [N][H][K][V] or NULL (zeros).
 *   scale              query scale (1.0 for the plain recurrence).
 *   o      out  bf16 [T][H][V]: exact outputs for pieces that start their
 *               sequence; for continuing pieces the output of the local run
 *               from a zero state (completed by kda_apply_boundary).
 *   A      out  fp32 [S][H][K][K]: the segment's transition; exactly 0 when a
 *               sequence starts inside the segment.
 *   B      out  fp32 [S][H][K][V]: the state at the segment end when the
 *               segment starts from a zero state (exact where the segment's
 *               last piece starts its sequence).
 *   final_state out fp32 [N][H][K][V]: exact for sequences whose last piece
 *               starts the sequence; local (zero-start) end state otherwise
 *               (completed by kda_apply_boundary).
 *   ws, ws_bytes  device workspace of at least off[3] bytes (kda_workspace_layout);
 *               its qhat and fin regions are written, its package region is
 *               scratch.
 * Two kernels run on 'stream': a chunk-parallel preparation of every (chunk,
 * head), which writes that chunk's operands (decayed queries and keys, the
 * WY factors of the intra-chunk transform, the masked query-key scores) as a
 * package, then the serial state pass of every piece, which reads them.
 * Returns KDA_ERR_WORKSPACE when ws_bytes is short.
 */
int kda_segment_forward(const int32_t *plan, const int32_t *plan_dev, int32_t H,
                        const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                        const float *g, const float *beta, const float *h0, float scale,
                        kda_bf16 *o, float *A, float *B, float *final_state,
                        void *ws, size_t ws_bytes, void *stream);

/*
 * kda_compose_summaries -- incoming state of every segment, S_in, by composing
 * the summaries in order (PR #136 §Summary: affine summary composition in
 * FP32).  S_in[0] = h0 of the first sequence; S_in[j] = h0 of the sequence
 * starting at b_j when one does; otherwise A[j-1] S_in[j-1] + B[j-1].
 *   A, B   device fp32 summaries from kda_segment_forward.
 *   h0     device fp32 [N][H][K][V] or NULL (zeros).
 *   S_in   out device fp32 [S][H][K][V].
 */
int kda_compose_summaries(const int32_t *plan, const int32_t *plan_dev, int32_t H,
                          const float *A, const float *B, const float *h0, float *S_in,
                          void *stream);

/*
 * kda_compose_summaries_blocked -- the same S_in as kda_compose_summaries by a
 * two-level scan that is log-depth across groups (PR #136 §Summary: affine
 * summary composition in FP32; the maps F_j of the chain, S_in[j] =
 * F_j(S_in[j-1]), composed as a prefix scan).  The segments are cut into
 * groups of m = ceil(sqrt(S)); three kernels run on 'stream':
 *   1. every group's total map C_g = F_last o ... o F_first, all groups and
 *      heads in parallel, carried as the K x (K + V) state [A~ | B~] from the
 *      identity;
 *   2. the chain over the group totals, E_{g+1} = C_g(E_g): each group's
 *      incoming state;
 *   3. every group in parallel from E_g through its own maps, writing S_in.
 * The depth is about 3 sqrt(S) products instead of S - 1, for about three
 * times the tensor work and twice the memory traffic of the chain.
 *   ws, ws_bytes  device scratch of at least kda_scan_workspace_bytes(plan, H)
 *                 bytes, 256-byte aligned (group totals and incoming states).
 * Other arguments and results as kda_compose_summaries; the outputs agree
 * with it within rounding.  Returns KDA_ERR_WORKSPACE when ws_bytes is short.
 */
int kda_compose_summaries_blocked(const int32_t *plan, const int32_t *plan_dev, int32_t H,
                                  const float *A, const float *B, const float *h0, float *S_in,
                                  void *ws, size_t ws_bytes, void *stream);

/* Device scratch bytes kda_compose_summaries_blocked needs: G*H*K*(K+V)*4
 * (group totals) + G*H*K*V*4 (incoming states), G = ceil(S / ceil(sqrt(S)));
 * 0 if the plan or H is invalid. */
size_t kda_scan_workspace_bytes(const int32_t *plan, int32_t H);

/*
 * kda_apply_boundary -- fix-up from the incoming states: for every token t of
 * a continuing piece in segment j, o_t = o_local,t + S_in[j]^T qhat_t,
 * rounded to bf16 (in 128-token tiles the correction is rounded to bf16 and
 * added by the memory system's bf16 add; in a shorter last tile the sum is
 * rounded once); for every sequence that ends in a continuing piece of
 * segment j, final = P_end S_in[j] + final_local (fp32).  Every output and
 * final-state element receives exactly one addition, so results are
 * deterministic.
 *   S_in        device fp32 [S][H][K][V] from kda_compose_summaries.
 *   ws          the workspace kda_segment_forward wrote (qhat and fin regions).
 *   o           in/out bf16 [T][H][V].   final_state in/out fp32 [N][H][K][V].
 */
int kda_apply_boundary(const int32_t *plan, const int32_t *plan_dev, int32_t H,
                       const float *S_in, const void *ws, size_t ws_bytes,
                       kda_bf16 *o, float *final_state, void *stream);

/*
 * kda_forward_segmented -- the whole segmented forward: kda_segment_forward,
 * the composition and kda_apply_boundary in order on 'stream', with A, B and
 * S_in held in the workspace (kda_workspace_bytes(plan, H) bytes).  The
 * composition takes the chain (kda_compose_summaries) or, from 16 segments
 * on, the two-level scan (kda_compose_summaries_blocked) when its depth,
 * counted in products per CTA over the waves this device's SMs need, is the
 * smaller: with few heads and many segments, where the chain's CTAs leave
 * most SMs idle.
 * Outputs o and final_state equal the monolithic recurrence of every sequence
 * (PR #136 §Walkthrough: compared with a monolithic reference).
 */
int kda_forward_segmented(const int32_t *plan, const int32_t *plan_dev, int32_t H,
                          const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                          const float *g, const float *beta, const float *h0, float scale,
                          kda_bf16 *o, float *final_state, void *ws, size_t ws_bytes,
                          void *stream);

/*
 * kda_forward_two_pass -- the segmented forward from preceding summaries: the
 * forward run takes each segment's incoming state as an input instead of being
 * fixed up afterwards (PR #136 §Summary: the cuDNN KDA forward takes the
 * preceding state update and transition).  Same arguments, results and
 * workspace as kda_forward_segmented; the workspace's qhat and fin regions
 * are not used.  Four kernels run on 'stream':
 *   1. the chunk-parallel preparation of every (chunk, head) package;
 *   2. the state pass of the last piece of each segment only, writing that
 *      segment's A and B and nothing else;
 *   3. the composition into S_in (as kda_compose_summaries);
 *   4. the state pass of every piece again, from its true incoming state
 *      (h0 of its sequence, or S_in of its segment for a piece that continues
 *      a sequence), reading the same packages and writing o and final_state.
 * The state pass runs twice and the fix-up and qhat traffic disappear.
 * Returns as kda_forward_segmented.
 */
int kda_forward_two_pass(const int32_t *plan, const int32_t *plan_dev, int32_t H,
                         const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                         const float *g, const float *beta, const float *h0, float scale,
                         kda_bf16 *o, float *final_state, void *ws, size_t ws_bytes,
                         void *stream);

/*
 * kda_backward_segmented -- gradients of the segmented forward, segment-
 * parallel through the following summaries (PR #136 §Summary and its
 * walkthrough's sequence diagram: the following FP32 summaries are gathered
 * during the backward; PR #110 §Correctness: output and Q/K/V/g/beta
 * gradients).  The loss is L = sum_t <do_t, o_t> + sum_seq <dfinal, S_end>,
 * o and S_end those of kda_forward_segmented on the same inputs.
 *   q, k, v, g, beta, h0, scale   the forward's inputs (device), as above.
 *   dout     device bf16 [T][H][V]: the gradient of the outputs.
 *   dfinal   device fp32 [N][H][K][V] or NULL (zeros): of the final states.
 *   dq, dk   out device fp32 [T][H][K];   dv out fp32 [T][H][V];
 *   dg       out device fp32 [T][H][K];   dbeta out fp32 [T][H];
 *   dh0      out device fp32 [N][H][K][V] (the gradient of the initial
 *            states, defined also when h0 is NULL) or NULL (not written).
 *   ws, ws_bytes  device workspace of at least kda_backward_workspace_bytes.
 * Steps on 'stream': the forward's preparation (which also leaves each
 * chunk's terms for the backward), local state pass and composition (S_in,
 * the segment transitions A and the final-state transitions of continuing
 * pieces); every piece from its true incoming
 * state, recording each chunk's start state; the incoming-state gradient of
 * every continuing piece through its own outputs; the following summaries,
 * last segment first, giving each segment's end-state gradient; every piece
 * backwards from it, recording each chunk's end-state gradient and giving
 * dh0; and every (chunk, head) in parallel for dq, dk, dv, dg and dbeta.
 * Matrices are kept in FP32; every product runs on the tensor cores as a
 * three-term bf16 split (about 2^-16 relative, FP32 accumulation).  Returns
 * KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_WORKSPACE or KDA_ERR_CUDA; a bounded
 * wait that gave up is reported by kda_device_status() as KDA_ERR_TIMEOUT.
 */
int kda_backward_segmented(const int32_t *plan, const int32_t *plan_dev, int32_t H,
                           const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                           const float *g, const float *beta, const float *h0, float scale,
                           const kda_bf16 *dout, const float *dfinal,
                           float *dq, float *dk, float *dv, float *dg, float *dbeta, float *dh0,
                           void *ws, size_t ws_bytes, void *stream);

/* Device workspace bytes kda_backward_segmented needs (0 if the plan or H is
 * invalid): the forward's (kda_workspace_bytes), then scratch for the
 * forward's outputs, the chunk start states and end-state gradients
 * (2 * H * n_chunks * K * V * 4 bytes), the segment gradients
 * (2 * S * H * K * V * 4 bytes), the kernels' working areas, each chunk's
 * FP32 terms for the gradient pass (49,152 bytes per chunk and head), and
 * each chunk's bf16 operand images for the reverse chains and the gradient
 * pass (214,016 bytes per chunk and head). */
size_t kda_backward_workspace_bytes(const int32_t *plan, int32_t H);

/*
 * kda_forward_segmented_noalloc -- kda_forward_segmented without a caller
 * workspace.  The pages have no counterpart to this entry point.
 *
 * For callers that cannot allocate device memory: code that is handed only its
 * input and output buffers by a host framework that owns every device
 * allocation (a plugin inside an inference engine, for instance), and code that
 * must not call cudaMalloc in its steady-state loop because an allocation there
 * can synchronise the device and stall other work.  The workspace lives in a
 * fixed device array inside the library, KDA_NOALLOC_SCRATCH_BYTES (32 MiB)
 * long, which every GPU that loads the library holds until the process exits.
 *   - Arguments and results are those of kda_forward_segmented; the caller
 *     still passes every input and output buffer.
 *   - Returns KDA_ERR_WORKSPACE when kda_workspace_bytes(plan, H) exceeds
 *     KDA_NOALLOC_SCRATCH_BYTES (the workspace is dominated by the 123 KB chunk
 *     packages of every chunk and head: T = 1024, H = 4, S = 2 needs about
 *     10 MiB and fits; T = 4096, H = 8, S = 4 needs about 73 MiB and does not).
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it; make that first call before any
 *     stream capture.  The cached address belongs to the context it was looked
 *     up in: after cudaDeviceReset, or once the primary context is destroyed
 *     and created again, the next call finds a new context id and looks the
 *     address up again (so that call, too, should come before any capture).
 *   - Nothing is allocated, freed or cleared: every workspace region is fully
 *     written before it is read within a call.
 *   - All calls on a device share the one array, which keeps the last call's
 *     contents: calls that overlap on the GPU (other streams, other host
 *     threads) race on it and must be serialised by the caller.
 */
enum { KDA_NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024 };

int kda_forward_segmented_noalloc(const int32_t *plan, const int32_t *plan_dev, int32_t H,
                                  const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                                  const float *g, const float *beta, const float *h0, float scale,
                                  kda_bf16 *o, float *final_state, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
