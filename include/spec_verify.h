/*
 * spec_verify.h -- C ABI of the batched verification step of speculative
 * decoding and of the paged-KV commit / rollback that follows it.
 *
 * Sources (page titles; sections as printed on the pages):
 *   [SD] "Speculative decoding: accelerate LLM generation without changing its
 *        answers" -- section 2 "Draft, verify, correct", section 3 "Why this
 *        preserves the target distribution", section 4 "Data flow and
 *        performance trade-offs", section 5 "Reproducible toy lab",
 *        section 6 "Production failures, debugging, and security".
 *   [KV] "Walk through KV-cache updates when speculative decoding rejects some
 *        draft tokens" (provisional append, left-to-right acceptance, free the
 *        pages / rewind the write pointer, the cache invariant).
 *   [RJ] "Rejected speculative tokens remain in KV", paragraphs 1-3
 *        (allocation is not acceptance; partially valid blocks).
 *   [CV] "Keep cache validity aligned with the committed token history",
 *        paragraphs 1-5 (pending-token convention; block tables, ownership and
 *        reference counts; shared-prefix isolation; tree implementations keep
 *        the accepted path; the cases to test: EOS, output caps, tree branch
 *        switches).
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is a DEVICE pointer owned by the caller, unless
 *     the comment says "host".  The library keeps no pointer after a call.
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and is asynchronous.  No call synchronises, except
 *     sv_get_error().  No call allocates device memory, except sv_create().
 *   - Arguments the host can check (null pointers, sizes, alignment, dtype
 *     combinations) are checked before anything is launched: a failing check
 *     returns SV_ERR_INVALID / SV_ERR_UNSUPPORTED and launches nothing.
 *   - Conditions only the device can see (a bad token id, NaN logits, an
 *     exhausted block pool, inconsistent block tables) are reported through
 *     per-request status bits and the handle's device error word, which
 *     sv_get_error() reads and clears.  Nothing traps or asserts on the device.
 *   - Only one call per handle may be in flight on the GPU at a time when it
 *     uses the handle's workspace (calls that overlap race on it).
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* sv_stream_t; /* == cudaStream_t */
typedef struct sv_handle sv_handle;      /* opaque: device error word + launch cache */

typedef enum {
  SV_OK = 0,
  SV_ERR_INVALID = -1,     /* bad argument (host-checked) */
  SV_ERR_OOM = -2,         /* block pool exhausted in bfl_reserve (device) */
  SV_ERR_CUDA = -3,        /* a CUDA runtime call failed */
  SV_ERR_TIMEOUT = -4,     /* a bounded device-side wait gave up (device) */
  SV_ERR_UNSUPPORTED = -5, /* valid but not provided (dtype mix, V too large) */
  SV_ERR_STATE = -6,       /* block tables / refcounts inconsistent (device) */
  SV_ERR_TOO_LARGE = -7    /* batch beyond spec_verify_static's fixed scratch */
} sv_status;

typedef enum { SV_BF16 = 0, SV_FP32 = 1 } sv_dtype;
typedef enum { SV_DRAFT_LOGITS = 0, SV_DRAFT_PROBS = 1 } sv_draft_kind;

/* per-request status bits (sv_verify_args.status) */
#define SV_ST_Q_ZERO 1u         /* a tested draft had q(y) = 0 ([SD] s5, variation 2) */
#define SV_ST_BAD_INPUT 2u      /* NaN/+inf/empty row, bad T, top_p, k or token id */
#define SV_ST_RESIDUAL_EMPTY 4u /* rejected but max(0, p - q) == 0 numerically: drew from p */
#define SV_ST_TIMEOUT 8u        /* the request's outcome was not resolved in time */
#define SV_ST_EOS 16u           /* an accepted draft was the request's EOS id: it ended there */
#define SV_ST_CAPPED 32u        /* the output cap stopped the walk after accepted drafts */

/* sv_verify_args.flags */
#define SV_FLAG_NO_SKIP 1u /* also process rows after a known rejection (debug) */
/* Testing aid for the bounded waits: row 0 of request 0 never publishes its
 * decision, and the waits that depend on it give up after 1024 polls (about
 * 0.25 ms) instead of about 2^20.  Request 0 then never resolves: the call
 * reports SV_ST_TIMEOUT for it (accepted = -1, no tokens) and SV_ERR_TIMEOUT
 * in the error word, every other request is unaffected, and the context stays
 * usable.  Meant for inputs where row 0 of request 0 is accepted (a rejection
 * there resolves nothing either way, but then the request's outcome would not
 * depend on the withheld row). */
#define SV_FLAG_TEST_WITHHOLD 2u
/* Kernel selection (both kernels compute the same results).  By default a
 * call runs on the cluster-resident kernel.  SV_FLAG_STREAM_PATH asks for the
 * streaming kernel (persistent producer/consumer/finisher CTAs, window and
 * race items queued across SMs), which serves calls without top-k or the
 * repetition penalty whose top-p, if any, is on bf16 logit rows; other calls
 * stay on the cluster kernel.  SV_FLAG_CLUSTER_PATH forces the cluster kernel
 * and wins over SV_FLAG_STREAM_PATH. */
#define SV_FLAG_CLUSTER_PATH 4u
#define SV_FLAG_STREAM_PATH 8u

/* sv_row_debug.state */
#define SV_ROW_NONE 0
#define SV_ROW_ACCEPTED 1
#define SV_ROW_REJECTED 2
#define SV_ROW_SKIPPED 3 /* not processed: an earlier row was already rejected */
#define SV_ROW_INVALID 4
#define SV_ROW_BONUS 5
#define SV_ROW_TERMINAL 6 /* accepted, and the request ends here (EOS id or output cap) */

/* Optional per-row record, [B][kmax+1], written for every processed row. */
typedef struct {
  float p_y, q_y, u;    /* accept-test operands (draft rows only, else 0)   */
  float p_kept, q_kept; /* kept fraction of the pre-filter mass after top-p  */
  int32_t state;        /* SV_ROW_*                                          */
  int32_t p_thr_key;    /* order key of the smallest kept target value, or -1 */
  int32_t q_thr_key;    /* same for the draft row                             */
} sv_row_debug;

/*
 * Arguments of spec_verify ([SD] s2-s4; [KV]).
 *
 * Row i of request b (i = 0 .. k_b) is the target's prediction for the token
 * at absolute position S_b + 1 + i, where S_b = seq_len[b] is the number of
 * processed tokens before the pass and the pending token sits at S_b ([CV] 1).
 * Draft row i (i < k_b) is the draft distribution that proposed
 * draft_tokens[b][i].
 *
 * target  [B][kmax+1][target_ld] logits, bf16 or fp32.  Elements >= V of a row
 *         are never used but the caller must allocate the whole row: rows are
 *         read in 16-byte vectors.  target_ld >= V, target_ld * elem % 16 == 0,
 *         base 16-byte aligned.
 * draft   [B][kmax][draft_ld]: logits (bf16/fp32) or probabilities (fp32,
 *         non-negative, need not sum to 1).  Same layout rules.  May be NULL
 *         when kmax == 0.
 * draft_tokens [B][kmax] int32 proposals (entries >= k_b ignored).
 * k            [B] int32 drafts per request, 0 <= k_b <= kmax (ragged); NULL = kmax.
 * temperature  [B] fp32 >= 0; 0 = greedy limit (uniform over tied maxima).
 * top_p        [B] fp32 in (0, 1]; NULL = 1.  Applied to p and q alike.
 * request_id   [B] uint32 Philox stream id; NULL = b.
 * seq_len      [B] int32 S_b (read only here); NULL = 0.
 * seed         Philox4x32-10 key (lo, hi words).
 * eos_id       [B] int32 end-of-sequence token per request (< 0: none); NULL =
 *              none.  An ACCEPTED draft equal to it ends the request: it is
 *              emitted and no correction or bonus follows (SV_ST_EOS).
 * max_new      [B] int32 most tokens to emit in this call (>= 1); NULL = no
 *              cap.  Once max_new_b accepted drafts are emitted the walk stops
 *              (SV_ST_CAPPED); a correction or bonus is drawn only while the
 *              cap allows it.  A cap below 1 is bad input.  ([CV] paragraph 5
 *              lists EOS and output caps among the cases to test.)
 * rep_penalty  [B] fp32 repetition penalty theta_b per request, finite > 0
 *              (1 = none; anything else makes the request bad input); NULL =
 *              none.  [SD] s4 ("When it wins") counts repetition penalties
 *              among the transforms p and q are taken after and s6 requires
 *              target and draft to apply the same ones; the rule is CTRL's
 *              (Keskar et al. 2019): the logit l of a penalised token becomes
 *              l / theta if l > 0, else l * theta, in fp32 (round to nearest),
 *              rounded back to bf16 (ties to even) in a bf16 row.  Row i's
 *              penalised set is rep_tokens[b] together with draft_tokens[b][0
 *              .. i-1]; each token counts once however often it occurs.  Target
 *              rows and draft LOGIT rows are penalised alike; probability
 *              drafts are taken as given.
 * rep_tokens   [B][rep_ld] int32 the request's generated history (or any
 *              token set to penalise); entries outside [0, V) (e.g. -1
 *              padding) are ignored.  May be NULL when rep_ld == 0.
 * rep_ld       row stride of rep_tokens, 0 .. 2^24 (else SV_ERR_INVALID); read
 *              only when rep_penalty is set.  The inputs are read, never
 *              written; the penalty costs each CTA one pass over rep_ld + i ids
 *              per row.
 * top_k        [B] int32; NULL = none.  0 < top_k_b < V keeps, in p and in q,
 *              every token whose transformed probability is at least the
 *              top_k_b-th largest one (repeats counted, so ties at that value
 *              are all kept), renormalised; top-p then applies to the
 *              renormalised top-k distribution.  Any other value: no top-k.
 *              No effect at T = 0.  ([SD] s4 names top-k among the transforms
 *              p and q are taken after; the set-based reading is this
 *              library's.)
 * Outputs: accepted [B] (a_b in [0, k_b], or -1 when the request's input is
 *   bad), out_tokens [B][kmax+1] (the a_b accepted drafts, then the correction
 *   or bonus token unless EOS or the cap ended the walk, then -1), num_emitted
 *   [B] (a_b + 1, or a_b after EOS / cap, or 0), status [B].
 * debug  optional [B][kmax+1] sv_row_debug.  probs_p / probs_q optional
 *   [B][kmax+1][V] / [B][kmax][V] fp32 normalised transformed rows (debug
 *   only: the kernel then writes 4 bytes per element of every processed row).
 */
typedef struct {
  int32_t B, kmax, V;
  uint32_t flags;
  const void* target;
  int64_t target_ld;
  int32_t target_dtype; /* sv_dtype */
  int32_t draft_dtype;  /* sv_dtype */
  int32_t draft_kind;   /* sv_draft_kind */
  int32_t reserved0;
  const void* draft;
  int64_t draft_ld;
  const int32_t* draft_tokens;
  const int32_t* k;
  const float* temperature;
  const float* top_p;
  const uint32_t* request_id;
  const int32_t* seq_len;
  uint64_t seed;
  int32_t* accepted;
  int32_t* out_tokens;
  int32_t* num_emitted;
  uint32_t* status;
  sv_row_debug* debug;
  float* probs_p;
  float* probs_q;
  const int32_t* eos_id;
  const int32_t* max_new;
  const float* rep_penalty;
  const int32_t* rep_tokens;
  int64_t rep_ld;
  const int32_t* top_k;
} sv_verify_args;

/* Paged block pool: a LIFO free stack plus per-block reference counts
 * ([CV] 3: block tables, ownership and reference counts decide validity). */
typedef struct {
  int32_t num_blocks;  /* blocks in the pool                       */
  int32_t block_size;  /* token slots per block (BS)               */
  int32_t* free_stack; /* [num_blocks]; entries [0, *free_top) free */
  int32_t* free_top;   /* [1]                                       */
  int32_t* refcount;   /* [num_blocks]; 0 = free                    */
} bfl_state;

/* K/V payload of a paged cache (used only by the copy entry points):
 * data [num_blocks][layers][2][heads][block_size][head_dim] (2 = K, V), every
 * block's payload contiguous; 16-byte aligned, head_dim * elem_bytes a
 * multiple of 16.  elem_bytes 2 (bf16 / fp16) or 4; values are moved, never
 * interpreted. */
typedef struct {
  void* data;
  int32_t layers, heads, head_dim, elem_bytes;
} kv_payload;

/* sizeof(sv_verify_args) as compiled, for bindings to check their layout. */
size_t sv_verify_args_size(void);

/* Create a handle on `device` (allocates a few device words: the error word).
 * The device becomes current for the call.  Returns SV_ERR_CUDA on failure. */
sv_status sv_create(int device, sv_handle** handle);
sv_status sv_destroy(sv_handle* handle);

/* Bytes of workspace spec_verify needs for these arguments (host only; reads
 * B and kmax).  The workspace is caller-owned device memory, 256-byte aligned,
 * zero-filled before its FIRST use; afterwards spec_verify leaves it ready for
 * the next call.  Re-zero it after an SV_ERR_TIMEOUT or a CUDA error. */
sv_status sv_workspace_size(const sv_verify_args* args, size_t* bytes);

/* The verification step ([SD] s2 and s3; [KV]): for every request, the
 * temperature / top-p transformed target p_i and draft q_i; accept draft i iff
 * u_i * q_i(y_i) < p_i(y_i) (== u_i < min(1, p_i/q_i)), left to right; stop at
 * the first rejection; there draw the correction by the exponential race
 * argmax_x max(0, p_i - q_i)_x / E_x, or, when all k_b drafts are accepted,
 * the bonus token argmax_x p_{k_b,x} / E_x.  u and E come from Philox4x32-10:
 * key = (seed lo, seed hi), counter = (x >> 2, S_b + 1 + i, request_id_b,
 * stream), word x & 3, stream 0 for E_x and 1 for u_i (x = 0);
 * U = (2 * (r >> 9) + 1) * 2^-24, E = -ln U.
 * Rows after a rejection that is already known are skipped (their output does
 * not depend on them) unless SV_FLAG_NO_SKIP is set.
 * Errors: SV_ERR_INVALID / SV_ERR_UNSUPPORTED (host checks, nothing launched),
 * SV_ERR_CUDA (launch failed); device-side conditions go to status[] and the
 * error word. */
sv_status spec_verify(sv_handle* handle, const sv_verify_args* args, void* workspace,
                      size_t workspace_bytes, sv_stream_t stream);

/* Most rows (B * (kmax + 1)) one spec_verify_static call accepts. */
#define SV_STATIC_MAX_ROWS 16384

/* spec_verify for callers that cannot allocate device memory.  The pages
 * have no counterpart: this is a deployment variant of the same step.
 * Callers inside a memory pool or allocator hook (which must not re-enter the
 * allocator), runtimes that hand out all device memory up front and have no
 * scratch to give, and service loops that forbid allocation after start-up
 * cannot obtain the workspace spec_verify needs.  This entry point computes
 * exactly what spec_verify computes, with the same arguments, but takes no
 * handle and no workspace: its scratch (the ticket counters and one decision
 * word per row, about 64 KB) is a fixed array in device global memory, one
 * per device, kept for the life of the process.  It calls no cudaMalloc,
 * cudaFree or allocating library routine.
 *  - Limit: B * (kmax + 1) <= SV_STATIC_MAX_ROWS, else SV_ERR_TOO_LARGE and
 *    nothing is launched.  Other argument errors as spec_verify.
 *  - Set-up: the first call on a device (the current one) looks up the
 *    array's address with cudaGetSymbolAddress and reads the SM count; make
 *    that first call before any stream capture on that device.
 *  - Sharing: every call on a device uses the same array.  Each call clears
 *    the counters and its own rows' decision words with one cudaMemsetAsync
 *    on `stream` (at most 64 KB), then launches the kernel.  Calls whose GPU work overlaps (two streams without ordering
 *    between them) race on the array and give wrong results; issue them on
 *    one stream or order them with events.
 *  - Errors: no handle, so no device error word; device-side conditions are
 *    reported in status[] only. */
sv_status spec_verify_static(const sv_verify_args* args, sv_stream_t stream);

/*
 * Token-tree verification ([CV] paragraph 3: a tree implementation keeps the
 * accepted path; paragraph 5: test tree branch switches; the law of each test
 * is [SD] s2-s3).  Request b proposes a tree of n_b <= N nodes below its
 * pending token (node 0, the root).  Node i (1..n_b) is the proposal
 * tokens[b][i-1] following parent[b][i-1], a node with a LOWER index (so a
 * node's ancestors come before it).  Children of one node are independent
 * draws from the draft's distribution at that node (repeats allowed).
 *
 * Walk (reading; the pages give no law for trees): from the root, the
 * children c_1 .. c_m of the current node j (ascending index) are tested in
 * turn: accept c_r iff u_r * q_j(y) < p_r(y), with p_1 = p_j and p_{r+1} =
 * normalize(max(0, p_r - q_j)) after a rejection.  The first accepted child
 * becomes the current node.  If every child is rejected, the correction is
 * drawn from p_{m+1} (from p_j with SV_ST_RESIDUAL_EMPTY if that residual is
 * numerically empty); at a node without children the bonus is drawn from p_j.
 * Each test is one step of the linear law, so the emitted tokens follow the
 * target's distribution however the tree branches.  Transforms (T, top-k,
 * top-p) are those of spec_verify, applied to p_j and q_j.
 * Randomness: node depth d puts its token at position S_b + d; the tests
 * among j's children use the accept uniform of position S_b + d_j + 1 with
 * slot r - 1 (counter (slot >> 2, pos, request_id, 1), word slot & 3); the
 * correction or bonus after node j races with position S_b + d_j + 1.  A
 * chain-shaped tree gives exactly spec_verify's result.
 *
 * target [B][N+1][target_ld]: row j = the target's distribution of the token
 *        after node j (row 0: after the pending token).  draft [B][N+1]
 *        [draft_ld]: row j = the draft's distribution at node j (rows of
 *        leaves are never read).  Layout rules as in sv_verify_args.
 * parent, tokens [B][N] int32; n_nodes [B] (NULL = N); temperature [B];
 * top_p [B] (NULL = 1); top_k [B] (NULL = none); request_id [B] (NULL = b);
 * seq_len [B] S_b (NULL = 0); seed.
 * eos_id [B] (NULL = none) and max_new [B] (NULL = no cap; below 1: bad input):
 * an accepted child whose token is the request's EOS id ends the walk
 * (SV_ST_EOS), and so does the max_new_b-th accepted child (SV_ST_CAPPED);
 * then no correction or bonus follows ([CV] paragraph 5).
 * rep_penalty [B], rep_tokens [B][rep_ld], rep_ld: the repetition penalty of
 * sv_verify_args; node j's rows (target, and draft logits) are penalised for
 * the history ids plus the tokens of the accepted path up to and including j.
 * Outputs: accepted [B] = length a_b of the accepted path (-1 on bad input:
 *   a bad T / top_p / n_b / max_new / rep_penalty, a parent not below its node, a token outside
 *   [0, V), or a NaN / +inf / empty row on the walk); path [B][N] = the
 *   accepted node ids in depth order, then -1; out_tokens [B][N+1] = their
 *   tokens, then the correction or bonus token (none after EOS or the cap),
 *   then -1; num_emitted [B] = a_b + 1 (a_b after EOS or the cap; 0 on bad
 *   input); status [B] (SV_ST_* bits).
 * Each cluster of CTAs walks one request at a time, taking requests from a
 * counter the handle owns: only one spec_verify_tree call per handle may be in
 * flight on the GPU at a time (calls in one stream are ordered).  No
 * workspace is needed.
 */
#define SV_TREE_MAX_NODES 4096
typedef struct {
  int32_t B, N, V;
  uint32_t flags; /* reserved, 0 */
  const void* target;
  int64_t target_ld;
  int32_t target_dtype; /* sv_dtype */
  int32_t draft_dtype;  /* sv_dtype */
  int32_t draft_kind;   /* sv_draft_kind */
  int32_t reserved0;
  const void* draft;
  int64_t draft_ld;
  const int32_t* parent;
  const int32_t* tokens;
  const int32_t* n_nodes;
  const float* temperature;
  const float* top_p;
  const int32_t* top_k;
  const uint32_t* request_id;
  const int32_t* seq_len;
  uint64_t seed;
  int32_t* accepted;
  int32_t* path;
  int32_t* out_tokens;
  int32_t* num_emitted;
  uint32_t* status;
  const int32_t* eos_id;  /* [B] or NULL: as in sv_verify_args, for the path's tokens */
  const int32_t* max_new; /* [B] or NULL: at most max_new_b accepted nodes, then stop */
  const float* rep_penalty;  /* [B] or NULL: as in sv_verify_args */
  const int32_t* rep_tokens; /* [B][rep_ld] history ids (-1 padded) */
  int64_t rep_ld;
} sv_tree_args;

size_t sv_tree_args_size(void);
sv_status spec_verify_tree(sv_handle* handle, const sv_tree_args* args, sv_stream_t stream);

/* stack = [n-1, ..., 1, 0] (blocks pop as 0, 1, 2, ...), free_top = n,
 * refcount = 0. */
sv_status bfl_init(sv_handle* handle, const bfl_state* st, sv_stream_t stream);

/* Lookahead allocation before the verify pass ([RJ] 1: allocation is not
 * acceptance): make request b's table cover positions [0, S_b + k_b + 1).
 * Request b holds ceil(S_b/BS) blocks; it receives ceil((S_b+k_b+1)/BS) -
 * ceil(S_b/BS) more, popped in request order.  All-or-nothing: on a shortage
 * the device error word gets SV_ERR_OOM and nothing changes.  Appending into
 * a partially filled block whose refcount is above 1 is refused
 * (SV_ERR_STATE); bfl_reserve_cow copies such a block first.
 * seq_len [B], k [B] (NULL = 0), block_table [B][max_blocks] in/out. */
sv_status bfl_reserve(sv_handle* handle, const bfl_state* st, int32_t B, const int32_t* seq_len,
                      const int32_t* k, int32_t* block_table, int32_t max_blocks,
                      sv_stream_t stream);

/* Share whole blocks ([CV] 4): for pair p, dst[p] gets the first n_blocks[p]
 * blocks of src[p] (its entries must be -1) and each shared block's refcount
 * grows by one.  The caller sets dst's seq_len.  src, dst, n_blocks [n_pairs];
 * block_table [n_rows][max_blocks].  Ids outside [0, n_rows), src == dst, or a
 * dst entry that is not -1: SV_ERR_STATE, nothing changes.  A dst must not be
 * the src of another pair in the same call. */
sv_status bfl_fork_prefix(sv_handle* handle, const bfl_state* st, int32_t n_pairs,
                          const int32_t* src, const int32_t* dst, const int32_t* n_blocks,
                          int32_t* block_table, int32_t n_rows, int32_t max_blocks,
                          sv_stream_t stream);

/* Drop every block the listed requests hold (their table rows become -1,
 * seq_len 0).  Shared blocks lose one reference and stay intact; a block
 * whose refcount reaches 0 is pushed on the free stack, in (list order, j)
 * order.  req_ids [n] (distinct, in [0, n_rows)), block_table [n_rows][max_blocks],
 * n_freed optional [n].  An id out of range: SV_ERR_STATE, nothing changes. */
sv_status bfl_release(sv_handle* handle, const bfl_state* st, int32_t n, const int32_t* req_ids,
                      int32_t* seq_len, int32_t* block_table, int32_t n_rows, int32_t max_blocks,
                      int32_t* n_freed, sv_stream_t stream);

/* Commit / rollback after the verify pass ([KV]; [CV] 2-3): seq_len_b becomes
 * S_b + 1 + a_b (the old pending token and the a_b accepted drafts are now
 * processed; the correction or bonus token stays pending), or stays S_b when
 * a_b = -1.  Blocks j in [ceil(new/BS), ceil((S_b+k_b+1)/BS)) leave the
 * table; each loses a reference and is pushed on the free stack when that
 * reaches 0, in (request, j) order.  A block with at least one valid slot is
 * kept ([RJ] 2).  K/V payload is never touched.  k [B] (NULL = 0), accepted
 * [B], seq_len [B] in/out, block_table in/out, n_freed optional [B].
 * Inconsistent tables or accepted > k: SV_ERR_STATE, nothing changes. */
sv_status kv_commit_rollback(sv_handle* handle, const bfl_state* st, int32_t B, const int32_t* k,
                             const int32_t* accepted, int32_t* seq_len, int32_t* block_table,
                             int32_t max_blocks, int32_t* n_freed, sv_stream_t stream);

/* Lookahead allocation with copy-on-write ([CV] paragraph 4: copy-on-write
 * addresses physical sharing while the decoder keeps the token and position
 * mapping).  As bfl_reserve, but a request whose last held block is partially
 * filled (r = S_b % BS > 0) and shared (refcount > 1 when the call starts)
 * first gets a fresh block holding a copy of that block's valid slots [0, r)
 * (every layer, K/V and head of kv); the table entry points at the copy and
 * the shared block loses one reference per copy, unchanged for its other
 * owners.  Pops run in (request, j) order, the copy taking j = have - 1; a
 * shared block left without references is pushed on the free stack after
 * every pop, in request order.  cow_scratch [B][3] is caller-owned device
 * memory the call uses between its two kernels.  All or nothing: an exhausted
 * pool (SV_ERR_OOM) or an inconsistent table (SV_ERR_STATE) changes nothing. */
sv_status bfl_reserve_cow(sv_handle* handle, const bfl_state* st, int32_t B, const int32_t* seq_len,
                          const int32_t* k, int32_t* block_table, int32_t max_blocks,
                          const kv_payload* kv, int32_t* cow_scratch, sv_stream_t stream);

/* Commit by copy ([KV]: candidate K/V is appended provisionally, only the
 * accepted part is kept; [RJ] paragraph 1: allocation is not acceptance).
 * The verify pass wrote the K/V of positions S_b .. S_b + k_b (the pending
 * token and the drafts) to stage [B][kmax + 1][layers][2][heads][head_dim];
 * entries i = 0 .. a_b go to their paged slots (block_table[b][p / BS], slot
 * p % BS, p = S_b + i); a_b = -1 copies nothing and rejected entries are never
 * written.  seq_len [B]: S_b, the length BEFORE kv_commit_rollback updates it;
 * accepted [B].  A position without a block in [0, num_blocks): SV_ERR_STATE
 * in the error word, that entry skipped. */
sv_status kv_commit_copy(sv_handle* handle, int32_t B, int32_t kmax, const int32_t* accepted,
                         const int32_t* seq_len, const int32_t* block_table, int32_t max_blocks,
                         int32_t block_size, int32_t num_blocks, const void* stage,
                         const kv_payload* kv, sv_stream_t stream);

/* Commit by copy for a token tree ([CV] paragraph 3: gather the accepted path
 * into the cache layout and drop the sibling states).  stage [B][N+1][L][2]
 * [H][D] holds one K/V entry per tree node (entry 0: the pending token).
 * Position S_b receives entry 0 and position S_b + i (1 <= i <= a_b) the entry
 * of path[b][i-1]; entries of nodes off the path are never written, so no
 * cache position refers to them.  accepted [B] (a_b <= max_depth, the
 * longest path any tree of the batch can give), path [B][N] from
 * spec_verify_tree, seq_len [B] = S_b before kv_commit_rollback (called with
 * k_b = max_depth, or the request's own depth).  A position without a block,
 * or a path entry outside [1, N]: SV_ERR_STATE in the error word, that entry
 * skipped. */
sv_status kv_commit_tree(sv_handle* handle, int32_t B, int32_t N, int32_t max_depth,
                         const int32_t* accepted, const int32_t* path, const int32_t* seq_len,
                         const int32_t* block_table, int32_t max_blocks, int32_t block_size,
                         int32_t num_blocks, const void* stage, const kv_payload* kv,
                         sv_stream_t stream);

/* Draft-cache realignment ([SD] section 4, "update cache state": the draft
 * cache is reconciled with the corrected token; [CV] paragraph 4: the draft
 * follows its own processed-state convention and is never filled from target
 * K/V).  The draft's own pool and table: draft_len_b (in: D_b, the positions
 * the draft processed, however far its proposal loop went) becomes
 * min(D_b, S_b + 1 + a_b), or min(D_b, S_b) when a_b = -1, i.e. only
 * committed tokens stay; a shorter draft catches up on them next round.
 * Blocks j in [ceil(new/BS), ceil(D_b/BS)) leave the table; each loses a
 * reference and is pushed on the free stack when that reaches 0, in
 * (request, j) order.  seq_len [B]: the TARGET length before the pass (S_b;
 * call this before kv_commit_rollback updates it), accepted [B], draft_len [B]
 * in/out, draft_table [B][max_blocks] in/out, n_freed optional [B].
 * A table row not covering its length or accepted < -1: SV_ERR_STATE,
 * nothing changes. */
sv_status kv_commit_draft(sv_handle* handle, const bfl_state* st, int32_t B,
                          const int32_t* seq_len, const int32_t* accepted, int32_t* draft_len,
                          int32_t* draft_table, int32_t max_blocks, int32_t* n_freed,
                          sv_stream_t stream);

/* Contiguous cache ([KV]: rewind the write pointer): write_ptr_b (in: S_b)
 * becomes S_b + 1 + a_b, or stays S_b when a_b = -1.  [B] each. */
sv_status kv_rollback_contig(sv_handle* handle, int32_t B, const int32_t* accepted,
                             int32_t* write_ptr, sv_stream_t stream);

/* Synchronise `stream`, then read and clear the handle's device error word
 * (host *device_code = 0 or an sv_status).  Returns SV_ERR_CUDA if the sync
 * itself failed. */
sv_status sv_get_error(sv_handle* handle, sv_stream_t stream, int32_t* device_code);

#ifdef __cplusplus
}
#endif
#endif /* SPEC_VERIFY_H */
