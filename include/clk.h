/*
 * clk.h -- C ABI of the GB300 (sm_103a) hot path of context-lookup
 * speculative decoding ("lookup drafting").
 *
 * The method (HyperQwen 上下文复述加速：lookup 草稿如何把 25k 文档复读推到
 * 381 tok/s, section "lookup 草稿的原理：三步走"): before every decode step,
 * each request looks up the most recent earlier occurrence of the longest
 * 4-12-token suffix of its own token history and proposes the tokens that
 * follow it (Step 1); that draft is fused with a draft model's 7 head
 * proposals into a verify block of 8 or 16 tokens (Step 2); a per-request
 * scheduler uses the 16-token block only while a copy is in progress, with a
 * sticky exit (Step 3); the target's logits over the block are verified
 * greedily.  The history lookup runs over an index that is maintained
 * incrementally as tokens are committed (the forum thread 单卡 RTX 3090 跑
 * Qwen3.8-27B 381 tok/s？HyperQwen 的思路其实比数字更有意思, the reply's
 * point ①: a full rescan per step backfires on long contexts).
 *
 * Conventions for every entry point
 * ---------------------------------
 * - Return value: CLK_OK (0) or a negative CLK_E* code.  Host-side argument
 *   checks return CLK_EINVAL and launch nothing.  A failed kernel launch
 *   returns CLK_ECUDA.  No C++ exception crosses this boundary.
 * - Asynchrony: every call that takes a clk_stream_t (a cudaStream_t) only
 *   enqueues work on that stream; none synchronises, except clk_status,
 *   clk_read_counters, clk_read_slot_info, clk_lookup_read_history and
 *   clk_lookup_restore_state, which say so.
 * - Device errors: problems that can only be seen on the device (a history
 *   capacity overflow, a token outside [0, vocab), a bad slot index, a bad
 *   block length) are latched into a status word inside the lookup
 *   workspace; the first one wins; clk_status reads it.  The work item that
 *   hit the error is skipped; the rest of the batch proceeds.
 * - Memory: the library never allocates device memory.  Every buffer is
 *   owned by the caller (e.g. PyTorch tensors) and passed as a plain device
 *   pointer ("d_" prefix) or host pointer ("h_" prefix).  Integer arrays are
 *   int32, C-contiguous, 4-byte aligned, with the shapes given below.
 * - Logits: d_logits of the verify entry points may also point into
 *   page-locked host memory (cudaHostAlloc / cudaMallocHost, or
 *   cudaHostRegister'ed), which unified addressing lets kernels load from
 *   with the same pointer.  The kernels then read the rows they verify in
 *   place over the host link, and only those rows: no staging copy of the
 *   whole [B, rows, V] array.  Results are identical to device logits.
 * - Requests are addressed by slot (0 <= slot < max_slots).  A batch is a
 *   device array d_slots[B] of distinct slots; per-request arrays of the
 *   call are indexed by batch position b, not by slot.
 * - Threading: one lookup handle is used from one stream at a time.
 * - Sentinel: CLK_SENT (-1) marks an empty draft or output slot.  It never
 *   equals an argmax, so verification always stops on it.
 */
#ifndef CLK_H
#define CLK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* clk_stream_t; /* the same type as cudaStream_t */

#if defined(__GNUC__)
#define CLK_API __attribute__((visibility("default")))
#else
#define CLK_API
#endif

enum {
    CLK_OK = 0,
    CLK_EINVAL = -1,    /* bad argument */
    CLK_ECAPACITY = -2, /* history or index capacity exceeded */
    CLK_ECUDA = -3,     /* CUDA runtime error */
    CLK_ENOTIMPL = -4,  /* not supported by the compiled library */
    CLK_ESTATE = -5     /* call out of order (e.g. handle not set up) */
};

enum { CLK_DTYPE_BF16 = 0, CLK_DTYPE_F32 = 1 };

#define CLK_SENT (-1)
#define CLK_BLOCK 16        /* slots in a verify block and in a lookup draft */
#define CLK_MAX_K 16        /* upper limit of max_k */
#define CLK_MAX_BATCH 8192  /* upper limit of B in one call */

/* Method constants (defaults in brackets).  Step 2 and Step 3 of the
 * article's "三步走" section fix the defaults; the block is 1 committed
 * token + head + tail drafts. */
typedef struct clk_params {
    int32_t min_k;           /* [4]  shortest suffix match that counts (Step 1: 4-12) */
    int32_t max_k;           /* [12] longest suffix searched (<= CLK_MAX_K) */
    int32_t head;            /* [7]  draft-model head slots 1..head (Step 2) */
    int32_t tail;            /* [8]  lookup-only tail slots (Step 2; DFLASH_TOKENS=15) */
    int32_t head_replace_k;  /* [8]  match that replaces the head outright */
    int32_t head_agree_k;    /* [6]  match that replaces it if the drafter agrees */
    int32_t head_agree_n;    /* [2]  leading proposals that must agree */
    int32_t tail_k;          /* [4]  match that fills the tail (and raises the flag) */
    int32_t enter_streak;    /* [2]  consecutive qualifying steps to enter the long block */
    int32_t sticky;          /* [3]  flag-down steps kept in the long block (STICKY=3) */
    int32_t near_full_slack; /* [1]  rejected drafts that still count as nearly full */
} clk_params;

/* Per-slot counters (clk_read_counters).  accept_hist[x][a] counts steps with
 * block class x (0 = short, 1 = long) that accepted a drafts. */
typedef struct clk_counters {
    int64_t steps;      /* scheduler steps */
    int64_t hits;       /* steps whose lookup matched (k >= min_k) */
    int64_t long_steps; /* steps that used the long block */
    int64_t drafted;    /* non-sentinel drafts placed in verify blocks */
    int64_t accepted;   /* drafts accepted (sum of a) */
    int64_t emitted;    /* tokens committed by steps (sum of a + 1) */
    int64_t accept_hist[2][16];
} clk_counters;

/* Scheduler and history state of one slot (clk_read_slot_info). */
typedef struct clk_slot_info {
    int32_t n;        /* history length */
    int32_t mode;     /* 0 = short block, 1 = long block */
    int32_t streak;   /* consecutive qualifying steps while short */
    int32_t miss;     /* consecutive flag-down steps while long */
    int32_t has_prev; /* a scheduler step has run since the slot was set up */
    int32_t cur_len;  /* block length chosen by the last scheduler step, 0 after append */
    int32_t n_indexed; /* the index holds every k-gram ending before position n_indexed - 1; the
                          positions committed since are indexed by the next proposal launches, and
                          n_indexed is raised by the launch after the one that indexed them */
} clk_slot_info;

typedef struct clk_lookup clk_lookup; /* opaque host handle */

/* Fills *p with the defaults above. */
CLK_API void clk_params_default(clk_params* p);

/* CLK_OK if *p is usable: 1 <= min_k <= max_k <= CLK_MAX_K,
 * 1 + head + tail <= CLK_BLOCK, head_agree_n <= head, enter_streak >= 1,
 * and the other fields >= 0; CLK_EINVAL otherwise. */
CLK_API int clk_params_check(const clk_params* p);

/* Text for a status code (static storage). */
CLK_API const char* clk_status_string(int code);

/* ---------------------------------------------------------------------- */
/* Lookup state: histories, the incremental index, scheduler state.        */
/* ---------------------------------------------------------------------- */

/* Bytes of device workspace for `max_slots` requests whose histories hold up
 * to `max_hist` tokens each (prompt plus every committed token).  The
 * workspace holds the histories, the per-request k-gram index (one
 * open-addressing table of 2^ceil(log2(2*max_hist)) 4-byte entries per match
 * length min_k..max_k: 8 * 9 = 72 bytes of index per history token at the
 * defaults, before each table is rounded up to a power of two), the
 * scheduler state with a copy of each history's last 64 tokens, the
 * counters, the fused verify's scratch and the status word.  Returns
 * CLK_EINVAL for bad sizes. */
CLK_API int clk_lookup_workspace_bytes(const clk_params* p, int32_t max_slots, int64_t max_hist, size_t* bytes);

/* Creates a host handle over a caller-owned device workspace of at least
 * clk_lookup_workspace_bytes bytes, 256-byte aligned.  Allocates only the
 * host handle (freed by clk_lookup_destroy).  Tokens must lie in
 * [0, vocab) (vocab <= 0: any token >= 0).  The workspace content is
 * undefined until clk_lookup_reset has run on it. */
CLK_API int clk_lookup_create(clk_lookup** h, const clk_params* p, int32_t max_slots, int64_t max_hist,
                              int32_t vocab, void* d_workspace, size_t bytes);

/* Zeroes the whole workspace (every slot empty, status clear). */
CLK_API int clk_lookup_reset(clk_lookup* h, clk_stream_t s);

/* Sets up the B slots d_slots[B] with the prompts given in CSR layout:
 * request b's prompt is d_prompt[d_prompt_off[b] .. d_prompt_off[b+1]) (int64
 * offsets, device).  Each slot's history becomes its prompt, its scheduler
 * state and counters are cleared, and its k-gram index is rebuilt from the
 * prompt (the 4-gram level and the longer levels, each mapping a k-gram to
 * its most recent end position, so that the lookup never rescans the
 * history).  A prompt must hold 1 .. max_hist tokens; otherwise the slot is
 * left empty and CLK_ECAPACITY (too long) or CLK_EINVAL (empty) is latched. */
CLK_API int clk_lookup_init(clk_lookup* h, const int32_t* d_slots, int32_t B, const int32_t* d_prompt,
                            const int64_t* d_prompt_off, clk_stream_t s);

/* Commits tokens: appends d_tok[b][0 .. d_count[b]) (d_tok is [B,16]) to slot
 * d_slots[b]'s history and inserts every k-gram that the new tokens complete
 * into its index.  A count of 0 is allowed.  A count outside [0, 16], a
 * token outside [0, vocab) or an overflow of max_hist latches an error and
 * skips that request.  If the slot's last scheduler step has not been
 * committed yet, the append counts as that step's commit (a = count - 1)
 * in the counters.  (Article, "三步走" Step 1: the lookup runs over the
 * request's own history, which grows by the committed tokens.) */
CLK_API int clk_lookup_append(clk_lookup* h, const int32_t* d_slots, int32_t B, const int32_t* d_tok,
                              const int32_t* d_count, clk_stream_t s);

/* Step 1 of "三步走": for each request, k = the longest suffix length in
 * [min_k, max_k] of its history h[0..n) that occurred earlier, overlap
 * allowed, and j = the largest position with h[j-k .. j) == h[n-k .. n) and
 * k <= j <= n-1 (the most recent occurrence of that suffix); k = 0, j = -1
 * when none.  The draft is d_draft[b][i] = h[j + (i mod (n - j))] for
 * i = 0..15: the tokens that followed the occurrence, continued as an LZ77
 * copy at distance n - j past the end of the history (all CLK_SENT when
 * k = 0).  Outputs: d_draft [B,16], d_k [B], d_j [B].  The launch also
 * indexes tokens committed by clk_verify_append since the slot's earlier
 * proposals: all of them when more than 16 are pending or B > 32; else it
 * may leave up to 16 to the next proposal launch on the handle (which runs
 * them before its own wait when a clk_verify_append came in between).  The
 * answers never depend on which launch indexes a position: pending
 * positions are checked directly. */
CLK_API int clk_lookup_propose(clk_lookup* h, const int32_t* d_slots, int32_t B, int32_t* d_draft, int32_t* d_k,
                               int32_t* d_j, clk_stream_t s);

/* The same proposal as clk_lookup_propose, by the pages' own method: a scan
 * of the whole history h[0..n) for every earlier occurrence of the suffix
 * ("三步走", Step 1: one scan per request; most candidates fail on their first
 * tokens, the survivors are extended up to max_k), without the index.  Cost
 * O(n) per request per call; kept as the ablation of the incremental index.
 * ctas_per_request: 1 scans each request's history in one CTA, the pages'
 * form (one program per request); n > 1 splits it over n CTAs; 0 takes one
 * CTA per 4,096 positions of the workspace's history capacity.  Any value
 * gives the same answers.  Outputs and errors as clk_lookup_propose
 * (CLK_EINVAL for a negative ctas_per_request); the index is not touched. */
CLK_API int clk_lookup_propose_scan(clk_lookup* h, const int32_t* d_slots, int32_t B, int32_t ctas_per_request,
                                    int32_t* d_draft, int32_t* d_k, int32_t* d_j, clk_stream_t s);

/* Step 3 of "三步走" (the long-block scheduler), one step per request.  The
 * flag is k >= tail_k (the lookup can fill the tail); nearly full means the
 * previous step accepted prev_accept >= prev_len - 1 - near_full_slack
 * drafts (there is no previous step right after clk_lookup_init).  A short
 * request enters the long block when the flag and the nearly-full signal
 * held on enter_streak consecutive steps; a long request leaves it when the
 * flag has been down on more than `sticky` consecutive steps.  Writes
 * d_len[b] = 1 + head + tail (long) or 1 + head (short).  d_len may alias
 * d_prev_len, and d_prev_accept may alias an output of the previous step.
 * Updates the slot's steps / hits / long_steps / drafted counters. */
CLK_API int clk_sched_step(clk_lookup* h, const int32_t* d_slots, int32_t B, const int32_t* d_k,
                           const int32_t* d_prev_accept, const int32_t* d_prev_len, int32_t* d_len, clk_stream_t s);

/* Step 2 of "三步走" (fusion), stateless.  d_block[b][0] = d_last_tok[b];
 * head slots 1..head take the lookup draft d_draft[b][0..head) when
 * k >= head_replace_k, or when k >= head_agree_k and the draft model's first
 * head_agree_n proposals d_head[b][..] equal the lookup's; otherwise they
 * take d_head[b][0..head).  Tail slots head+1 .. head+tail take
 * d_draft[b][head ..] when d_len[b] is the long length and k >= tail_k;
 * otherwise, and beyond the block, CLK_SENT.  d_head is [B, head]. */
CLK_API int clk_fuse(const clk_params* p, int32_t B, const int32_t* d_last_tok, const int32_t* d_draft, const int32_t* d_k,
                     const int32_t* d_head, const int32_t* d_len, int32_t* d_block, clk_stream_t s);

/* clk_sched_step followed by clk_fuse in one launch, with the last token read
 * from the slot's history.  Bit-identical to the two calls. */
CLK_API int clk_fuse_sched(clk_lookup* h, const int32_t* d_slots, int32_t B, const int32_t* d_draft, const int32_t* d_k,
                           const int32_t* d_head, const int32_t* d_prev_accept, const int32_t* d_prev_len, int32_t* d_len,
                           int32_t* d_block, clk_stream_t s);

/* clk_lookup_propose, clk_sched_step and clk_fuse in one launch (one CTA per
 * request).  Bit-identical to the three calls.  Like clk_lookup_propose it
 * first waits for the preceding launch on the stream (programmatic dependent
 * launch) and indexes the tokens that clk_verify_append committed since the
 * slot's earlier proposals (some of them possibly left to the next
 * proposal, as there).  When the handle's last fused verify was
 * clk_verify_append, the launch lets the next launch on the stream (the
 * step's clk_verify_append, which starts streaming its predicted rows) begin
 * before that wait; otherwise only after it. */
CLK_API int clk_propose_fuse_sched(clk_lookup* h, const int32_t* d_slots, int32_t B, const int32_t* d_head,
                                   const int32_t* d_prev_accept, const int32_t* d_prev_len, int32_t* d_draft,
                                   int32_t* d_k, int32_t* d_j, int32_t* d_len, int32_t* d_block, clk_stream_t s);

/* ---------------------------------------------------------------------- */
/* Greedy verification                                                     */
/* ---------------------------------------------------------------------- */

/* Scratch bytes for clk_verify_greedy with up to B requests. */
CLK_API int clk_verify_scratch_bytes(int32_t B, size_t* bytes);

/* Zeroes a verify scratch buffer; required once before its first use (each
 * call leaves it zeroed again; re-run it after any failed call). */
CLK_API int clk_verify_scratch_init(void* d_scratch, size_t bytes, clk_stream_t s);

/* Greedy verification (article, "三步走", last paragraph: greedy
 * verification never reads the draft distribution; the Polish page "Jak
 * DFlash2 przyspiesza Qwen3.8 i skraca kontekst": the first rejected
 * proposal ends the run).  For request b with block length L = d_len[b]
 * (1..16) and block d_block[b][0..16):
 *   g_r = argmax_v logits[b, r, v] for r < L (values compared as float32,
 *         the lowest index wins ties, +0 == -0, the first NaN wins);
 *   a   = the largest a <= L-1 with d_block[b][r+1] == g_r for all r < a;
 *   emitted = a + 1: the accepted drafts and the target's token after them.
 * Logits element (b, r, v) is at d_logits + b*req_stride + r*row_stride + v
 * (element strides), dtype CLK_DTYPE_BF16 or CLK_DTYPE_F32; rows r >= L are
 * never read.  Outputs: d_argmax [B,16] (g_r, CLK_SENT for r >= L),
 * d_accept [B], d_emitted [B], d_out_tok [B,16] (g_0..g_a, then CLK_SENT).
 * A request whose L is outside 1..16 gets a = 0, emitted = 0 and all-SENT
 * rows.  d_scratch: clk_verify_scratch_bytes(B) bytes, zeroed once by
 * clk_verify_scratch_init; calls that share a scratch buffer must not
 * overlap.  Runs as one grid sized to fill every SM. */
CLK_API int clk_verify_greedy(const void* d_logits, int32_t dtype, int64_t row_stride, int64_t req_stride, int32_t V,
                              int32_t B, const int32_t* d_block, const int32_t* d_len, int32_t* d_argmax,
                              int32_t* d_accept, int32_t* d_emitted, int32_t* d_out_tok, void* d_scratch,
                              size_t scratch_bytes, clk_stream_t s);

/* clk_verify_greedy for callers that cannot allocate device memory at all:
 * for example a plugin that is handed only its input and output pointers,
 * or a serving engine whose free HBM is already committed to its own pools
 * and which has no way to give this library a scratch buffer.  It takes
 * the same arguments minus the scratch and computes the same outputs.  It
 * allocates nothing: its scratch is a fixed array of
 * CLK_STATIC_VERIFY_MAX_BATCH * 17 * 8 bytes (139,264 bytes) inside the
 * library, which every GPU that loads the library keeps until the process
 * exits.  B above CLK_STATIC_VERIFY_MAX_BATCH returns CLK_ECAPACITY (any such
 * B, also beyond CLK_MAX_BATCH) and launches nothing.  The first call on
 * each device looks up the array's device address (cudaGetSymbolAddress),
 * and so does the first call after the device's context changed (after
 * cudaDeviceReset, say); make that first call before any stream capture.  Each call clears the part of the array it uses on its
 * stream and then launches the verify kernel.  All calls share the one
 * array, so calls whose executions overlap on the GPU (other streams, other
 * threads) race and corrupt each other's results: serialise them.  The
 * pages describe no counterpart; this entry point exists for such callers. */
#define CLK_STATIC_VERIFY_MAX_BATCH 1024
CLK_API int clk_verify_greedy_static(const void* d_logits, int32_t dtype, int64_t row_stride, int64_t req_stride,
                                     int32_t V, int32_t B, const int32_t* d_block, const int32_t* d_len,
                                     int32_t* d_argmax, int32_t* d_accept, int32_t* d_emitted, int32_t* d_out_tok,
                                     clk_stream_t s);

/* clk_verify_greedy followed by clk_lookup_append of its d_out_tok /
 * d_emitted, in one launch: each request's tokens are committed to its
 * history as soon as its rows are verified; the k-grams they complete are
 * indexed by the following clk_lookup_propose / clk_propose_fuse_sched /
 * clk_lookup_append calls on the slot (which see the same answers as with an
 * immediate index update).  Uses the scratch inside the lookup workspace.
 * Results are bit-identical to the two calls.
 * Launch order: the launch is a programmatic dependent of the preceding
 * launch on the stream, and d_block / d_len may come from that launch
 * (clk_propose_fuse_sched).  Before it waits for it, it reads the rows of a
 * predicted length of every request: max(1 + head, d_len_hint[b]) when the
 * hint is a valid length, else 1 + head (the short block, which every block
 * covers); after the wait it reads the rows the prediction missed.
 * d_len_hint (nullable) is only a prediction, e.g. the previous step's
 * lengths in a buffer the preceding launch does not write: any value gives
 * the same results, a good one saves a second pass.  So the logits must
 * already be complete when this call is made (as after any ordinary kernel
 * or copy on the stream) and must hold every predicted row (16 rows per
 * request serve any hint).  Consecutive calls on a handle alternate between
 * two halves of the scratch in the workspace, so that a call may start
 * streaming while the previous one finishes (clk_propose_fuse_sched between
 * them lets it); a call lets the next launch on the stream start only after
 * its own wait. */
CLK_API int clk_verify_append(clk_lookup* h, const int32_t* d_slots, const void* d_logits, int32_t dtype,
                              int64_t row_stride, int64_t req_stride, int32_t V, int32_t B, const int32_t* d_block,
                              const int32_t* d_len, const int32_t* d_len_hint, int32_t* d_argmax,
                              int32_t* d_accept, int32_t* d_emitted, int32_t* d_out_tok, clk_stream_t s);

/* Sampling verification with point-mass drafts (HyperQwen context-lookup
 * article, closing paragraph of "lookup 草稿的原理：三步走": for sampled
 * requests every drafted position is a point mass on its proposed token,
 * a proposal the standard speculative rejection sampler accepts, so the
 * emitted tokens follow plain sampling from the target).
 *
 * For request b, row r < L_b of the logits gives the target distribution
 * p_r = softmax(x_r * inv_temp[b]).  The draft c = block[b][r + 1] is
 * accepted iff u[b][r][0] < p_r(c).  At the first rejected row the emitted
 * token is drawn from p_r with c removed (renormalised) using u[b][r][1]; if
 * all L_b - 1 drafts are accepted, the bonus token is drawn from p_{L_b - 1}
 * using u[b][L_b - 1][1].  A draw with uniform u is the first token whose
 * running probability sum exceeds u.  A draft outside [0, V) (CLK_SENT) is
 * rejected and its row's whole distribution is drawn from.
 *
 * Layouts are those of clk_verify_greedy: logits [B, rows >= L_b, V] with
 * element strides, block [B, 16], len [B].  inv_temp: float32 [B], 1 /
 * temperature, > 0 and finite.  uniform: float32 [B, 16, 2] in [0, 1), the
 * acceptance and the draw uniform of every row (the caller's random
 * numbers; rows past L_b are not read).  Outputs: d_accept [B] (accepted
 * drafts a), d_emitted [B] (a + 1), d_out_tok [B, 16] (the a accepted drafts,
 * the drawn token, then CLK_SENT).  A request with L_b outside 1..16 or an
 * invalid inv_temp gets accept 0, emitted 0 and all CLK_SENT.  Logits must
 * be finite (-inf entries have weight 0).
 *
 * Computation is in float32; the results do not depend on the launch
 * configuration or on timing.  Only the L_b rows are read, once, plus one
 * 16,384-element segment of the drawn row.
 *
 * Scratch: a caller-owned device buffer of at least
 * clk_verify_sample_scratch_bytes(dtype, V, B) bytes, 16-byte aligned,
 * zeroed once before its first use (e.g. clk_verify_scratch_init); every
 * call leaves it ready for the next.  Calls sharing a scratch buffer must
 * not overlap on the GPU.  Errors: CLK_EINVAL for a bad dtype, size,
 * stride, pointer or scratch size (nothing is launched); CLK_ECUDA for a
 * launch failure. */
CLK_API int clk_verify_sample_scratch_bytes(int32_t dtype, int32_t V, int32_t B, size_t* bytes);
CLK_API int clk_verify_sample(const void* d_logits, int32_t dtype, int64_t row_stride, int64_t req_stride,
                              int32_t V, int32_t B, const int32_t* d_block, const int32_t* d_len,
                              const float* d_inv_temp, const float* d_uniform, int32_t* d_accept,
                              int32_t* d_emitted, int32_t* d_out_tok, void* d_scratch, size_t scratch_bytes,
                              clk_stream_t s);

/* clk_verify_sample with the target's weights defined as integers, so that
 * every acceptance and every draw is an integer comparison: the results are
 * a fixed function of the logits, drafts, lengths, temperatures and
 * uniforms, which another implementation of the same definition reproduces
 * bit for bit.  The rule (accept iff u_acc < p_r(c), draw from the residual
 * or the last row, inverse CDF) is clk_verify_sample's; only p_r changes:
 *
 *   s = fl32(inv_temp * fl32(log2 e)); each row is cut into chunks of 1024
 *   entries (the last one ragged).  Chunk k's reference is
 *   R_k = ceil(fl32(M_k * s)), M_k its largest entry.  An entry x of chunk k
 *   weighs q = Q(fma(x, s, -R_k)) with, for d >= -32, n = rint(d) (ties to
 *   even), r = d - n, f = P(r) the degree-6 Taylor polynomial of
 *   2^(r + 1/2) (coefficients sqrt(2) (ln 2)^j / j! rounded to float,
 *   evaluated by Horner's rule with fused multiply-adds) and
 *   Q(d) = floor(64 (bits(f) - bits(0.5f)) / 2^-n + 1/2), about
 *   2^(d + 29.5); Q(d) = 0 below -32.  S_k = the chunk's sum of q.  Row
 *   units are 2^-12 of a unit of the row's reference R = max_k R_k: a chunk
 *   quantity v counts U(v, e) = floor(v * 2^(12 - e)), e = R - R_k, and the
 *   row's total is T = sum_k U(S_k, e_k).
 *   A draft c in chunk kc is accepted iff floor(k(u_acc) T / 2^24) <
 *   U(q_c, e_kc), with k(u) = floor(u * 2^24) clamped to [0, 2^24 - 1].
 *   The draw with u_smp takes t = floor(k(u_smp) T' / 2^24), T' the sum of
 *   the chunks' totals with c's weight taken out of its chunk (nothing taken
 *   out after a full acceptance or a sentinel draft); the chunk is the
 *   first whose running total exceeds t, and the token the first entry of
 *   it (c skipped) whose running sum of q exceeds the remainder of t taken
 *   back to chunk units (times 2^(e - 12), rounded down).
 *
 * p_r differs from the float softmax by about 2^-22 relative per weight
 * (the polynomial and float rounding) plus half a unit of each weight;
 * entries more than about 30 binades below their chunk's largest entry
 * weigh 0.  A request any of whose L_b rows has a chunk with
 * |fl32(M_k * s)| > 2^22, or only -inf entries, gets the empty result, as
 * does an invalid length or temperature.  V is at most 4,194,304
 * (CLK_EINVAL above).  Logits must be finite or -inf (NaN entries:
 * unspecified result, no fault).
 *
 * Arguments, layouts, outputs and errors are those of clk_verify_sample;
 * the scratch must hold clk_verify_sample_exact_scratch_bytes(dtype, V, B)
 * bytes (16-byte aligned, zeroed once before its first use, left ready for
 * the next call; calls sharing it must not overlap on the GPU).  Every row
 * is read once, plus one 1024-entry chunk of the drawn row. */
CLK_API int clk_verify_sample_exact_scratch_bytes(int32_t dtype, int32_t V, int32_t B, size_t* bytes);
CLK_API int clk_verify_sample_exact(const void* d_logits, int32_t dtype, int64_t row_stride, int64_t req_stride,
                                    int32_t V, int32_t B, const int32_t* d_block, const int32_t* d_len,
                                    const float* d_inv_temp, const float* d_uniform, int32_t* d_accept,
                                    int32_t* d_emitted, int32_t* d_out_tok, void* d_scratch, size_t scratch_bytes,
                                    clk_stream_t s);

/* clk_verify_sample followed by clk_lookup_append of its d_out_tok /
 * d_emitted, in one launch: the sampled step of a decode loop.  Each
 * request's emitted tokens are committed to the history of d_slots[b] as
 * soon as its draw is made; the k-grams they complete are indexed by the
 * next proposal call on the slot.  The results equal those of the two
 * calls.  The launch is a programmatic dependent of the preceding launch on
 * the stream, and d_block / d_len may come from that launch
 * (clk_propose_fuse_sched).  As in clk_verify_append, it first reads the
 * rows of a predicted length of every request with a valid temperature:
 * max(1 + head, d_len_hint[b]) when the hint is a valid length, else
 * 1 + head; after waiting for that launch it reads the rows the prediction
 * missed.  d_len_hint (nullable, e.g. the previous step's lengths in a
 * buffer the preceding launch does not write) is only a prediction: any
 * value gives the same results.  So the logits (every predicted row; 16
 * rows per request serve any hint), the inverse temperatures and the
 * uniforms must be complete when the call is made.  A request with an
 * invalid length or temperature gets the empty result, commits nothing and
 * latches CLK_EINVAL in the handle's status (as do a bad slot, an
 * out-of-vocabulary token or a full history, which clk_lookup_append would
 * reject).  Scratch as for clk_verify_sample; calls sharing it must not
 * overlap on the GPU.  A scratch whose halves (each half of its size,
 * rounded down to a multiple of 256 bytes) each hold the needed size is used
 * as two halves that consecutive calls on the handle alternate (all of it
 * zeroed before the first use; the halves do not move with the batch): then,
 * as after
 * clk_verify_append, the next clk_propose_fuse_sched lets the next call
 * start streaming before its own wait, and a call lets the next launch on
 * the stream start only after its own wait.  With a smaller scratch the next
 * proposal lets the next call start only after that wait. */
CLK_API int clk_verify_sample_append(clk_lookup* h, const int32_t* d_slots, const void* d_logits, int32_t dtype,
                                     int64_t row_stride, int64_t req_stride, int32_t V, int32_t B,
                                     const int32_t* d_block, const int32_t* d_len, const int32_t* d_len_hint,
                                     const float* d_inv_temp, const float* d_uniform, int32_t* d_accept,
                                     int32_t* d_emitted, int32_t* d_out_tok, void* d_scratch, size_t scratch_bytes,
                                     clk_stream_t s);

/* clk_verify_sample_exact followed by clk_lookup_append of its d_out_tok /
 * d_emitted, in one launch: the sampled step of a decode loop on the exact
 * (fixed-point) weights.  Everything else is as for
 * clk_verify_sample_append: a programmatic dependent of the preceding launch,
 * the rows of a predicted length read before the wait (d_len_hint only a
 * prediction), the empty result, no commit and CLK_EINVAL latched for an
 * invalid length, temperature, slot or token, and the two scratch halves;
 * the scratch holds clk_verify_sample_exact_scratch_bytes(dtype, V, B) (or
 * twice that, rounded up to 256 bytes, for the halves).  A request with a row
 * that cannot be weighed (clk_verify_sample_exact) also gets the empty
 * result, commits nothing and latches CLK_EINVAL.  The results equal those
 * of clk_verify_sample_exact and clk_lookup_append. */
CLK_API int clk_verify_sample_exact_append(clk_lookup* h, const int32_t* d_slots, const void* d_logits, int32_t dtype,
                                           int64_t row_stride, int64_t req_stride, int32_t V, int32_t B,
                                           const int32_t* d_block, const int32_t* d_len, const int32_t* d_len_hint,
                                           const float* d_inv_temp, const float* d_uniform, int32_t* d_accept,
                                           int32_t* d_emitted, int32_t* d_out_tok, void* d_scratch,
                                           size_t scratch_bytes, clk_stream_t s);

/* ---------------------------------------------------------------------- */
/* Status, counters, inspection (these synchronise the stream)             */
/* ---------------------------------------------------------------------- */

/* Synchronises `s`, returns the latched device status in *dev_status (CLK_OK
 * if none) and, if detail != NULL, the slot (or batch position) it came
 * from.  The status stays latched until clk_status_clear. */
CLK_API int clk_status(clk_lookup* h, int32_t* dev_status, int32_t* detail, clk_stream_t s);
CLK_API int clk_status_clear(clk_lookup* h, clk_stream_t s);

/* Synchronises `s` and copies slot `slot`'s counters (slot = -1: the sum
 * over all slots) into *out. */
CLK_API int clk_read_counters(clk_lookup* h, int32_t slot, clk_counters* out, clk_stream_t s);

/* Synchronises `s` and copies slot `slot`'s scheduler/history state. */
CLK_API int clk_read_slot_info(clk_lookup* h, int32_t slot, clk_slot_info* out, clk_stream_t s);

/* Synchronises `s` and copies up to `cap` tokens of slot `slot`'s history
 * into host memory h_out; *n_out receives the history length. */
CLK_API int clk_lookup_read_history(clk_lookup* h, int32_t slot, int32_t* h_out, int64_t cap, int64_t* n_out,
                                    clk_stream_t s);

/* Checkpoint / resume of one request.  A snapshot is three reads:
 * clk_lookup_read_history, clk_read_slot_info and clk_read_counters (the
 * slot's own).  To resume it, in the same or another workspace with the same
 * parameters: clk_lookup_init(slot, history) rebuilds the history and its
 * index, then this call writes back the scheduler state (mode, streak, miss,
 * has_prev, cur_len) and the counters.  info->n must equal the slot's
 * history length; mode must be 0 or 1, streak and miss >= 0, has_prev 0 or
 * 1, cur_len 0 or a block length 1..16; else CLK_EINVAL and nothing is
 * written.  n_indexed and the index itself stay as clk_lookup_init left
 * them.  The caller keeps the previous step's accepted count and block
 * length (the inputs of the next scheduler step) with the snapshot.
 * Synchronises `s`. */
CLK_API int clk_lookup_restore_state(clk_lookup* h, int32_t slot, const clk_slot_info* info,
                                     const clk_counters* counters, clk_stream_t s);

/* Launch setting of the handle's fused verify calls (clk_verify_append,
 * clk_verify_sample_append).  alone = 0 (the default): a call expects to
 * follow the step's proposal launch directly on the stream and to overlap
 * it, so it gives its CTAs that will be dispatched behind the proposal's
 * CTAs a smaller share of the rows.  alone = 1: each call is launched with
 * nothing to overlap (e.g. other work or event records between the
 * launches), and every CTA gets an even share.  Results do not depend on it;
 * only the timing does.  Host-side only: affects the calls made after it.
 * CLK_ESTATE for a bad handle. */
CLK_API int clk_lookup_set_alone(clk_lookup* h, int32_t alone);

/* Frees the host handle (not the workspace). */
CLK_API void clk_lookup_destroy(clk_lookup* h);

#ifdef __cplusplus
}
#endif

#endif /* CLK_H */
