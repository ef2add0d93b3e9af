/*
 * sdva.h -- C ABI of the speculative-decoding verify step on one GB300 GPU.
 *
 * One speculative round of single-model LLM serving ends with a verify step:
 * the main model takes the lane's window of 1 + d tokens (the last committed
 * token followed by d drafted tokens), writes their K/V into the paged KV
 * cache, runs one attention pass of the whole window over the cached context,
 * and accepts the longest drafted prefix its own argmax agrees with.
 * Sources: Baseten talk summary, section "추측 디코드" (drafts are checked
 * by the main model in a single forward pass and the accepted ones are
 * streamed); NInfer review (blog.123qwe.co.kr/?p=4624), section "아키텍처 ③"
 * (MTP proposes 1..5 drafts, DFlash/DFlash2 1..15) and section "아키텍처 ①"
 * (output stays provisional until the model accepts the commit).
 *
 * This library implements the three data-parallel calls of that step:
 *   kv_append_quant  -- write new K/V rows into the quantised, paged cache
 *   kv_append_quant_ragged -- the same with a token count per lane
 *   verify_attn      -- batched, causal-in-window, GQA attention of every
 *                       lane's window over its whole cached context
 *   verify_attn_tree -- the same for a window that holds a draft tree
 *   verify_attn_ragged -- the same with a window row count per lane
 *   spec_accept      -- argmax per window position, longest agreeing draft
 *                       prefix, optional commit of the new lengths
 *   spec_accept_lazy -- the same acceptance reading each lane's rows only up
 *                       to its first disagreement, with per-lane draft counts
 *   spec_accept_tree -- greedy acceptance of a tree of drafted tokens
 *   spec_accept_sampled -- lossless stochastic acceptance with the draft
 *                       distribution (ratio test, residual draw)
 *   verify_step      -- append, verify_attn and spec_accept as one chain of
 *                       programmatic dependent launches
 *
 * Conventions for every call
 *   - Every pointer argument is a DEVICE pointer (cudaMalloc / torch CUDA
 *     memory on the current device) unless stated otherwise; the caller owns
 *     all memory.  The library allocates nothing, keeps no per-call state and
 *     never synchronises: every call only enqueues kernels on `stream`
 *     (NULL = the legacy default stream) and returns.
 *   - Host-side argument errors are returned as negative codes (SDVA_ERR_*)
 *     before anything is enqueued.  Errors that depend on device data (a bad
 *     page id, a lane whose length does not fit, an out-of-vocabulary draft,
 *     a per-lane count out of range, a draft tree whose parent is not an
 *     earlier slot) are reported by OR-ing SDVA_STATUS_* bits into the
 *     optional device int `*status`; the affected lane is skipped as
 *     documented per call, never trapped.  Read `*status` after the stream
 *     has completed.
 *   - Launch shapes depend only on host arguments, so every call can be
 *     captured in a CUDA graph and replayed.
 *   - Inputs are not modified except where a parameter says "in/out".
 *     Outputs must not alias inputs.
 *
 * KV cache layout (reading taken for the pages' "FP8 E4M3" KV and 4-bit KV;
 * NInfer review section "성능과 평가", MegaCapybara announcement item 2):
 *   page_size = 64 tokens, head_dim = 128, pages shared by all kv heads.
 *   SDVA_KV_FP8_E4M3:
 *     k_codes, v_codes : uint8  [num_pages][num_kv_heads][64][128]  OCP E4M3
 *     k_scales, v_scales: float [num_pages][num_kv_heads]
 *     value = e4m3(code) * scale.  The scale of a (page, head) only grows while
 *     the page fills: an append starting at page offset 0 sets it to amax/448;
 *     a later append into the same page raises it to max(old, amax/448) and,
 *     if it grew, re-encodes the page's earlier tokens as
 *     e4m3_rne_sat(fp32(e4m3(c) * s_old) / s_new).  New tokens are encoded as
 *     e4m3_rne_sat(x / s) (fp32 IEEE division, round to nearest even,
 *     saturating to +-448); a zero scale gives zero codes.
 *   SDVA_KV_INT4_G32:
 *     k_codes, v_codes : uint8  [num_pages][num_kv_heads][64][64]
 *                        dim 2i in the low nibble, dim 2i+1 in the high
 *                        nibble, two's complement, values in [-7, 7]
 *     k_scales, v_scales: fp16 bits [num_pages][num_kv_heads][64][4]
 *                        one scale per token and group of 32 head dims
 *     s = fp16_rne(min(amax_group / 7, 65504)); code = clamp(rint(x / s), -7, 7)
 *     with halves to even; value = code * s.
 *   SDVA_KV_INT8_G64 (the same review section's "INT8 group-64"):
 *     k_codes, v_codes : int8   [num_pages][num_kv_heads][64][128]  two's complement
 *     k_scales, v_scales: fp16 bits [num_pages][num_kv_heads][64][2]
 *                        one scale per token and group of 64 head dims
 *     s = fp16_rne(min(amax_group / 127, 65504)); code = clamp(rint(x / s), -127, 127)
 *     with halves to even; value = code * s.
 *   SDVA_KV_FP8_ROW (the same section's "FP8 E4M3 row-256", read as one
 *   scale per row of a token's head, 128 dims here):
 *     k_codes, v_codes : uint8  [num_pages][num_kv_heads][64][128]  OCP E4M3
 *     k_scales, v_scales: float [num_pages][num_kv_heads][64]  one per token
 *     s = amax_row / 448 (fp32 IEEE division); code = e4m3_rne_sat(x / s); a
 *     zero scale gives zero codes.  Every token carries its own scale, so
 *     nothing is re-encoded.
 *   The four arrays must be 16-byte aligned (else SDVA_ERR_INVALID).
 *   verify_attn reads INT4, INT8 and FP8-row caches through fp16 (see
 *   there): a dequantised value above 65504 in magnitude is out of range.
 *   page_table: int32 [num_lanes][max_pages_per_lane]; entry p of lane b is
 *     the physical page holding the lane's tokens [64p, 64p + 64).
 *   seq_lens: int32 [num_lanes], L_b = tokens already cached for lane b
 *     before the step (the same pre-step array is passed to all three calls;
 *     spec_accept's commit is the last thing to change it).
 */
#ifndef SDVA_H
#define SDVA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL selects the legacy default stream. */
typedef struct CUstream_st* sdva_stream_t;

typedef enum {
    SDVA_KV_FP8_E4M3 = 0, /* one fp32 scale per (page, kv head) */
    SDVA_KV_INT4_G32 = 1, /* one fp16 scale per (token, kv head, 32 dims) */
    SDVA_KV_INT8_G64 = 2, /* one fp16 scale per (token, kv head, 64 dims) */
    SDVA_KV_FP8_ROW = 3   /* one fp32 scale per (token, kv head) */
} sdva_kv_dtype;

/* Description of a caller-owned cache; all four arrays are device memory
 * laid out as above. */
typedef struct {
    int32_t dtype;        /* sdva_kv_dtype */
    int32_t num_pages;    /* physical pages in the pool */
    int32_t page_size;    /* must be 64 */
    int32_t num_kv_heads; /* >= 1 */
    int32_t head_dim;     /* must be 128 */
    void* k_codes;
    void* v_codes;
    void* k_scales;
    void* v_scales;
} sdva_kv_cache;

/* Host return codes. */
#define SDVA_OK 0
#define SDVA_ERR_INVALID (-1)     /* null pointer, non-positive size, Hq % Hkv != 0, ... */
#define SDVA_ERR_UNSUPPORTED (-2) /* head_dim != 128, page_size != 64, window > 16, dtype */
#define SDVA_ERR_WORKSPACE (-3)   /* workspace missing or smaller than required */
#define SDVA_ERR_CUDA (-4)        /* a kernel launch failed (cudaGetLastError) */

/* Device status bits, OR-ed into *status. */
#define SDVA_STATUS_BAD_PAGE 1  /* a needed page_table entry is outside [0, num_pages) */
#define SDVA_STATUS_OVERFLOW 2  /* L_b < 0, or L_b + n does not fit the lane's row / max_context */
#define SDVA_STATUS_BAD_DRAFT 4 /* a draft id is outside [0, vocab) */
#define SDVA_STATUS_TIMEOUT 8   /* a bounded device wait gave up */
#define SDVA_STATUS_BAD_COUNT 16 /* a per-lane draft or token count is out of range */
#define SDVA_STATUS_BAD_TREE 32 /* a draft tree's parent is not an earlier slot */

/*
 * kv_append_quant -- write tokens [L_b, L_b + n_new) of every lane into the
 * cache (in/out), quantising as described above.
 *   k_new, v_new : bf16 [num_lanes][n_new][num_kv_heads][128]
 *   n_new        : >= 1; the verify window (1 + d) in a speculative step, or
 *                  any chunk length when filling a context.
 *   page_table, max_pages_per_lane, seq_lens: as above (seq_lens is read only).
 *   status       : nullable device int.
 * A lane with L_b < 0 or L_b + n_new > 64 * max_pages_per_lane gets
 * SDVA_STATUS_OVERFLOW; a lane whose touched pages include an invalid id gets
 * SDVA_STATUS_BAD_PAGE; in both cases nothing of that lane is written.
 * Precondition: inputs are finite; no two lanes map the same physical page
 * within one call; appends to a lane arrive in position order.
 * Returns SDVA_OK or a negative SDVA_ERR_*.
 */
int kv_append_quant(const sdva_kv_cache* cache, const void* k_new, const void* v_new, int num_lanes, int n_new,
                    const int32_t* page_table, int max_pages_per_lane, const int32_t* seq_lens, int32_t* status,
                    sdva_stream_t stream);

/*
 * kv_append_quant_ragged -- kv_append_quant with a token count per lane, for a
 * padded window whose lanes drafted different numbers of tokens (the draft
 * count is chosen per workload: NInfer review, section "아키텍처 ③").
 *   n_lane: int32 [num_lanes] (device, required): lane b writes only its
 *           first n_lane[b] tokens, positions [L_b, L_b + n_lane[b]); the
 *           rest of its n_new input rows are not read.  The result is what
 *           appending each lane's truncated window on its own writes, so
 *           padding never touches the cache or an FP8 page scale.
 * A lane with n_lane[b] == 0 is not examined.  A count outside [0, n_new]
 * sets SDVA_STATUS_BAD_COUNT and skips the lane; the other rules, layouts
 * and return codes are those of kv_append_quant (the range and page checks
 * apply to [L_b, L_b + n_lane[b])).
 */
int kv_append_quant_ragged(const sdva_kv_cache* cache, const void* k_new, const void* v_new, int num_lanes,
                           int n_new, const int32_t* n_lane, const int32_t* page_table, int max_pages_per_lane,
                           const int32_t* seq_lens, int32_t* status, sdva_stream_t stream);

/*
 * verify_attn_workspace_size -- bytes of device scratch verify_attn needs for
 * these sizes (split-K partial results).  Pure host function.  num_sms = 0
 * queries the current device; pass the same arguments to verify_attn.
 * Returns 0 for arguments verify_attn would reject.
 */
size_t verify_attn_workspace_size(int num_lanes, int window, int num_q_heads, int num_kv_heads, int max_context,
                                  int num_sms);

/*
 * verify_attn -- for lane b, window position i in [0, window) and q head h:
 *     out[b][i][h] = softmax_j(sm_scale * q . K_j) . V_j  over j in [0, L_b + i]
 * with K_j, V_j the dequantised cache rows of kv head h / (Hq / Hkv): the
 * cached context followed by the window's own tokens, which must already
 * have been appended (causal inside the window).
 *   q   : bf16 [num_lanes][window][num_q_heads][128]   (|q| < 65504)
 *   out : bf16 [num_lanes][window][num_q_heads][128]   (written in full)
 *   q and out must be 16-byte aligned (else SDVA_ERR_INVALID).
 *   window: 1 .. 16.   max_context: host upper bound on every L_b.
 *   workspace: device scratch of at least verify_attn_workspace_size(...) bytes,
 *     256-byte aligned, used only during the call's kernels (its contents
 *     between calls do not matter; calls that share a workspace must not
 *     overlap on the GPU).
 * A lane with L_b < 0, L_b > max_context or L_b + window > 64 *
 * max_pages_per_lane gets SDVA_STATUS_OVERFLOW; a lane with an invalid page id
 * among its first ceil((L_b + window) / 64) entries gets SDVA_STATUS_BAD_PAGE;
 * the output rows of such a lane are set to zero.
 * Formats: FP8 keys enter the tensor core as stored codes; INT4 and INT8 K
 * and V are widened to fp16 (code * scale, one rounding); FP8-row V is
 * widened to fp16 as code * (s_j / s_max), s_max the largest V row scale of
 * the page's written rows, so a row whose scale is below 2^-14 s_max keeps
 * fewer significant bits (fp16 subnormals).  INT8 and FP8-row are served by
 * the tensor-core kernels only, which need at most 128 rows per kv head
 * (window * Hq / Hkv <= 128), at most 1024 lanes, num_pages * num_kv_heads *
 * 64 < 2^31 and num_lanes * (max_pages_per_lane + 16) * num_kv_heads < 2^31
 * (else SDVA_ERR_UNSUPPORTED; FP8 and INT4 calls outside these limits run on
 * the mma.sync kernels, causal window only).
 * Returns SDVA_OK or a negative SDVA_ERR_*.
 */
int verify_attn(const sdva_kv_cache* cache, const void* q, int num_q_heads, int num_lanes, int window,
                const int32_t* page_table, int max_pages_per_lane, const int32_t* seq_lens, int max_context,
                float sm_scale, void* out, void* workspace, size_t workspace_bytes, int32_t* status,
                sdva_stream_t stream);

/*
 * verify_attn_tree -- verify_attn for a window that holds a tree of drafted
 * tokens instead of a chain (MegaCapybara announcement, item 1: drafts and
 * draft trees).  Reading taken: window slot 0 is the root (the last
 * committed token) and slot i >= 1 hangs under parent[b][i] < i; the window
 * is appended in slot order as usual (slot i at position L_b + i).  Row i
 * attends to the cached context [0, L_b) and to the window keys of its
 * ancestors and of itself:
 *     out[b][i][h] = softmax_j(sm_scale * q . K_j) . V_j
 *                    over j in [0, L_b) and j = L_b + k, k in anc(i) + {i}.
 * A chain (parent[b][i] = i - 1) gives exactly verify_attn's result.
 *   parent: int32 [num_lanes][window] (device; entry 0 is not read); may be
 *           NULL only when window == 1.
 *   Every other argument, layout and return code is that of verify_attn.
 * A lane with a parent outside [0, i) gets SDVA_STATUS_BAD_TREE and its
 * output rows are set to zero (other lanes are unaffected).  Supported up to
 * 128 rows per kv head (window * num_q_heads / num_kv_heads); larger returns
 * SDVA_ERR_UNSUPPORTED.
 */
int verify_attn_tree(const sdva_kv_cache* cache, const void* q, int num_q_heads, int num_lanes, int window,
                     const int32_t* parent, const int32_t* page_table, int max_pages_per_lane,
                     const int32_t* seq_lens, int max_context, float sm_scale, void* out, void* workspace,
                     size_t workspace_bytes, int32_t* status, sdva_stream_t stream);

/*
 * verify_attn_ragged -- verify_attn for a padded window whose lanes drafted
 * different numbers of tokens (the draft count is chosen per workload:
 * NInfer review, section "아키텍처 ③"), the attention counterpart of
 * kv_append_quant_ragged.
 *   n_lane: int32 [num_lanes] (device, required): lane b's window is its
 *           first n_lane[b] = 1 + d_b rows.  Rows i < n_lane[b] equal
 *           verify_attn's (they see keys 0 .. L_b + i, all written by the
 *           ragged append); rows i >= n_lane[b] are written as zeros.
 * A count outside [0, window] sets SDVA_STATUS_BAD_COUNT and zeroes the
 * lane's rows.  Every other argument, layout and return code is that of
 * verify_attn.  Supported up to 128 rows per kv head (window * num_q_heads /
 * num_kv_heads); larger returns SDVA_ERR_UNSUPPORTED.  The tensor-core tile
 * holds every window row of a kv head, so the rows past a lane's count cost
 * no key bytes but still occupy the tile.
 */
int verify_attn_ragged(const sdva_kv_cache* cache, const void* q, int num_q_heads, int num_lanes, int window,
                       const int32_t* n_lane, const int32_t* page_table, int max_pages_per_lane,
                       const int32_t* seq_lens, int max_context, float sm_scale, void* out, void* workspace,
                       size_t workspace_bytes, int32_t* status, sdva_stream_t stream);

/* Bytes of the fixed device scratch behind verify_attn_noalloc (32 MiB). */
#define SDVA_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

/*
 * verify_attn_noalloc -- verify_attn without a workspace argument, for callers
 * that cannot allocate device memory at call time: runtimes that plan all of
 * their device memory once at start-up and keep no headroom for per-call
 * scratch, plugin hosts that give an operator only its own input and output
 * tensors, and latency-critical loops that cannot pay for an allocator's
 * implicit device synchronisation.  (The pages describe no such call; it is
 * an addition of this library.)
 *   Arguments, outputs, status bits and return codes are those of verify_attn.
 *   The split-K scratch is a fixed, 256-byte-aligned array of
 *   SDVA_NOALLOC_SCRATCH_BYTES compiled into this library's device image; every
 *   GPU that loads the library holds it until the process exits.  The call
 *   itself allocates nothing (no cudaMalloc / cudaFree).
 *   Sizes whose verify_attn_workspace_size(...) exceeds
 *   SDVA_NOALLOC_SCRATCH_BYTES are rejected with SDVA_ERR_WORKSPACE before
 *   anything is enqueued.
 *   Every call looks up the array's device address for the device current at
 *   that call (a host-side query that allocates nothing); the first call on a
 *   device may also load the library's device code there, so make it before
 *   any stream capture.
 *   All calls share the one array and it keeps the last call's contents
 *   (nothing in it needs to start at zero): calls whose kernels overlap on the
 *   GPU -- on different streams, or from different threads -- race on it and
 *   must be serialised by the caller.
 */
int verify_attn_noalloc(const sdva_kv_cache* cache, const void* q, int num_q_heads, int num_lanes, int window,
                        const int32_t* page_table, int max_pages_per_lane, const int32_t* seq_lens,
                        int max_context, float sm_scale, void* out, int32_t* status, sdva_stream_t stream);

/*
 * verify_step -- one whole verify step: kv_append_quant (the window's K/V,
 * n_new = window), verify_attn and spec_accept, on one stream, with results
 * identical to those three calls made in that order (Baseten talk summary,
 * section "추측 디코드": the main model checks the drafts in one pass).  The
 * kernels are chained as programmatic dependent launches, so that each one's
 * prologue runs while its predecessor drains: the attention's set-up under
 * the append, the acceptance's argmax beside the attention's merge.
 *   Arguments: as in the three calls.  k_new, v_new: the window's K/V, bf16
 *   [num_lanes][window][num_kv_heads][128]; q, out, workspace, max_context,
 *   sm_scale: as verify_attn; logits, vocab, drafts, accept_len, out_tokens:
 *   as spec_accept; seq_lens: the pre-step L_b, and with commit != 0 it is
 *   advanced by 1 + accept_len at the end of the step (in/out).
 * Preconditions, status bits and return codes are those of the three calls;
 * the arguments of all three are checked before anything is enqueued (a
 * call that returns an error enqueues nothing, except that an error from a
 * CUDA launch may leave earlier kernels of the step enqueued).
 */
int verify_step(const sdva_kv_cache* cache, const void* k_new, const void* v_new, const void* q, int num_q_heads,
                int num_lanes, int window, const int32_t* page_table, int max_pages_per_lane, int32_t* seq_lens,
                int max_context, float sm_scale, void* out, void* workspace, size_t workspace_bytes,
                const float* logits, int vocab, const int32_t* drafts, int32_t* accept_len, int32_t* out_tokens,
                int commit, int32_t* status, sdva_stream_t stream);

/*
 * spec_accept -- greedy acceptance of a verify window.
 *   logits    : fp32 [num_lanes][window][vocab]; row i scores the token that
 *               follows window position i.
 *   drafts    : int32 [num_lanes][window - 1]; drafts[b][i] is window token
 *               i + 1 (nullable when window == 1).
 *   out_tokens: int32 [num_lanes][window] (out): argmax of each row, ties to
 *               the lowest index, NaN never wins, an all-NaN row gives 0.
 *   accept_len: int32 [num_lanes] (out): a = number of leading i < window - 1
 *               with drafts[b][i] == out_tokens[b][i].  The bonus token is
 *               out_tokens[b][a].
 *   seq_lens_inout: nullable int32 [num_lanes] (in/out): when given, the
 *               commit adds 1 + a to each lane's length.
 * window: 1 .. 16 (SDVA_ERR_UNSUPPORTED above), num_lanes <= 65535.
 * An out-of-vocabulary draft id never matches and sets SDVA_STATUS_BAD_DRAFT.
 * Returns SDVA_OK or a negative SDVA_ERR_*.
 */
int spec_accept(const float* logits, int num_lanes, int window, int vocab, const int32_t* drafts,
                int32_t* accept_len, int32_t* out_tokens, int32_t* seq_lens_inout, int32_t* status,
                sdva_stream_t stream);

/*
 * spec_accept_lazy -- greedy acceptance that reads a lane's logits rows only
 * up to its first disagreement, with a draft count per lane.
 *   The accepted prefix ends at the first draft that disagrees with the
 *   target argmax (Baseten talk summary, section "추측 디코드"), so the rows
 *   after it decide nothing; the draft count is chosen per workload (NInfer
 *   review, section "아키텍처 ③"), and a batch may mix lanes that drafted
 *   different numbers of tokens into one padded window.
 *   logits, drafts, seq_lens_inout: as for spec_accept (drafts keeps the
 *               row stride window - 1; entries past a lane's count are not
 *               read).
 *   num_drafts: nullable int32 [num_lanes]: d_b, the lane's draft count,
 *               0 <= d_b <= window - 1; NULL means window - 1 for every lane.
 *               Rows past d_b are never read.
 *   accept_len: int32 [num_lanes] (out): a = number of leading i < d_b with
 *               drafts[b][i] == argmax of row i.
 *   out_tokens: int32 [num_lanes][window] (out): the argmax of rows 0 .. a
 *               (same tie rules as spec_accept; the bonus token is
 *               out_tokens[b][a]) and -1 in every later position.
 * With SDVA_LAZY_WALK_MIN_LANES (48) lanes or more a lane reads rows 0 .. a
 * from memory (one CTA
 * cluster walks them in order) and may prefetch row a + 1 into L2; with fewer
 * lanes, where that serial walk is slower than one pass over the GPU, rows
 * 0 .. d_b of every lane are reduced at once.  Both give the same results.
 * A lane whose count is outside
 * [0, window - 1] sets SDVA_STATUS_BAD_COUNT and gets accept_len 0,
 * out_tokens all -1 and no commit.  An out-of-vocabulary id among a lane's
 * first d_b drafts sets SDVA_STATUS_BAD_DRAFT and never matches.
 * Limits and return codes as for spec_accept.
 */
#define SDVA_LAZY_WALK_MIN_LANES 48 /* spec_accept_lazy walks rows from this many lanes on */

int spec_accept_lazy(const float* logits, int num_lanes, int window, int vocab, const int32_t* drafts,
                     const int32_t* num_drafts, int32_t* accept_len, int32_t* out_tokens, int32_t* seq_lens_inout,
                     int32_t* status, sdva_stream_t stream);

/*
 * spec_accept_tree -- greedy acceptance of a draft tree.
 *   The pages verify chains of drafts (Baseten talk summary, section
 *   "추측 디코드"); a tree of candidates is this library's reading of the
 *   same check: window slot 0 is the root (the last committed token) and
 *   slot i >= 1 hangs under parent[b][i] < i.  From the root, the walk moves
 *   to the first child (in slot order) whose token is the argmax of the
 *   current node's logits row, and stops when no child agrees.
 *   logits    : fp32 [num_lanes][window][vocab]; row i scores the token that
 *               follows slot i.
 *   tokens    : int32 [num_lanes][window]: the window's tokens (slot 0 is
 *               not read); parent: int32 [num_lanes][window] (slot 0 not
 *               read).  Both nullable when window == 1.
 *   accept_len: int32 [num_lanes] (out): a, the nodes accepted after the root.
 *   path      : int32 [num_lanes][window] (out): the accepted slots, root
 *               (0) first, -1 after; also used as scratch by the call.
 *   out_tokens: int32 [num_lanes][window] (out): the accepted tokens, then
 *               the bonus token (argmax of the last node's row), -1 after.
 *   seq_lens_inout: nullable: adds 1 + a.
 * Argmax ties go to the lowest index, NaN never wins (as spec_accept).  A
 * lane with a parent outside [0, i) sets SDVA_STATUS_BAD_TREE and gets a = 0,
 * path and out_tokens all -1, no commit.  A token outside [0, vocab) sets
 * SDVA_STATUS_BAD_DRAFT and never matches.  Limits as spec_accept.
 */
int spec_accept_tree(const float* logits, int num_lanes, int window, int vocab, const int32_t* tokens,
                     const int32_t* parent, int32_t* accept_len, int32_t* path, int32_t* out_tokens,
                     int32_t* seq_lens_inout, int32_t* status, sdva_stream_t stream);

/*
 * spec_accept_sampled -- lossless stochastic acceptance of a verify window
 * (sampling at temperature 1 that keeps the target model's distribution).
 *   DFlash2 keeps the draft model's conditional distribution q (NInfer
 *   review, section "아키텍처 ③"); with it, the verifier accepts draft i when
 *   u_i * q_i(x_i) < p_i(x_i), p_i = softmax(logits row i); at the first
 *   rejection a it draws one token from max(0, p_a - q_a) normalised, and
 *   from p_d when all d = window - 1 drafts are accepted.  The draw is the
 *   inverse CDF in index order at u_sample * Z (Z = the weights' sum): the
 *   smallest k whose running sum exceeds it, else the last index of positive
 *   weight; a residual of zero mass falls back to p_a.
 *   logits     : fp32 [num_lanes][window][vocab], finite.
 *   draft_probs: fp32 [num_lanes][window - 1][vocab]: row i is q_i, the
 *                distribution drafts[b][i] was drawn from (non-negative;
 *                need not be renormalised).  Nullable when window == 1.
 *   drafts     : int32 [num_lanes][window - 1] (nullable when window == 1).
 *   u_accept   : fp32 [num_lanes][window - 1] uniforms in [0, 1).
 *   u_sample   : fp32 [num_lanes] uniforms in [0, 1).
 *   accept_len : int32 [num_lanes] (out): a.
 *   out_tokens : int32 [num_lanes][window] (out): drafts[b][0 .. a), the
 *                drawn token at position a, -1 after.
 *   seq_lens_inout: nullable int32 [num_lanes] (in/out): adds 1 + a.
 *   workspace  : device memory of spec_accept_sampled_workspace_size()
 *                bytes, 8-byte aligned (per-row softmax statistics,
 *                per-slice sums of the drawn rows and per-lane counters;
 *                no initialisation needed, not shared by calls in flight
 *                at the same time).
 * Arithmetic is fp32 (hardware exp2): a decision within fp32 rounding of its
 * boundary may differ from an exact evaluation.  An out-of-vocabulary draft
 * is a rejection and sets SDVA_STATUS_BAD_DRAFT.  window 1 .. 16,
 * num_lanes * window <= 65535.  Returns SDVA_OK, SDVA_ERR_INVALID,
 * SDVA_ERR_UNSUPPORTED, SDVA_ERR_WORKSPACE or SDVA_ERR_CUDA.
 */
size_t spec_accept_sampled_workspace_size(int num_lanes, int window);
int spec_accept_sampled(const float* logits, const float* draft_probs, int num_lanes, int window, int vocab,
                        const int32_t* drafts, const float* u_accept, const float* u_sample, int32_t* accept_len,
                        int32_t* out_tokens, int32_t* seq_lens_inout, void* workspace, size_t workspace_bytes,
                        int32_t* status, sdva_stream_t stream);

/*
 * sdva_debug_set_wait_limit -- diagnostic hook (no counterpart in the pages).
 * Every device-side wait of verify_attn's tensor-core kernels gives up after
 * `cycles` clock cycles (default about 4e9, two seconds); the CTA then
 * raises SDVA_STATUS_TIMEOUT, waits (with its own bound) for the copies and
 * tensor-core work it issued, frees its tensor memory and returns, leaving
 * the context usable (the output of such a call is undefined).  A negative
 * value restores the default.  Returns the previous limit.  Applies to
 * calls enqueued after it returns; not synchronised with concurrent calls.
 * Meant for tests that make a wait run out.
 */
long long sdva_debug_set_wait_limit(long long cycles);

/* Static description of a return code or status bit set (never NULL). */
const char* sdva_status_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* SDVA_H */
