/*
 * inkling_rel_attn.h -- C ABI of libinkling_rel_attn.so
 *
 * Paged-KV, RoPE-free grouped-query attention with a learned additive
 * relative-position bias, for one attention layer per call, on an sm_103a GPU.
 *
 * What is computed (Support Inkling-NVFP4 model, TensorRT-LLM PR #17062,
 * "Architecture" and "Implementation"; Fail fast on Inkling's unsupported GPU
 * architectures, vLLM PR #51560, "Purpose"): for a query token t at absolute
 * position p of sequence b and query head h, with h_kv = h / (H_q / H_kv),
 *
 *   K_j = k_cache[page_table[b * page_table_stride + j / page_size],
 *                 j % page_size, h_kv, :]            (V_j likewise)
 *   key j is visible iff j <= p and (window <= 0 or p - j < window)
 *   s_j = scale * <q[t, h, :], K_j> + rel_logits[t, h, min(p - j, R - 1)]
 *   out[t, h, :] = sum over visible j of softmax(s)_j * V_j
 *   lse[t, h]    = log(sum over visible j of exp(s_j))          (natural log)
 *
 * A query with no visible key (a sequence of length 0) gets out = 0 and
 * lse = -inf.  The local layers of the model use window 512 with 16 KV heads,
 * the global layers a full causal mask (window <= 0) with 8 KV heads; the
 * bias table rel_logits has a static shape [tokens, H_q, R] (TensorRT-LLM
 * PR #17062, "Implementation": that is what makes decode graph-capturable).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensor arguments are DEVICE pointers to dense row-major arrays owned
 *   by the caller.  The library never allocates, frees, synchronises or reads
 *   device data on the host, so every call can be captured in a CUDA graph
 *   once its workspace exists; device-side metadata (page_table, seq_lens,
 *   cu_seqlens_q) may change between graph replays.
 * - Element types: q, k_cache, v_cache, out are bf16 (raw 16-bit words);
 *   rel_logits and lse_out are fp32; page_table, seq_lens, cu_seqlens_q int32.
 * - Alignment: q, k_cache, v_cache, out and workspace must be 16-byte aligned;
 *   every other pointer 4-byte aligned.
 * - Supported shapes: D in {64, 128}; H_q % H_kv == 0 and H_q / H_kv <= 16;
 *   page_size a multiple of 16, at most 256; R >= 1 (prefill: R % 4 == 0).
 * - Return value: 0 on success, a negative INKLING_* code otherwise (see
 *   inkling_rel_attn_error_string).  Validation looks at host scalars and
 *   pointer values only.  Nothing is launched when a call fails validation.
 * - device_error (optional, may be NULL): a device int32 word into which
 *   kernels OR an INKLING_DEVERR_* bit when they meet bad device data (a page
 *   id outside [0, num_pages), a sequence longer than its page-table row) or a
 *   pipeline wait that timed out.  Kernels never trap; bad page ids read zeros.
 *   The caller clears the word and reads it back when it chooses.
 * - stream: the CUDA stream (cudaStream_t) everything is enqueued on.
 */
#ifndef INKLING_REL_ATTN_H
#define INKLING_REL_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define INKLING_OK 0
#define INKLING_ERR_ARG (-1)        /* bad scalar, NULL required pointer, unsupported shape */
#define INKLING_ERR_ALIGN (-2)      /* a pointer violates the alignment rule above */
#define INKLING_ERR_WORKSPACE (-3)  /* workspace missing or smaller than required */
#define INKLING_ERR_DEVICE (-4)     /* current device is not an sm_103 GPU */
#define INKLING_ERR_CUDA (-5)       /* a CUDA runtime/driver call or launch failed */

#define INKLING_DEVERR_BAD_PAGE 1    /* page id out of range (read as zeros) */
#define INKLING_DEVERR_SEQ_TOO_LONG 2 /* seq_len > page_table_stride*page_size (clamped) */
#define INKLING_DEVERR_TIMEOUT 4     /* a pipeline wait gave up; outputs are invalid */
#define INKLING_DEVERR_BAD_CHUNK 8   /* prefill: q_len > seq_len or q_len > max_q_len */
#define INKLING_DEVERR_BAD_SLOT 16   /* kv_conv_append: state pool row out of range */

/*
 * inkling_rel_attn_decode -- one query token per sequence.
 *
 * Definition: the formula above with t = b and p = seq_lens[b] - 1 (the
 * current token's K/V are already in the cache; TensorRT-LLM PR #17062 commit
 * notes on skip_kv_write: the attention step writes K/V before it reads them).
 * Split-KV with a log-sum-exp merge (vLLM PR #51560, "Changes":
 * inkling_fa4_num_splits; gist "serving Inkling-NVFP4 on 8x H200": split-KV
 * path with num_splits=32): each sequence's visible keys are cut into up to
 * num_splits contiguous ranges, each range is reduced to a normalised partial
 * output and its lse, and a second kernel merges them.
 *
 *   q           bf16 [B, H_q, D]
 *   k_cache     bf16 [num_pages, page_size, H_kv, D]
 *   v_cache     bf16 [num_pages, page_size, H_kv, D]
 *   page_table  int32 [B, page_table_stride]; row b lists sequence b's
 *               physical pages in logical order
 *   seq_lens    int32 [B]; keys of sequence b incl. the current token (0 ok)
 *   rel_logits  fp32 [B, H_q, R]
 *   window      > 0: sliding window of that many keys; <= 0: full causal
 *   scale       multiplies <q, k> before the bias is added
 *   max_seq_len host-side upper bound on seq_lens (sizes the split plan;
 *               a longer sequence is still computed correctly)
 *   out         bf16 [B, H_q, D], fully overwritten (never read)
 *   lse_out     fp32 [B, H_q] natural-log lse, or NULL
 *   workspace   device scratch of at least
 *               inkling_rel_attn_decode_workspace_size(...) bytes when the
 *               chosen split count is > 1; may be NULL when it is 1
 *   num_splits  0 = automatic (inkling_rel_attn_choose_splits with the
 *               device's SM count), > 0 = forced (clamped to [1, 128] and to
 *               one split per 64 keys)
 */
int inkling_rel_attn_decode(
    const void* q, const void* k_cache, const void* v_cache,
    const int32_t* page_table, int32_t page_table_stride,
    const int32_t* seq_lens, const float* rel_logits,
    int32_t B, int32_t H_q, int32_t H_kv, int32_t D, int32_t page_size,
    int32_t num_pages, int32_t R, int32_t window, float scale,
    int32_t max_seq_len, void* out, float* lse_out, void* workspace,
    size_t workspace_bytes, int32_t num_splits, int32_t* device_error,
    void* stream);

/*
 * inkling_rel_attn_decode_noalloc -- inkling_rel_attn_decode without a
 * caller-provided workspace, for callers that cannot allocate device memory
 * (for example a plugin inside a host framework that owns all device memory
 * and forbids allocation during a step, or a binding with no access to the
 * CUDA allocator).  The pages describe no such entry point; it has no
 * counterpart there.
 *
 * Same arguments and result as inkling_rel_attn_decode minus workspace /
 * workspace_bytes.  Split partials live in a fixed 32 MiB device array inside
 * the library (one per GPU that loads it, held until process exit).  A call
 * needing more scratch than that (see
 * inkling_rel_attn_decode_workspace_size) returns INKLING_ERR_WORKSPACE and
 * launches nothing.  Nothing is allocated.  All calls on a device share the
 * array: calls whose kernels may overlap on the GPU race and must be ordered
 * by the caller.  The first call on each device resolves the array's device
 * address (cudaGetSymbolAddress) with that device current; make it outside any
 * stream capture.
 */
int inkling_rel_attn_decode_noalloc(
    const void* q, const void* k_cache, const void* v_cache,
    const int32_t* page_table, int32_t page_table_stride,
    const int32_t* seq_lens, const float* rel_logits,
    int32_t B, int32_t H_q, int32_t H_kv, int32_t D, int32_t page_size,
    int32_t num_pages, int32_t R, int32_t window, float scale,
    int32_t max_seq_len, void* out, float* lse_out, int32_t num_splits,
    int32_t* device_error, void* stream);

/*
 * inkling_rel_attn_decode_multi -- decode of q_len >= 1 new tokens per
 * sequence (multi-token prediction / speculative verification: the model's
 * draft layers share the attention, TensorRT-LLM PR #17062, "Architecture").
 *
 * Sequence b's q_len query tokens are its LAST q_len tokens (their K/V already
 * in the cache): token i sits at position p = seq_lens[b] - q_len + i and sees
 * keys j <= p (and p - j < window when window > 0), with the bias
 * rel_logits[b * q_len + i, h, min(p - j, R - 1)].  The result equals
 * inkling_rel_attn_prefill with q_len tokens per sequence; the K/V of a
 * (sequence, KV head) is read once per group of tokens (groups of
 * min(q_len, 16 / G) tokens, G = H_q / H_kv), not once per token.
 *
 *   q          bf16 [B * q_len, H_q, D] (token-major: row b * q_len + i)
 *   rel_logits fp32 [B * q_len, H_q, R]
 *   out        bf16 [B * q_len, H_q, D]; lse_out fp32 [B * q_len, H_q] or NULL
 *   q_len      1 .. 64 (1 is inkling_rel_attn_decode); seq_lens[b] >= q_len
 *   workspace  inkling_rel_attn_decode_multi_workspace_size bytes when the
 *              call splits the keys, else may be NULL
 * Other arguments, ownership, errors and graph safety as for decode.  A
 * sequence shorter than q_len sets INKLING_DEVERR_BAD_CHUNK and gets out = 0,
 * lse = -inf.
 */
int inkling_rel_attn_decode_multi(
    const void* q, const void* k_cache, const void* v_cache,
    const int32_t* page_table, int32_t page_table_stride,
    const int32_t* seq_lens, const float* rel_logits, int32_t B, int32_t q_len,
    int32_t H_q, int32_t H_kv, int32_t D, int32_t page_size, int32_t num_pages,
    int32_t R, int32_t window, float scale, int32_t max_seq_len, void* out,
    float* lse_out, void* workspace, size_t workspace_bytes,
    int32_t num_splits, int32_t* device_error, void* stream);

/* Workspace bytes of inkling_rel_attn_decode_multi for these scalars (0 when
 * the call does not split the keys).  Host only; num_sms as for
 * inkling_rel_attn_decode_workspace_size. */
size_t inkling_rel_attn_decode_multi_workspace_size(int32_t B, int32_t q_len,
                                                    int32_t H_q, int32_t H_kv,
                                                    int32_t D, int32_t window,
                                                    int32_t max_seq_len,
                                                    int32_t num_splits,
                                                    int32_t num_sms);

/*
 * inkling_rel_attn_prefill -- chunked / paged prefill (TensorRT-LLM PR #17062,
 * "Implementation": paged prefill over the cache).
 *
 * Sequence b owns the packed query tokens cu_seqlens_q[b] ..
 * cu_seqlens_q[b+1]-1.  They are the LAST q_len_b = cu_seqlens_q[b+1] -
 * cu_seqlens_q[b] tokens of a sequence whose seq_lens[b] keys (cached prefix
 * plus this chunk) are all in the cache, so query i sits at position
 * p = seq_lens[b] - q_len_b + i.
 *
 *   q            bf16 [T, H_q, D]
 *   cu_seqlens_q int32 [B + 1], non-decreasing, cu_seqlens_q[0] = 0,
 *                cu_seqlens_q[B] = T, every q_len_b <= max_q_len
 *   seq_lens     int32 [B], q_len_b <= seq_lens[b]
 *   rel_logits   fp32 [T, H_q, R]
 *   max_q_len    host-side bound on q_len_b (sizes the grid)
 *   out          bf16 [T, H_q, D]; lse_out fp32 [T, H_q] or NULL
 *   workspace    unused by this version (pass NULL / 0)
 * Other arguments as for decode.
 */
int inkling_rel_attn_prefill(
    const void* q, const int32_t* cu_seqlens_q, const void* k_cache,
    const void* v_cache, const int32_t* page_table, int32_t page_table_stride,
    const int32_t* seq_lens, const float* rel_logits, int32_t B, int32_t T,
    int32_t max_q_len, int32_t H_q, int32_t H_kv, int32_t D, int32_t page_size,
    int32_t num_pages, int32_t R, int32_t window, float scale,
    int32_t max_seq_len, void* out, float* lse_out, void* workspace,
    size_t workspace_bytes, int32_t* device_error, void* stream);

/*
 * inkling_rel_attn_kv_append -- write the new tokens' K and V rows into the
 * paged cache, the step right before decode / prefill reads it (TensorRT-LLM
 * PR #17062, commit notes: the attention op writes the step's K/V into the
 * cache itself before reading it -- `skip_kv_write` for the backend).
 *
 * Token numbering is the prefill's: sequence b owns the packed tokens
 * cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1, the LAST q_len_b of its seq_lens[b]
 * tokens, so token i sits at position p = seq_lens[b] - q_len_b + i (decode:
 * cu_seqlens_q = 0, 1, .., B and p = seq_lens[b] - 1).  Its K row (all H_kv
 * heads, H_kv * D bf16, contiguous) is copied to
 * k_cache[page_table[b * page_table_stride + p / page_size]][p % page_size],
 * and likewise its V row.  No other byte of the cache is written.
 *
 *   k_new, v_new  bf16 [T, H_kv, D] (device), 16-byte aligned
 *   k_cache, v_cache bf16 [num_pages, page_size, H_kv, D] (device), written
 *   cu_seqlens_q  int32 [B + 1] (device), non-decreasing, [0] = 0, [B] = T
 *   seq_lens      int32 [B] (device), total tokens incl. the appended ones
 *   page_table    int32 [B, page_table_stride] (device)
 * The caller owns every buffer; nothing is allocated or synchronised, and the
 * call can be captured in a CUDA graph.  Returns INKLING_OK or a negative
 * INKLING_ERR_* code (arguments are checked on the host before anything
 * launches: D in {64, 128}, page_size a multiple of 16 up to 256, positive
 * pool / stride, 16-byte alignment).  On the device a token whose chunk is
 * inconsistent (q_len_b > seq_lens[b]) sets INKLING_DEVERR_BAD_CHUNK, one past
 * its page-table row INKLING_DEVERR_SEQ_TOO_LONG, one whose page id is outside
 * [0, num_pages) INKLING_DEVERR_BAD_PAGE; such tokens are not written.
 */
int inkling_rel_attn_kv_append(
    const void* k_new, const void* v_new, const int32_t* cu_seqlens_q,
    const int32_t* seq_lens, const int32_t* page_table,
    int32_t page_table_stride, int32_t B, int32_t T, int32_t H_kv, int32_t D,
    int32_t page_size, int32_t num_pages, void* k_cache, void* v_cache,
    int32_t* device_error, void* stream);

/*
 * inkling_rel_attn_kv_conv_append -- the causal short convolutions on K and V
 * of the new tokens, then the KV append of the convolved rows (TensorRT-LLM
 * PR #17062, "Architecture": two causal short convolutions inside attention,
 * on K and on V, carrying per-request state across decode steps;
 * "pyexecutor" row: the state lives in a pool with one row per request).
 *
 * The pages give no width, layout, bias or activation; this is the plainest
 * form: depthwise over the C = H_kv * D channels of a token's row, causal
 * along the tokens, no bias, no activation.  For channel c of token i of
 * sequence b (tokens numbered as in inkling_rel_attn_kv_append):
 *
 *   y_i[c] = sum_{j=0}^{width-1} w[c * width + j] * x_{i-(width-1)+j}[c]
 *
 * (tap width-1 multiplies the current token) where the inputs before the
 * sequence's new tokens are the rows of its state, state[state_slots[b]]: its
 * last width-1 inputs, oldest first (zeros for a new request).  y (rounded to
 * bf16, fp32 accumulation) goes to the cache slot of the token's position, as
 * inkling_rel_attn_kv_append places rows; afterwards the state row holds the
 * sequence's last width-1 inputs (raw, not convolved).  K and V have their own
 * taps and states.
 *
 *   k_new, v_new      bf16 [T, H_kv, D] (device), 16-byte aligned
 *   conv_w_k, conv_w_v fp32 [H_kv, D, width] (device)
 *   width             1 .. 8 (1: no state; the state pointers may be NULL)
 *   conv_state_k, conv_state_v bf16 [num_slots, width - 1, H_kv, D] (device),
 *                     16-byte aligned, read and rewritten in place
 *   state_slots       int32 [B] (device): the pool row of each sequence; rows
 *                     must be distinct within a call
 *   cu_seqlens_q, seq_lens, page_table, k_cache, v_cache: as for
 *                     inkling_rel_attn_kv_append
 *   max_q_len         host bound on the new tokens of one sequence (the grid
 *                     covers max_q_len tokens per sequence)
 * The caller owns every buffer; nothing is allocated or synchronised, and the
 * call can be captured in a CUDA graph.  Returns INKLING_OK or a negative
 * INKLING_ERR_* code after host checks (width, D in {64, 128}, page_size,
 * positive pool / stride / num_slots, alignment, B * ceil(max_q_len / 32) <=
 * 65535).  On the device: an
 * inconsistent chunk (q_len_b > seq_lens[b]) sets INKLING_DEVERR_BAD_CHUNK and
 * the sequence is skipped; q_len_b > max_q_len sets it too and the tokens past
 * max_q_len are not written (the state row still moves to the end of the
 * chunk); a state row outside [0, num_slots) sets
 * INKLING_DEVERR_BAD_SLOT and the sequence is skipped; positions past the
 * page-table row and bad page ids set INKLING_DEVERR_SEQ_TOO_LONG /
 * INKLING_DEVERR_BAD_PAGE and those rows are not written.
 */
int inkling_rel_attn_kv_conv_append(
    const void* k_new, const void* v_new, const int32_t* cu_seqlens_q,
    const int32_t* seq_lens, const int32_t* page_table,
    int32_t page_table_stride, const float* conv_w_k, const float* conv_w_v,
    int32_t width, void* conv_state_k, void* conv_state_v,
    const int32_t* state_slots, int32_t num_slots, int32_t B, int32_t T,
    int32_t max_q_len, int32_t H_kv, int32_t D, int32_t page_size,
    int32_t num_pages, void* k_cache, void* v_cache, int32_t* device_error,
    void* stream);

/*
 * inkling_rel_attn_choose_splits -- the decode split count, a pure host
 * function of host scalars (so it is identical at graph capture and replay,
 * and independent of physical page ids).  vLLM PR #51560, "Changes": the
 * split count is computed per call and capped at 128.
 *
 * keys per query = min(window, max_seq_len) (or max_seq_len when window <= 0);
 * the count aims at >= 3 CTAs per SM over B * H_kv (sequence, KV head) pairs,
 * keeps every split >= 256 keys, caps a split at 1024 keys, and is <= 128.
 * num_sms <= 0 means 152 (a GB300).  Returns >= 1.
 */
int32_t inkling_rel_attn_choose_splits(int32_t B, int32_t H_kv, int32_t window,
                                       int32_t max_seq_len, int32_t num_sms);

/*
 * inkling_rel_attn_decode_workspace_size -- bytes of workspace decode needs
 * for these scalars: fp32 partial outputs [B, H_q, S, D] plus fp32 partial
 * lse [B, H_q, S], S = the split count the call will use (num_splits as for
 * decode; 0 = automatic with num_sms SMs, num_sms <= 0 = the current device's
 * SM count, or 152 if no device is visible).  0 when S == 1.  Host only.
 */
size_t inkling_rel_attn_decode_workspace_size(int32_t B, int32_t H_q,
                                              int32_t H_kv, int32_t D,
                                              int32_t window,
                                              int32_t max_seq_len,
                                              int32_t num_splits,
                                              int32_t num_sms);

/* Workspace bytes prefill needs (0 in this version).  Host only. */
size_t inkling_rel_attn_prefill_workspace_size(int32_t T, int32_t H_q,
                                               int32_t D);

/*
 * inkling_rel_attn_selftest_timeout -- failure-path self-test.  Launches one
 * tiny kernel whose bounded pipeline wait (the routine every kernel of the
 * library uses for its mbarrier waits) can never succeed: it gives up after
 * timeout_ms milliseconds (1..10000), ORs INKLING_DEVERR_TIMEOUT into
 * *device_error and returns, without trapping; the CUDA context stays usable.
 * No counterpart on the pages (they describe fail-fast capability checks, vLLM
 * #51560 "Changes", not device waits).
 */
int inkling_rel_attn_selftest_timeout(int32_t* device_error, int32_t timeout_ms, void* stream);

/* Static, human-readable text for an INKLING_* return code. */
const char* inkling_rel_attn_error_string(int32_t code);

/* Library version as major*10000 + minor*100 + patch. */
int32_t inkling_rel_attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* INKLING_REL_ATTN_H */
