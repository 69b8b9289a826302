/*
 * pkvqk — paged KV-cache decode attention for GB300 (sm_103a): C ABI.
 *
 * The decode step of an attention layer over a paged KV cache, in three
 * calls that follow the problem statement of InfiniLM PR #585 ("perf: Qwen3
 * offline inference — hybrid attention backend, fused rms_norm_rope, chunked
 * prefill + prompt-lookup spec decoding"), section "概述 / Summary":
 *
 *   1. pkvqk_norm_rope_append — item 2: fused per-head RMSNorm + full-rotary
 *      (neox rotate-half) RoPE on q and k; k and v then go into the paged
 *      BSHD cache (item 1) through a slot mapping.
 *   2. pkvqk_paged_decode     — item 1: split-KV paged decode attention with
 *      GQA read straight from the strided BSHD cache; with q_len > 1 it is
 *      the causal multi-query verify of item 4 (k + 1 tokens per sequence).
 *   3. pkvqk_lse_combine      — item 1 ("splitkv"): log-sum-exp merge of the
 *      split partials.
 *   4. pkvqk_paged_prefill    — item 4 (chunked prefill): the same causal
 *      attention for many new tokens per sequence (a prefill chunk after
 *      its prior context), on the tensor cores; pkvqk_paged_prefill_varlen
 *      takes a different number of new tokens per sequence (item 1's
 *      varlen prefill).
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every buffer is owned by the caller; the library allocates no device
 *   memory and keeps no state beyond a per-thread error message, facts it
 *   caches per device (the SM count; each kernel's shared-memory limit, set
 *   once), the rotary sin/cos knot table it builds once on the host, and the
 *   fixed scratch of pkvqk_paged_decode_static_ws (below).
 * - Pointers marked "device" must be device (or managed) memory of the
 *   current device; they are checked with cudaPointerGetAttributes and a
 *   host pointer is rejected with PKVQK_ERR_POINTER_RESIDENCY.
 * - bf16 means IEEE bfloat16 (raw 16-bit storage).  Strides are in elements.
 * - Work is enqueued on `stream`; no call synchronises, reads device memory
 *   on the host, or allocates, so every call can be recorded into a CUDA
 *   graph.  Argument errors are detected on the host before any launch and
 *   leave all buffers untouched.
 * - `status_flags` (optional, may be NULL) is a device int32 into which the
 *   kernels OR the PKVQK_FLAG_* bits below when they meet bad data (an
 *   out-of-range block id or slot) or a pipeline wait that timed out.  The
 *   caller zeroes it and reads it back when convenient.
 * - On failure the call returns a non-zero pkvqk_status and
 *   pkvqk_last_error() describes it.
 */
#ifndef PKVQK_H
#define PKVQK_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKVQK_API __attribute__((visibility("default")))
#else
#define PKVQK_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same handle as cudaStream_t / CUstream; NULL is the legacy default stream. */
typedef struct CUstream_st* pkvqk_stream_t;

typedef enum pkvqk_status {
  PKVQK_OK = 0,
  PKVQK_ERR_INVALID_ARG = 1,          /* null pointer, bad size, misaligned   */
  PKVQK_ERR_UNSUPPORTED = 2,          /* valid but not implemented (e.g. D)   */
  PKVQK_ERR_WORKSPACE_TOO_SMALL = 3,
  PKVQK_ERR_POINTER_RESIDENCY = 4,    /* host pointer where device expected   */
  PKVQK_ERR_CUDA = 5                  /* a CUDA runtime/driver call failed    */
} pkvqk_status;

/* Bits OR-ed into *status_flags by the kernels. */
#define PKVQK_FLAG_BAD_SLOT      0x1  /* slot >= num_blocks*block_size: skipped */
#define PKVQK_FLAG_BAD_BLOCK_ID  0x2  /* block id outside [0, num_blocks): its keys read as zeros */
#define PKVQK_FLAG_WAIT_TIMEOUT  0x4  /* a pipeline wait gave up: output invalid */

/*
 * Layout of a paged cache, shared by the K and the V cache of a layer:
 * element (block, slot, head, d) lives at
 *     base + block*block_stride + slot*slot_stride + head*head_stride + d.
 * The default BSHD layout [num_blocks, block_size, num_kv_heads, head_dim]
 * has block_stride = block_size*num_kv_heads*head_dim,
 * slot_stride = num_kv_heads*head_dim, head_stride = head_dim; any strides
 * that are multiples of 8 elements (16 bytes) are accepted, so K and V may be
 * two views into one interleaved or stacked allocation (no copy is made).
 * block_size must be a multiple of 16 (16..256); head_dim must be 128.
 */
typedef struct pkvqk_cache_layout {
  int64_t num_blocks;
  int32_t block_size;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t reserved;                  /* set to 0 */
  int64_t block_stride;
  int64_t slot_stride;
  int64_t head_stride;
} pkvqk_cache_layout;

/* Message of the last failing call made on this thread ("" if none). */
PKVQK_API const char* pkvqk_last_error(void);

/* ABI version of this header: 1. */
PKVQK_API int32_t pkvqk_abi_version(void);

/*
 * Fused per-head RMSNorm + neox RoPE on q and k, then the k/v append.
 * Source: InfiniLM PR #585, "概述 / Summary" item 2 ("rms_norm_rope"), item 1
 * (BSHD paged cache).
 *
 * For each token t < num_tokens and head h, with x the head's D values:
 *   y = x / sqrt(mean(x^2) + eps) * gamma          (gamma_q for q, gamma_k for k)
 *   for i < D/2, a = positions[t] * theta^(-2i/D):
 *     y'[i]       = y[i] cos a - y[i + D/2] sin a
 *     y'[i + D/2] = y[i + D/2] cos a + y[i] sin a
 * rounded once to bf16 (round-to-nearest-even).  q is overwritten in place.
 * With s = slot_mapping[t] in [0, num_blocks*block_size), the rotated k and
 * the unchanged v of every kv head go to block s / block_size, slot
 * s % block_size of k_cache / v_cache.  s < 0 (padding) writes nothing; a
 * too-large s writes nothing and sets PKVQK_FLAG_BAD_SLOT.
 *
 *   q             device bf16, element (t, h, d) at q[t*q_stride_t + h*q_stride_h + d]
 *   k, v          device bf16, same form with their own strides, Hkv heads
 *   positions     device int64 [num_tokens]
 *   slot_mapping  device int64 [num_tokens]
 *   gamma_q/_k    device bf16 [head_dim]
 *   k_cache, v_cache  device bf16, layout as described by `layout`
 * Two tokens mapped to the same slot race (caller error).  Strides and base
 * pointers must be 16-byte aligned.
 */
PKVQK_API pkvqk_status pkvqk_norm_rope_append(
    void* q, int64_t q_stride_t, int64_t q_stride_h,
    const void* k, int64_t k_stride_t, int64_t k_stride_h,
    const void* v, int64_t v_stride_t, int64_t v_stride_h,
    const int64_t* positions, const int64_t* slot_mapping,
    const void* gamma_q, const void* gamma_k,
    float theta, float eps,
    int32_t num_tokens, int32_t num_q_heads,
    void* k_cache, void* v_cache, const pkvqk_cache_layout* layout,
    int32_t* status_flags, pkvqk_stream_t stream);

/*
 * Bytes of a rotary table for positions 0 .. max_positions-1: 1 KiB per
 * position.  0 when max_positions is outside 1 .. 2^21.
 */
PKVQK_API size_t pkvqk_rope_table_bytes(int32_t max_positions);

/*
 * Fills `table` with the rotary sin/cos that pkvqk_norm_rope_append computes
 * for a token at each position p < max_positions (same source, item 2): for
 * i < D/2 the angle p * theta^(-2i/D), reduced and evaluated exactly as that
 * call does, kept as float-float pairs.  Build once per model (theta and the
 * longest context), before the steps that read it; the table depends on
 * nothing else.
 *
 *   table          device, 16-byte aligned, pkvqk_rope_table_bytes(max_positions)
 *                  bytes, owned by the caller; written by a kernel on `stream`
 *   max_positions  0 .. 2^21 (0: nothing to do)
 * Errors: PKVQK_ERR_INVALID_ARG (max_positions out of range, theta not > 0,
 * table not a 16-byte aligned device pointer).
 */
PKVQK_API pkvqk_status pkvqk_rope_table_build(void* table, int32_t max_positions, float theta,
                                              pkvqk_stream_t stream);

/*
 * pkvqk_norm_rope_append with the angles of tokens at positions
 * 0 .. table_positions-1 read from a table built by pkvqk_rope_table_build
 * (with the same theta) instead of computed per token.  Tokens at other
 * positions compute theirs as pkvqk_norm_rope_append does.  The results are
 * bit-identical to pkvqk_norm_rope_append's.  Every other argument and error
 * as there; table_positions 0 .. 2^21 (0: no table is read).
 */
PKVQK_API pkvqk_status pkvqk_norm_rope_append_cached(
    void* q, int64_t q_stride_t, int64_t q_stride_h,
    const void* k, int64_t k_stride_t, int64_t k_stride_h,
    const void* v, int64_t v_stride_t, int64_t v_stride_h,
    const int64_t* positions, const int64_t* slot_mapping,
    const void* gamma_q, const void* gamma_k,
    float theta, float eps,
    int32_t num_tokens, int32_t num_q_heads,
    void* k_cache, void* v_cache, const pkvqk_cache_layout* layout,
    const void* rope_table, int32_t table_positions,
    int32_t* status_flags, pkvqk_stream_t stream);

/*
 * Schedule for pkvqk_paged_decode from host-side facts only (no device
 * read): batch, kv heads, rows per kv head (q_len * Hq/Hkv), the longest
 * sequence, the total key count and the SM count (0 = query the current
 * device).  Returns 0 (the balanced schedule: chosen for large batches whose
 * total keys are under half of batch x longest) or a split count in
 * [1, 256]; above 16 rows per kv head
 * (run on the tensor-core kernel, see pkvqk_paged_decode) it returns
 * pkvqk_choose_prefill_splits(batch, num_kv_heads, rows_per_kv_head, 1, ...).
 * Source: the "decode routing hint (host side, zero device sync)" of
 * InfiniLM PR #585, Summary item 3.
 */
PKVQK_API int32_t pkvqk_choose_num_splits(int32_t batch, int32_t num_kv_heads,
                                int32_t rows_per_kv_head, int32_t max_seq_len,
                                int64_t total_tokens, int32_t block_size,
                                int32_t sm_count);

/*
 * Workspace bytes pkvqk_paged_decode needs on the current device:
 * - num_splits == 1: 0;
 * - num_splits >= 2: batch*q_len*Hq*num_splits*(head_dim + 1)*4, rounded up
 *   to 256.  Layout: fp32 partial outputs [rows][num_splits][head_dim], then
 *   fp32 partial lse [rows][num_splits] (rows = (b*q_len + t)*Hq + h);
 * - num_splits == 0 (balanced): an upper bound for any kv-head count,
 *   ((SMs + batch)*q_len*Hq*(head_dim + 1)*4 + batch*Hq*8) rounded up, where
 *   SMs is the current device's multiprocessor count (internal layout).
 * Nothing in the workspace needs to start at zero, and calls of any shape and
 * schedule may share one (in stream order).
 */
PKVQK_API size_t pkvqk_decode_workspace_bytes(int32_t batch, int32_t q_len,
                                    int32_t num_q_heads, int32_t head_dim,
                                    int32_t num_splits);

/*
 * Split-KV paged decode attention with GQA; causal multi-query verify when
 * q_len > 1.  Source: InfiniLM PR #585, "概述 / Summary" items 1 and 4.
 *
 * For sequence b, query token t < q_len and q head h (kv head h / (Hq/Hkv)):
 *   visible keys  n < seq_lens[b] - q_len + t + 1, key n at block
 *                 block_tables[b*max_blocks_per_seq + n / block_size],
 *                 slot n % block_size
 *   s_n = scale * <q, K_n>   (scale <= 0 selects head_dim^-1/2)
 *   out = sum_n softmax(s)_n V_n,  lse = log sum_n exp(s_n)
 * A row with no visible key outputs 0 and lse = -inf.
 *
 * Schedules (the result does not depend on them, up to rounding):
 * - num_splits >= 1 (split-KV): with C = ceil(ceil(max_seq_len_hint /
 *   block_size) / num_splits) pages, split j < S-1 of a sequence covers pages
 *   [j*C, (j+1)*C) and split S-1 covers [(S-1)*C, end), so every key is
 *   covered whatever the hint.  Each split keeps an online softmax; for
 *   num_splits > 1 the partials go to the workspace and a log-sum-exp
 *   combine kernel that this call launches (as a programmatic dependent, so
 *   its launch overlaps the decode kernel's tail) merges them.
 *   pkvqk_choose_num_splits gives a host-side choice.
 * - num_splits == 0 (balanced): a persistent grid of 0.84 CTAs per SM; the
 *   pages of all (sequence, kv-head group) pairs are laid end to end and
 *   every CTA takes an equal contiguous share, crossing sequence boundaries;
 *   a sequence covered by one CTA is written directly, one cut across CTAs is
 *   merged by a combine kernel this call launches.  Balances any mix of
 *   lengths.
 *
 *   q             device bf16, element (b*q_len + t, h, d) at
 *                 q[(b*q_len + t)*q_stride_t + h*q_stride_h + d]
 *   block_tables  device int32 [batch, max_blocks_per_seq]
 *   seq_lens      device int32 [batch], counting the q_len new tokens
 *   num_splits    0 (balanced schedule) or 1..256 (split schedule)
 *   max_seq_len_hint  host int >= the longest seq_len (0 = max_blocks_per_seq*block_size)
 *   out           device bf16 [batch, q_len, Hq, head_dim], contiguous
 *   lse_out       device fp32 [batch, q_len, Hq] or NULL
 *   workspace     device, >= pkvqk_decode_workspace_bytes(batch, q_len, Hq,
 *                 head_dim, num_splits) on the current device (NULL if 0)
 * Supported: head_dim 128, Hq % Hkv == 0, q_len <= 16.  Up to 16 rows per
 * kv head (q_len*Hq/Hkv) run on the decode kernel; more (e.g. q_len 5 at
 * 8 q heads per kv head) run on the tensor-core multi-query kernel of
 * pkvqk_paged_prefill with the same split boundaries and partial layout,
 * and num_splits == 0 there becomes a split count whose partials fit the
 * balanced workspace bound.
 */
PKVQK_API pkvqk_status pkvqk_paged_decode(
    const void* q, int64_t q_stride_t, int64_t q_stride_h,
    const void* k_cache, const void* v_cache, const pkvqk_cache_layout* layout,
    const int32_t* block_tables, int32_t max_blocks_per_seq,
    const int32_t* seq_lens,
    int32_t batch, int32_t q_len, int32_t num_q_heads,
    int32_t num_splits, int32_t max_seq_len_hint, float scale,
    void* out, float* lse_out,
    void* workspace, size_t workspace_bytes,
    int32_t* status_flags, pkvqk_stream_t stream);

/*
 * As pkvqk_paged_decode but stops after the split pass: the partials stay in
 * the workspace (layout above) and are not merged (pkvqk_lse_combine merges
 * them).  num_splits must be >= 2 (no heuristic).
 */
PKVQK_API pkvqk_status pkvqk_paged_decode_partials(
    const void* q, int64_t q_stride_t, int64_t q_stride_h,
    const void* k_cache, const void* v_cache, const pkvqk_cache_layout* layout,
    const int32_t* block_tables, int32_t max_blocks_per_seq,
    const int32_t* seq_lens,
    int32_t batch, int32_t q_len, int32_t num_q_heads,
    int32_t num_splits, int32_t max_seq_len_hint, float scale,
    void* workspace, size_t workspace_bytes,
    int32_t* status_flags, pkvqk_stream_t stream);

/*
 * pkvqk_paged_decode without a caller workspace.  The pages describe no such
 * call: it has no counterpart there and exists for callers that cannot
 * allocate device memory — e.g. a plugin that a host engine hands only input
 * and output pointers, or code running while an allocator refuses to
 * allocate — and so cannot pass the split workspace.
 *
 * Same arguments and results as pkvqk_paged_decode minus workspace and
 * workspace_bytes, except that num_splits == 0 here picks the split count
 * with pkvqk_choose_num_splits (the split schedule) instead of the balanced
 * schedule.  The split partials go to a fixed 16 MiB array inside the
 * library (pkvqk_static_workspace_capacity()), held on every GPU that loads
 * the library until the process exits.  A call whose partials need more
 * (pkvqk_decode_workspace_bytes for its split count) returns
 * PKVQK_ERR_WORKSPACE_TOO_SMALL and launches nothing; so does a
 * num_splits == 0 call whose chosen split count needs more.  Arguments that
 * pkvqk_paged_decode rejects are rejected the same way here.  The call
 * allocates nothing.  The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress, with that device current) and caches it for
 * the CUDA context current at that time; a later call under another context
 * of the device (a driver context made current by the caller, or the primary
 * context re-created after cudaDeviceReset) looks it up again.  Make the
 * first call in each context before any stream capture.  All calls on a
 * device share the one array and it keeps the last call's partials: calls
 * that can overlap on the GPU (different streams, no ordering between them)
 * race and corrupt each other's results.  Nothing in it needs to start at
 * zero.
 */
PKVQK_API pkvqk_status pkvqk_paged_decode_static_ws(
    const void* q, int64_t q_stride_t, int64_t q_stride_h,
    const void* k_cache, const void* v_cache, const pkvqk_cache_layout* layout,
    const int32_t* block_tables, int32_t max_blocks_per_seq,
    const int32_t* seq_lens,
    int32_t batch, int32_t q_len, int32_t num_q_heads,
    int32_t num_splits, int32_t max_seq_len_hint, float scale,
    void* out, float* lse_out,
    int32_t* status_flags, pkvqk_stream_t stream);

/* Bytes of the array pkvqk_paged_decode_static_ws uses (16 MiB). */
PKVQK_API size_t pkvqk_static_workspace_capacity(void);

/*
 * Log-sum-exp merge of split partials.  Source: InfiniLM PR #585, Summary
 * item 1 ("splitkv").  For each row r < rows:
 *   M = max_j lse[r][j];  w_j = exp(lse[r][j] - M)
 *   out[r] = sum_j w_j o[r][j] / sum_j w_j,  lse_out[r] = M + log sum_j w_j
 * Splits with lse = -inf weigh 0; a row whose splits are all empty outputs
 * 0 and -inf.
 *   ws_o    device fp32 [rows][num_splits][head_dim]
 *   ws_lse  device fp32 [rows][num_splits]
 *   out     device bf16 [rows][head_dim];  lse_out device fp32 [rows] or NULL
 * head_dim must be 128.
 */
PKVQK_API pkvqk_status pkvqk_lse_combine(const float* ws_o, const float* ws_lse,
                               int32_t rows, int32_t head_dim,
                               int32_t num_splits, void* out, float* lse_out,
                               pkvqk_stream_t stream);

/*
 * Split count for pkvqk_paged_prefill from host-side facts only: batch, kv
 * heads, q_len, group (Hq/Hkv), the longest sequence (keys, counting the new
 * tokens) and the SM count (0 = the current device's).  Returns 1..256: 1
 * when the row tiles alone fill the GPU, else enough splits of >= 256 keys
 * to give about one CTA per SM.
 */
PKVQK_API int32_t pkvqk_choose_prefill_splits(int32_t batch, int32_t num_kv_heads,
                                    int32_t q_len, int32_t group,
                                    int32_t max_seq_len, int32_t sm_count);

/*
 * Workspace bytes of pkvqk_paged_prefill: 0 for num_splits == 1, else
 * batch*q_len*Hq*num_splits*(head_dim + 1)*4 rounded up to 256: fp32 partial
 * outputs [rows][num_splits][head_dim] then fp32 partial lse
 * [rows][num_splits], rows = (b*q_len + t)*Hq + h (the layout
 * pkvqk_lse_combine reads).  Nothing in it needs to start at zero.
 */
PKVQK_API size_t pkvqk_prefill_workspace_bytes(int32_t batch, int32_t q_len,
                                     int32_t num_q_heads, int32_t head_dim,
                                     int32_t num_splits);

/*
 * Causal multi-query paged attention on the tensor cores: a chunked-prefill
 * step (q_len new tokens per sequence, appended to the cache beforehand,
 * attend to their prior context and causally to each other) or, with small
 * q_len, a speculative-verify step.  Source: InfiniLM PR #585, "概述 /
 * Summary" item 4 (chunked prefill; fixed b x (k+1) verify shape) and item 1
 * (paged cache read through the block table).
 *
 * Same definition as pkvqk_paged_decode: query token t of sequence b sees the
 * keys n < seq_lens[b] - q_len + t + 1; q head h reads kv head h / (Hq/Hkv);
 * scale <= 0 selects head_dim^-1/2; a row with no visible key outputs 0 and
 * lse = -inf.  The rows (t, h) of one kv head are packed t*group + h%group
 * into tiles of 128, so one CTA's tile covers 128/group tokens.
 *
 * num_splits >= 1: split j covers pages [j*C, (j+1)*C) of every sequence,
 * C = ceil(ceil(max_seq_len_hint / block_size) / num_splits), the last split
 * also everything past (S-1)*C pages.  With num_splits > 1 the normalised
 * partials go to the workspace and this call then launches the log-sum-exp
 * combine (pkvqk_lse_combine) on the same stream.
 *
 *   q, out, lse_out, block_tables, seq_lens: as pkvqk_paged_decode
 *   num_splits    1..256 (pkvqk_choose_prefill_splits gives a choice)
 *   max_seq_len_hint  host int >= the longest seq_len (0 = max_blocks_per_seq*block_size)
 *   workspace     device, >= pkvqk_prefill_workspace_bytes(...) (NULL if 0)
 * Supported: head_dim 128, Hq % Hkv == 0, 1 <= q_len <= 16384,
 * q_len*Hq/Hkv <= 65536.  One CTA per SM (197 KiB of shared memory and 512
 * tensor-memory columns each).
 */
PKVQK_API pkvqk_status pkvqk_paged_prefill(
    const void* q, int64_t q_stride_t, int64_t q_stride_h,
    const void* k_cache, const void* v_cache, const pkvqk_cache_layout* layout,
    const int32_t* block_tables, int32_t max_blocks_per_seq,
    const int32_t* seq_lens,
    int32_t batch, int32_t q_len, int32_t num_q_heads,
    int32_t num_splits, int32_t max_seq_len_hint, float scale,
    void* out, float* lse_out,
    void* workspace, size_t workspace_bytes,
    int32_t* status_flags, pkvqk_stream_t stream);

/*
 * Varlen form of pkvqk_paged_prefill: every sequence brings its own number of
 * new tokens, packed back to back (the FlashAttention-2 varlen convention the
 * pages use for prefill, Summary item 1).  Source: InfiniLM PR #585, "概述 /
 * Summary" items 1 (varlen prefill, paged cache) and 4 (chunked prefill).
 *
 * Sequence b's q_len_b = cu_seqlens_q[b+1] - cu_seqlens_q[b] new tokens are
 * rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 of q, out and lse_out; token t
 * of it sees the keys n < seq_lens[b] - q_len_b + t + 1 (seq_lens counting the
 * new tokens).  A fresh prompt has seq_lens[b] == q_len_b; a later chunk of a
 * prompt, or a verify step, has more keys than new tokens.
 *
 *   q              device bf16, row i at q[i*q_stride_t + h*q_stride_h + d]
 *   cu_seqlens_q   device int32 [batch + 1], non-decreasing, cu_seqlens_q[0] = 0
 *   max_q_len      host int >= every q_len_b (1..16384): sizes the grid (no
 *                  device read); tokens past it are not computed
 *   total_q        host: rows of q / out / lse_out (= cu_seqlens_q[batch]);
 *                  rows at or past it are never written
 *   out            device bf16 [total_q, Hq, head_dim], contiguous
 *   lse_out        device fp32 [total_q, Hq] or NULL
 *   workspace      num_splits > 1: >= pkvqk_prefill_workspace_bytes(1, total_q,
 *                  Hq, head_dim, num_splits)
 * Everything else as pkvqk_paged_prefill.
 */
PKVQK_API pkvqk_status pkvqk_paged_prefill_varlen(
    const void* q, int64_t q_stride_t, int64_t q_stride_h,
    const int32_t* cu_seqlens_q, int32_t max_q_len, int64_t total_q,
    const void* k_cache, const void* v_cache, const pkvqk_cache_layout* layout,
    const int32_t* block_tables, int32_t max_blocks_per_seq,
    const int32_t* seq_lens,
    int32_t batch, int32_t num_q_heads,
    int32_t num_splits, int32_t max_seq_len_hint, float scale,
    void* out, float* lse_out,
    void* workspace, size_t workspace_bytes,
    int32_t* status_flags, pkvqk_stream_t stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif /* PKVQK_H */
