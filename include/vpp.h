/*
 * vpp.h -- C ABI of the GB300 (sm_103a) chunked-prefill causal-attention library.
 *
 * The operation is one chunked-prefill step of causal self-attention: a chunk
 * of C query tokens whose first token sits at absolute position P (the prefix
 * length) attends to every cached key/value at positions 0 .. P + i
 * (inclusive) for its i-th token.  Citations name the pages by title:
 *
 *   [VPP review]   "VPP: Virtual Pipeline Parallelism for Efficient Chunked
 *                  Prefill in Long-Context LLM Inference" (English technical
 *                  review): §2.1 (prefill fills the KV cache, decode reads
 *                  it), §2.2 Eq. (1) (softmax(Q K^T / sqrt(d)) V, token i
 *                  attends to tokens <= i), §2.3 (chunked prefill: a later
 *                  chunk attends to the whole cached prefix plus itself).
 *   [GLM PP note]  "02 · 并行策略与 PP 切分" (deployment note): §1 (paged KV
 *                  pool, block_size = 64), §7 (context-parallel attention
 *                  needs the backend to return the LSE of each partial).
 *   [FastPP summary] "Revisiting Pipeline Parallelism for LLM Serving":
 *                  section "预备知识：分块与三种气泡" (a micro-batch mixes
 *                  prefill chunks with one-token decode requests).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Memory.   Every tensor argument is caller-owned DEVICE memory unless the
 *           argument says HOST.  The library allocates no device memory in
 *           any call; scratch space is the caller's `workspace`.
 * Streams.  `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *           default stream).  Calls enqueue work and return without
 *           synchronising.  A launch failure returns VPP_ERR_CUDA.
 * Layouts.  Row-major, contiguous, 16-byte aligned base pointers.
 *             q, out        [T][heads][d]          (token-major)
 *             lse           [heads][T] float32, natural log of the softmax
 *                           denominator, ln sum_j exp(s_j)
 *             paged cache   k_cache [num_blocks][64][kv_heads][head_dim_qk]
 *                           v_cache [num_blocks][64][kv_heads][head_dim_v]
 *                           token j of a sequence lives in block
 *                           block_table[j / 64], row j % 64
 *             contiguous    k_cache [capacity][kv_heads][head_dim_qk]
 *                           (block_table == NULL); v_cache likewise
 *           bf16 means IEEE bfloat16 stored as uint16.
 * Heads.    GQA: query head h reads kv head h / (heads / kv_heads).
 *           heads == kv_heads is plain multi-head attention.
 * Scale.    softmax_scale <= 0 selects 1 / sqrt(head_dim_qk) ([VPP review]
 *           Eq. (1), d read as the per-head query/key dimension).
 * Supported head_dim_qk in {64, 128, 192}, head_dim_v in {64, 128},
 *           heads / kv_heads in {1, 2, 4, 8, 16}; anything else returns
 *           VPP_ERR_UNSUPPORTED.
 * Errors.   Arguments are validated on the host before any launch; nothing
 *           is enqueued when a call returns an error.  Kernels never trap: a
 *           wait that times out on the device records VPP_ERR_TIMEOUT in a
 *           device status word that vpp_last_device_status() reads.
 */
#ifndef VPP_H
#define VPP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    VPP_OK = 0,
    VPP_ERR_INVALID = -1,     /* bad pointer, size, alignment or range       */
    VPP_ERR_UNSUPPORTED = -2, /* valid but unsupported head dims / grouping  */
    VPP_ERR_CUDA = -3,        /* a CUDA runtime call failed                  */
    VPP_ERR_TIMEOUT = -4,     /* a device-side wait ran out (status word)    */
    VPP_ERR_WORKSPACE = -5    /* workspace missing or smaller than required  */
} vpp_status;

typedef enum {
    VPP_BF16 = 0,
    VPP_FP32 = 1
} vpp_dtype;

/* Human-readable name of a status code (static string, never NULL). */
const char *vpp_status_string(int status);

/* Library version as 10000*major + 100*minor + patch. */
int vpp_version(void);

/*
 * a1 -- KV append ([VPP review] §2.1: prefill fills the cache that later
 * chunks and decode read; [GLM PP note] §1: 64-token blocks).
 *
 * Copies the chunk's new keys k_new [chunk_len][kv_heads][head_dim_qk] and
 * values v_new [chunk_len][kv_heads][head_dim_v] into cache positions
 * prefix_len .. prefix_len + chunk_len - 1.  in_dtype is the type of
 * k_new/v_new: VPP_BF16 is a bit copy; VPP_FP32 is rounded to bf16
 * (round-to-nearest-even) on the way in.  The cache is always bf16.
 * block_table (device int32, >= ceil((prefix_len+chunk_len)/64) entries, each
 * in [0, num_blocks)) selects the paged layout; NULL selects the contiguous
 * layout, where num_blocks is instead the capacity in tokens.
 * Block-table entries are not read on the host; out-of-range entries are
 * skipped on the device and recorded as VPP_ERR_INVALID in the status word.
 * chunk_len == 0 is a no-op returning VPP_OK (pointers may then be NULL).
 */
int vpp_kv_append(const void *k_new, const void *v_new, int in_dtype,
                  void *k_cache, void *v_cache, const int32_t *block_table,
                  int32_t num_blocks, int64_t prefix_len, int64_t chunk_len,
                  int kv_heads, int head_dim_qk, int head_dim_v, void *stream);

/*
 * a2..a6 -- chunk attention, the plain form: contiguous bf16 cache
 * [prefix_len + chunk_len][kv_heads][head_dim], head_dim_qk = head_dim_v =
 * head_dim, default scale, no key splitting (no workspace).
 *
 * q [chunk_len][heads][head_dim] bf16 -> out [chunk_len][heads][head_dim]
 * bf16 and lse [heads][chunk_len] float32 (lse may be NULL).  Query i
 * attends keys 0 .. prefix_len + i of the cache ([VPP review] §2.2 Eq. (1),
 * §2.3).  The chunk's own K/V must already be in the cache (vpp_kv_append
 * first).  chunk_len == 0 is a no-op (pointers may then be NULL).
 */
int vpp_chunk_attn(const void *q, const void *k_cache, const void *v_cache,
                   int64_t prefix_len, int64_t chunk_len, int heads,
                   int kv_heads, int head_dim, void *out, float *lse,
                   void *stream);

/*
 * a2..a7 -- chunk attention, full form.
 *
 * q_dtype: VPP_BF16, or VPP_FP32 (q is then rounded to bf16 into the
 * workspace before the attention kernel reads it).  Cache as described in
 * the conventions (paged if block_table != NULL, num_blocks = blocks in the
 * pool; contiguous otherwise, num_blocks = capacity in tokens, which must be
 * >= prefix_len + chunk_len).
 * num_splits: 0 lets the library choose; 1 forbids splitting; S > 1 asks
 * for S key ranges over the prefix of every query token (clamped so every
 * range is non-empty).  The library's own choice may split only the query
 * tokens from some split token on (the heaviest query tiles, launched first),
 * leaving the earlier ones unsplit; vpp_chunk_attn_plan reports it.  With more
 * than one range, each range writes a float32 partial (output, lse) into the
 * workspace and a merge kernel combines the split tokens' partials
 * ([GLM PP note] §7):  L = ln sum_s exp(lse_s),  out = sum_s exp(lse_s - L) out_s.
 * workspace: device scratch of at least vpp_chunk_attn_workspace_size(...)
 * bytes for the same arguments (NULL allowed when that size is 0).
 * out [chunk_len][heads][head_dim_v] bf16, lse [heads][chunk_len] float32
 * (NULL allowed).
 */
int vpp_chunk_attn_ex(const void *q, int q_dtype, const void *k_cache,
                      const void *v_cache, const int32_t *block_table,
                      int32_t num_blocks, int64_t prefix_len,
                      int64_t chunk_len, int heads, int kv_heads,
                      int head_dim_qk, int head_dim_v, float softmax_scale,
                      int num_splits, void *out, float *lse, void *workspace,
                      size_t workspace_bytes, void *stream);

/*
 * Chunk attention without any allocation and without a caller workspace.
 * The pages have no counterpart to this entry point; it serves callers that
 * may not allocate device memory on their execution path and cannot hand
 * over scratch space (for example a plug-in whose host runtime owns all
 * device memory, or a binding that exposes only the plain signature).
 *
 * Same arguments and results as vpp_chunk_attn_ex with q_dtype = VPP_BF16 and
 * no workspace.  When the key range is split, the float32 partials live in a
 * fixed 32 MiB array in device memory that the library holds on every GPU
 * that loads it, until the process exits.  The partials take about
 * num_splits x chunk_len x heads x (head_dim_v + 1) x 4 bytes (exactly
 * vpp_chunk_attn_workspace_size for the same arguments).  With num_splits = 0
 * the library lowers its own choice of key ranges to the largest count whose
 * partials fit (one range needs none), so such a call always runs.  An
 * explicit num_splits > 1 whose partials exceed 32 MiB returns
 * VPP_ERR_WORKSPACE and launches nothing.  A device other than compute
 * capability 10.3 gives VPP_ERR_UNSUPPORTED.  The first call on a device looks up that array's device address (with the
 * device current); make that first call before any stream capture.  All calls
 * on a device share the array and it keeps the last call's contents (nothing
 * in it needs to start at zero), so calls that overlap on the GPU race: issue
 * them on one stream or synchronise between them.  Calls no allocating
 * routine.
 */
int vpp_chunk_attn_noalloc(const void *q, const void *k_cache,
                           const void *v_cache, const int32_t *block_table,
                           int32_t num_blocks, int64_t prefix_len,
                           int64_t chunk_len, int heads, int kv_heads,
                           int head_dim_qk, int head_dim_v,
                           float softmax_scale, int num_splits, void *out,
                           float *lse, void *stream);

/* Workspace bytes vpp_chunk_attn_ex needs for these arguments (0 if none). */
size_t vpp_chunk_attn_workspace_size(int q_dtype, int64_t prefix_len,
                                     int64_t chunk_len, int heads,
                                     int kv_heads, int head_dim_qk,
                                     int head_dim_v, int num_splits);

/*
 * The work plan vpp_chunk_attn_ex uses for these arguments: returns the
 * number of key ranges S (>= 1) or a negative status, and, if split_token is
 * not NULL, stores the first query token whose keys are split (0: every
 * token, or none when S = 1).  Tokens before it run unsplit.  Host-side; the
 * library's choice ([VPP review] §2.3: a chunk's cost grows with its prefix)
 * follows a list-scheduling model of the launch fitted on GB300 and is
 * remembered per shape.
 */
int vpp_chunk_attn_plan(int64_t prefix_len, int64_t chunk_len, int heads,
                        int kv_heads, int head_dim_qk, int head_dim_v,
                        int num_splits, int64_t *split_token);

/* The number of key ranges vpp_chunk_attn_ex will use for these arguments. */
int vpp_chunk_attn_num_splits(int64_t prefix_len, int64_t chunk_len,
                              int heads, int kv_heads, int head_dim_qk,
                              int head_dim_v, int num_splits);

/*
 * a8..a9 -- mixed micro-batch: prefill chunks and one-token decode rows over
 * one paged cache ([FastPP summary] "预备知识"; [VPP review] §2.1).
 *
 * q [total_q][heads][head_dim_qk] bf16, where sequence b owns rows
 * cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and its queries are its LAST
 * q_len_b = cu_seqlens_q[b+1] - cu_seqlens_q[b] positions: prefix
 * ctx_lens[b] - q_len_b.  ctx_lens[b] counts the sequence's own new tokens,
 * which must already be in the cache.  q_len_b == 1 is a decode row, served by
 * the split-KV decode kernel (1024-key ranges merged through their LSE) when
 * head_dim_qk == head_dim_v in {64, 128}, kv_heads <= 8 and heads/kv_heads is
 * 1, 2 or 4 (or 8 with head dim 64), and by the chunk-attention kernel
 * otherwise; q_len_b > 1 is a prefill chunk (chunk-attention kernel);
 * q_len_b == 0 is skipped.
 * cu_seqlens_q [batch+1] and ctx_lens [batch] are HOST int32 arrays (the
 * plan is built on the host and passed to the kernels by value; batch <=
 * 1024).  block_table is a device int32 [batch][max_blocks_per_seq].
 * out [total_q][heads][head_dim_v] bf16, lse [heads][total_q] float32 (NULL
 * allowed).  workspace >= vpp_mixed_attn_workspace_size(...) bytes.
 */
int vpp_mixed_attn(const void *q, const void *k_cache, const void *v_cache,
                   const int32_t *block_table, int32_t max_blocks_per_seq,
                   int32_t num_blocks, const int32_t *cu_seqlens_q,
                   const int32_t *ctx_lens, int32_t batch, int heads,
                   int kv_heads, int head_dim_qk, int head_dim_v,
                   float softmax_scale, void *out, float *lse,
                   void *workspace, size_t workspace_bytes, void *stream);

/* Workspace bytes vpp_mixed_attn needs (HOST cu_seqlens_q / ctx_lens). */
size_t vpp_mixed_attn_workspace_size(const int32_t *cu_seqlens_q,
                                     const int32_t *ctx_lens, int32_t batch,
                                     int heads, int kv_heads, int head_dim_qk,
                                     int head_dim_v);

/*
 * Varlen KV append for a mixed batch: the new K/V rows of every sequence,
 * packed like q in vpp_mixed_attn ([total_q][kv_heads][d]), go to the last
 * q_len_b positions of sequence b (HOST cu_seqlens_q / ctx_lens, device
 * block_table [batch][max_blocks_per_seq]).  bf16 in, bf16 cache.
 */
int vpp_kv_append_varlen(const void *k_new, const void *v_new, void *k_cache,
                         void *v_cache, const int32_t *block_table,
                         int32_t max_blocks_per_seq, int32_t num_blocks,
                         const int32_t *cu_seqlens_q, const int32_t *ctx_lens,
                         int32_t batch, int kv_heads, int head_dim_qk,
                         int head_dim_v, void *stream);

/*
 * fp8 KV cache ([GLM PP note] §1, §3.2: the deployment keeps its KV cache in
 * fp8, about half the bytes per token of bf16, which nearly doubles the
 * tokens one GPU holds).
 *
 * Element format: E4M3 of the OCP 8-bit floating point specification (1 sign
 * bit, 4 exponent bits with bias 7, 3 mantissa bits, largest finite value
 * 448, no infinities), one uint8 code per element, in the same layouts as the
 * bf16 cache (paged [num_blocks][64][kv_heads][d], or contiguous
 * [capacity][kv_heads][d] when block_table == NULL).
 * Scaling: k_scale and v_scale are DEVICE float32 [kv_heads], 4-byte aligned,
 * one factor per kv head, finite and > 0 (not checked on the device); an
 * element's value is E4M3(code) x scale.  The pages give only the byte
 * counts; the per-kv-head scaling is this library's reading.
 * NULL scales return VPP_ERR_INVALID.
 */

/*
 * a1 over an fp8 cache.  k_new/v_new are bf16 [chunk_len][kv_heads][d]; each
 * value x becomes code = E4M3(fl32(x / scale)): the float32 quotient (IEEE
 * round to nearest even) rounded to the nearest E4M3 value, ties to the even
 * code, magnitudes above 448 clamped to 448, the sign of zero kept.
 * Everything else as vpp_kv_append.
 */
int vpp_kv_append_fp8(const void *k_new, const void *v_new, void *k_cache,
                      void *v_cache, const float *k_scale,
                      const float *v_scale, const int32_t *block_table,
                      int32_t num_blocks, int64_t prefix_len,
                      int64_t chunk_len, int kv_heads, int head_dim_qk,
                      int head_dim_v, void *stream);

/* Varlen append (as vpp_kv_append_varlen) into an fp8 cache. */
int vpp_kv_append_varlen_fp8(const void *k_new, const void *v_new,
                             void *k_cache, void *v_cache,
                             const float *k_scale, const float *v_scale,
                             const int32_t *block_table,
                             int32_t max_blocks_per_seq, int32_t num_blocks,
                             const int32_t *cu_seqlens_q,
                             const int32_t *ctx_lens, int32_t batch,
                             int kv_heads, int head_dim_qk, int head_dim_v,
                             void *stream);

/*
 * a2..a7 over an fp8 cache: the contract of vpp_chunk_attn_ex with a bf16 q
 * and K, V read as code x scale.  Two ways, chosen by the workspace size:
 *  - workspace >= vpp_chunk_attn_fp8_workspace_size(...) (the key-split
 *    partials only, as for vpp_chunk_attn_ex: 0 without a split, independent
 *    of prefix_len): the kernel reads the codes and widens them to f16
 *    operands in shared memory (exact: every E4M3 value is an f16 value),
 *    turns q into f16 operands and applies k_scale to the scores and v_scale
 *    to the output of the row's kv head.  No copy of the cache is made; every
 *    CTA widens the tiles it reads, which costs prefill time.  q elements
 *    must lie within f16's range (|q| <= 65504): a larger one is reported as
 *    VPP_ERR_INVALID by vpp_last_device_status and its rows are not valid.
 *  - workspace >= vpp_chunk_attn_fp8_widen_workspace_size(...): keys
 *    0 .. prefix_len + chunk_len - 1 are first widened to bf16 in the
 *    workspace (exact), once, and the bf16 kernel reads that copy (faster;
 *    the copy grows with prefix_len).
 * workspace: DEVICE, 16-byte aligned.
 */
int vpp_chunk_attn_fp8(const void *q, const void *k_cache,
                       const void *v_cache, const float *k_scale,
                       const float *v_scale, const int32_t *block_table,
                       int32_t num_blocks, int64_t prefix_len,
                       int64_t chunk_len, int heads, int kv_heads,
                       int head_dim_qk, int head_dim_v, float softmax_scale,
                       int num_splits, void *out, float *lse, void *workspace,
                       size_t workspace_bytes, void *stream);

/* Workspace bytes vpp_chunk_attn_fp8 needs for these arguments (the
 * in-kernel widening). */
size_t vpp_chunk_attn_fp8_workspace_size(int64_t prefix_len,
                                         int64_t chunk_len, int heads,
                                         int kv_heads, int head_dim_qk,
                                         int head_dim_v, int num_splits);

/* Workspace bytes with which vpp_chunk_attn_fp8 widens the visible keys to a
 * bf16 copy first (the partials plus the copy). */
size_t vpp_chunk_attn_fp8_widen_workspace_size(int64_t prefix_len,
                                               int64_t chunk_len, int heads,
                                               int kv_heads, int head_dim_qk,
                                               int head_dim_v, int num_splits);

/*
 * a8..a9 over an fp8 paged cache: the contract of vpp_mixed_attn.  Decode
 * rows (the decode kernel's shapes as in vpp_mixed_attn) read the codes
 * directly.  The other sequences with queries go through the chunk-attention
 * kernel as in vpp_chunk_attn_fp8: reading the codes (q within f16's range)
 * with a workspace of vpp_mixed_attn_fp8_workspace_size(...) bytes (decode
 * partials only), or a bf16 copy of their contexts widened into a workspace
 * of vpp_mixed_attn_fp8_widen_workspace_size(...) bytes.
 */
int vpp_mixed_attn_fp8(const void *q, const void *k_cache,
                       const void *v_cache, const float *k_scale,
                       const float *v_scale, const int32_t *block_table,
                       int32_t max_blocks_per_seq, int32_t num_blocks,
                       const int32_t *cu_seqlens_q, const int32_t *ctx_lens,
                       int32_t batch, int heads, int kv_heads,
                       int head_dim_qk, int head_dim_v, float softmax_scale,
                       void *out, float *lse, void *workspace,
                       size_t workspace_bytes, void *stream);

/* Workspace bytes vpp_mixed_attn_fp8 needs (HOST cu_seqlens_q / ctx_lens). */
size_t vpp_mixed_attn_fp8_workspace_size(const int32_t *cu_seqlens_q,
                                         const int32_t *ctx_lens,
                                         int32_t batch, int heads,
                                         int kv_heads, int head_dim_qk,
                                         int head_dim_v);

/* Workspace bytes with which vpp_mixed_attn_fp8 widens the chunk-attention
 * sequences' contexts to bf16 first. */
size_t vpp_mixed_attn_fp8_widen_workspace_size(const int32_t *cu_seqlens_q,
                                               const int32_t *ctx_lens,
                                               int32_t batch, int heads,
                                               int kv_heads, int head_dim_qk,
                                               int head_dim_v);

/*
 * Top-k sparse prefix attention (DSA-style): [VPP review] §7 (sparse attention
 * breaks the linear per-chunk latency law) and [GLM PP note] §5.1 (an indexer
 * selects top-k earlier tokens for every query token; the main attention
 * reads only those).  The indexer is not part of this library: the indices
 * are inputs.
 *
 * Query token i of the chunk (absolute position prefix_len + i) attends the
 * key positions topk_idx[i][0 .. topk_len[i]-1] (DEVICE int32, row stride
 * topk, each row's valid entries first), with the same list for every head:
 *   out[i][h] = softmax_j(q[i][h] . k[j][h/G] * scale) v[j][h/G] over the list,
 * a position listed twice counting twice; lse as in vpp_chunk_attn_ex.
 * Entries outside 0 .. prefix_len + i, or in a block outside the pool, are
 * left out of the softmax and reported as VPP_ERR_INVALID in the status word;
 * a row with no usable entry (or topk_len outside 1 .. topk) gets out = 0 and
 * lse = -inf.  Cache: bf16, paged (block_table of the one sequence) or
 * contiguous (block_table NULL, num_blocks = capacity in tokens); the keys up
 * to prefix_len + chunk_len - 1 must be in it.  Shapes: those of the decode
 * kernel (head_dim 64 or 128, kv_heads <= 8, heads/kv_heads 1, 2, 4 or 8);
 * others return VPP_ERR_UNSUPPORTED.  workspace >=
 * vpp_topk_chunk_attn_workspace_size(...) (0 when topk <= 1024).
 */
int vpp_topk_chunk_attn(const void *q, const void *k_cache,
                        const void *v_cache, const int32_t *block_table,
                        int32_t num_blocks, int64_t prefix_len,
                        int64_t chunk_len, const int32_t *topk_idx,
                        const int32_t *topk_len, int32_t topk, int heads,
                        int kv_heads, int head_dim, float softmax_scale,
                        void *out, float *lse, void *workspace,
                        size_t workspace_bytes, void *stream);

/* The same over an fp8 (E4M3) cache with per-kv-head scales (see above). */
int vpp_topk_chunk_attn_fp8(const void *q, const void *k_cache,
                            const void *v_cache, const float *k_scale,
                            const float *v_scale, const int32_t *block_table,
                            int32_t num_blocks, int64_t prefix_len,
                            int64_t chunk_len, const int32_t *topk_idx,
                            const int32_t *topk_len, int32_t topk, int heads,
                            int kv_heads, int head_dim, float softmax_scale,
                            void *out, float *lse, void *workspace,
                            size_t workspace_bytes, void *stream);

/* Workspace bytes of vpp_topk_chunk_attn / _fp8 (key-range partials). */
size_t vpp_topk_chunk_attn_workspace_size(int64_t chunk_len, int32_t topk,
                                          int heads, int head_dim);

/*
 * Device status word: synchronises `stream`, stores the first error any
 * kernel of this library recorded since the last reset (VPP_OK if none) in
 * *code, and resets the word to VPP_OK.  Returns VPP_ERR_CUDA if the
 * synchronisation or copy fails.
 */
int vpp_last_device_status(void *stream, int *code);

/*
 * Self-test of the bounded device wait: launches one block that waits on a
 * shared-memory barrier nothing will ever complete, giving up after
 * timeout_us microseconds (1 .. 5,000,000).  The wait must run out and record
 * VPP_ERR_TIMEOUT in the status word; the context stays usable.
 */
int vpp_selftest_wait_timeout(int timeout_us, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* VPP_H */
