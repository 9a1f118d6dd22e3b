/*
 * ra.h — C ABI of the GB300 (sm_103a) blockwise ring attention library (libra.so).
 *
 * What it computes
 * ----------------
 * Exact softmax attention  out = softmax(Q K^T / sqrt(d)) V  per (batch, head)
 * ("Ring Attention with Blockwise Transformers for Near-Infinite Context",
 * paper review page, §三 核心公式 / 自注意力), evaluated the Ring Attention way:
 * the sequence is cut into `num_shards` equal contiguous blocks (same page,
 * 分块注意力), and every query block j combines the key/value blocks in ring
 * order k = (j - i) mod N, i = 0..N-1 (same page, 环形注意力算法), with the
 * lazy-softmax running max / numerator / denominator update
 * ("从论文到代码：深入理解RingAttention的块注意力计算逻辑", §2 数值稳定的注意力计算).
 * On one GPU the N ring devices are N virtual shards visited inside one
 * launch; there is no collective.  Masks:
 *   causal_block_size c > 0:  key j visible to query i iff i / c >= j / c
 *                             (integer division; code walk-through page §3).
 *                             Tiles with no visible element are skipped.
 *   segment_ids (optional):   key j visible to query i iff ids are equal.
 * The result does not depend on the visit order beyond rounding (paper review
 * page, 排列不变性), so query_chunk_size / key_chunk_size are validated (the
 * pages floor-divide the shard by them, code walk-through page §1) but do not
 * change the result; the kernels use their own 128-row tiles inside each shard.
 *
 * Layouts (all row-major, contiguous, device memory)
 * ------------------------------------------------
 *   q, k, v, out, dout, dq, dk, dv : [batch, seq, heads, head_dim], element type `dtype`
 *   lse                            : [batch, heads, seq] float32, natural-log
 *                                    log-sum-exp of the scaled scores of each query row
 *                                    (-inf for a row with no visible key; its out row is 0)
 *   segment_ids                    : [batch, seq] int32, or NULL for no segment mask
 *
 * Supported: dtype RA_BF16 with head_dim in {64, 128} (tensor-core path:
 * TMA-staged tiles, tcgen05 MMAs accumulating in tensor memory), and dtype
 * RA_F32 with 1 <= head_dim <= 128 (exact fp32 CUDA-core path).
 * Requirements (else RA_ERR_INVALID_ARG): non-NULL tensor pointers, every
 * pointer 16-byte aligned (pointers are not examined when seq = 0), batch, heads >= 1, seq >= 0, num_shards >= 1,
 * seq % num_shards == 0, (seq / num_shards) % query_chunk_size == 0 and
 * % key_chunk_size == 0 (chunk sizes >= 1; seq = 0 is an empty problem and
 * returns RA_OK at once), causal_block_size >= 0, and
 * batch*seq*heads*head_dim < 2^31.
 *
 * Ownership and streams
 * ---------------------
 * The caller allocates every buffer.  The library allocates no device memory,
 * keeps no pointer after a call returns, and enqueues all work on `stream`
 * (a cudaStream_t; NULL = the legacy default stream).  Calls are asynchronous:
 * a CUDA launch error is reported at once (RA_ERR_CUDA); a device-side wait
 * that ran out (RA_ERR_TIMEOUT) is recorded in a device status word and
 * reported by ra_sync_check.
 *
 * Errors
 * ------
 * Every function returns an ra_status.  On a non-OK status ra_last_error()
 * returns a message for the calling thread.  No function aborts the process.
 */
#ifndef RA_H_
#define RA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  RA_OK = 0,
  RA_ERR_INVALID_ARG = 1,  /* bad pointer, shape, alignment or divisibility */
  RA_ERR_UNSUPPORTED = 2,  /* valid request this library does not implement */
  RA_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed          */
  RA_ERR_TIMEOUT = 4       /* a bounded device-side wait ran out            */
} ra_status;

typedef enum { RA_F32 = 0, RA_BF16 = 1 } ra_dtype;

/*
 * Forward: out, lse <- attention(q, k, v).
 * One persistent kernel launch for RA_BF16; one launch for RA_F32.
 * RA_BF16 outside stream capture: before the launch the call takes a 16-byte
 * unit counter from a stream-ordered memory pool of the library's own (created
 * on the device's first call, memory kept between calls), zeroes it on
 * `stream` and frees it on `stream` after the launch, so that the kernel's
 * CTAs take query-tile units as they free up.  Under stream capture it uses a
 * fixed schedule instead; both give bit-identical results.
 */
ra_status ra_fwd(const void* q, const void* k, const void* v,
                 const int32_t* segment_ids, int causal_block_size,
                 int num_shards, int query_chunk_size, int key_chunk_size,
                 int batch, int seq, int heads, int head_dim, ra_dtype dtype,
                 void* out, float* lse, void* stream);

/*
 * Bytes of device scratch that ra_bwd needs for this shape (float32 dQ
 * accumulator, the per-row Delta = rowsum(dO * out), and for RA_BF16 the main
 * kernel's unit counter).  The caller allocates it; its contents on entry do
 * not matter (the call initialises what it reads).
 */
size_t ra_bwd_workspace_size(int batch, int seq, int heads, int head_dim, ra_dtype dtype);

/*
 * Backward: dq, dk, dv <- gradients of sum(dout * out) with respect to q, k, v,
 * recomputing P = exp(S - lse) from the saved lse (no S x S matrix is stored).
 * `out` and `lse` are the forward's results for the same inputs.  Same
 * arguments and rules as ra_fwd; `workspace` must hold
 * ra_bwd_workspace_size(...) bytes (16-byte aligned).
 */
ra_status ra_bwd(const void* q, const void* k, const void* v,
                 const void* out, const float* lse, const void* dout,
                 const int32_t* segment_ids, int causal_block_size,
                 int num_shards, int query_chunk_size, int key_chunk_size,
                 int batch, int seq, int heads, int head_dim, ra_dtype dtype,
                 void* dq, void* dk, void* dv,
                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * Decoding against a KV cache (the `cache_idx` inference path).
 *
 * T = new_tokens query tokens per batch row attend to a key/value cache of
 * capacity S = cache_len (comparison page "RingAttention与传统注意力机制对比为
 * 什么它是大语言模型的终极解决方案", §关键参数配置: cache_idx, the inference
 * cache index; §推理成本显著降低: incremental decoding with a KV cache).
 *   - New token t of batch row b sits at position cache_idx[b] + t.  Its key
 *     and value must already be in the cache at that position (the caller
 *     writes them; this call only reads the cache).
 *   - The cache holds L_b = clamp(cache_idx[b] + T, 0, S) filled entries;
 *     entries j >= L_b are not keys.  Key j is visible to token t iff j < L_b,
 *     the causal block rule (cache_idx[b] + t) / c >= j / c holds (c =
 *     causal_block_size > 0; a negative position sees nothing) and, with
 *     segment ids, q_segment_ids[b, t] == kv_segment_ids[b, j].
 *   - The cache is cut into num_shards contiguous virtual shards.  Each shard
 *     is reduced to lazy-softmax partials and every token merges the shards in
 *     ring order k = (j - i) mod N from its home shard j = pos / (S / N)
 *     (paper review page, 环形注意力算法; code walk-through page §2).
 * Layouts (row-major, contiguous, device memory):
 *   q, out                : [batch, new_tokens, heads, head_dim], element type `dtype`
 *   k_cache, v_cache      : [batch, cache_len, heads, head_dim], element type `dtype`
 *   cache_idx             : [batch] int32 (device memory, read by the kernels)
 *   q_segment_ids         : [batch, new_tokens] int32, kv_segment_ids: [batch, cache_len]
 *                           int32; both or neither (NULL = no segment mask)
 *   lse                   : [batch, heads, new_tokens] float32, natural log;
 *                           a token with no visible key gets out = 0, lse = -inf
 * Supported: dtype RA_BF16 or RA_F32 with head_dim in {64, 128}; 1 <= new_tokens
 * <= 64 (new_tokens = 0 returns RA_OK at once).  Requirements (else
 * RA_ERR_INVALID_ARG): batch, heads in [1, 65535], cache_len >= 0,
 * cache_len % num_shards == 0, causal_block_size >= 0, q, out, lse, cache_idx
 * non-NULL, k_cache and v_cache non-NULL when cache_len > 0, tensor pointers
 * 16-byte aligned and int32 pointers 4-byte aligned, workspace of at least
 * ra_decode_workspace_size(...) bytes (16-byte aligned; NULL allowed when
 * that size is 0).  Two kernel launches on `stream`, asynchronous.
 */
size_t ra_decode_workspace_size(int batch, int new_tokens, int cache_len, int heads, int head_dim,
                                int num_shards, ra_dtype dtype);

ra_status ra_decode(const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* cache_idx, const int32_t* q_segment_ids,
                    const int32_t* kv_segment_ids, int causal_block_size, int num_shards,
                    int batch, int new_tokens, int cache_len, int heads, int head_dim,
                    ra_dtype dtype, void* out, float* lse,
                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * Blockwise feed-forward network (the other half of a blockwise transformer
 * layer): out = FFN(x) = max(0, x W1 + b1) W2 + b2 for every row (paper review
 * page), computed on chunks of `chunk_size` rows of the flattened
 * (batch * seq) axis one after another, so that only one chunk's hidden
 * activation exists at a time ("Blockwise Feedforward网络详解RingAttention如何
 * 实现内存高效的前向传播", §核心技术原理, §分块重组机制).  The result does not
 * depend on chunk_size.
 * Layouts (row-major, contiguous, device memory, bf16 unless noted):
 *   x, out     : [batch, seq, model_dim]
 *   w1         : [ffn_dim, model_dim]  (W1 transposed, as a linear layer stores it)
 *   w2         : [model_dim, ffn_dim]  (W2 transposed)
 *   b1, b2     : [ffn_dim], [model_dim] float32, or NULL for no bias
 *   workspace  : ra_ffn_workspace_size(...) bytes: one chunk's hidden activation,
 *                [min(batch*seq, chunk_size), ffn_dim] bf16 (contents on entry do not matter)
 * Numerics: products in bf16 on the tensor cores with fp32 accumulation; the
 * bias and ReLU are applied in fp32, and the hidden activation is rounded to
 * bf16 once (it is stored in that type between the two products).
 * Supported: dtype RA_BF16.  Requirements (else RA_ERR_INVALID_ARG): batch,
 * model_dim, ffn_dim, chunk_size >= 1, seq >= 0 (0 returns RA_OK at once),
 * model_dim and ffn_dim multiples of 8, batch*seq < 2^31, non-NULL tensor
 * pointers (b1, b2 may be NULL), every pointer 16-byte aligned.  Two kernel
 * launches per chunk on `stream`, asynchronous.
 */
size_t ra_ffn_workspace_size(int batch, int seq, int ffn_dim, int chunk_size);

ra_status ra_blockwise_ffn(const void* x, const void* w1, const float* b1, const void* w2, const float* b2,
                           int batch, int seq, int model_dim, int ffn_dim, int chunk_size, ra_dtype dtype,
                           void* out, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Synchronize `stream`, then read and clear the device status word that the
 * kernels set when a bounded wait runs out.  Returns RA_ERR_TIMEOUT (message
 * names the wait site) if any kernel gave up since the last check,
 * RA_ERR_CUDA if the stream reports an error, else RA_OK.
 */
ra_status ra_sync_check(void* stream);

/* Message for the last non-OK status returned to the calling thread ("" if none). */
const char* ra_last_error(void);

/* Number of kernels this library has launched in this process (all devices). */
uint64_t ra_kernel_launches(void);

/*
 * Diagnostic: launch one tiny kernel that waits on a barrier nothing will
 * ever complete, bounded by `limit_ns` nanoseconds (<= 1e9).  The kernel gives
 * up, records a timeout in the device status word and returns, leaving the
 * context usable; ra_sync_check then reports RA_ERR_TIMEOUT.
 */
ra_status ra_selftest_timeout(int64_t limit_ns, void* stream);

/*
 * Size in bytes of the built-in scratch array used by ra_bwd_noalloc (64 MiB).
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot allocate device memory.
 */
#define RA_NOALLOC_SCRATCH_BYTES (64u << 20)

/*
 * Backward without a caller workspace, for callers that cannot allocate device
 * memory (no cudaMalloc where they run: fixed arenas, runtimes that forbid
 * allocation after start-up, code that must not synchronize the device).  Same
 * arguments, results and rules as ra_bwd, minus the workspace: the scratch is
 * a RA_NOALLOC_SCRATCH_BYTES array in the library's device image, held by
 * every GPU that uses this call until the process exits.  This function calls
 * no cudaMalloc, cudaFree or other allocating routine.
 *   - Problems whose ra_bwd_workspace_size(...) exceeds the array are
 *     rejected with RA_ERR_INVALID_ARG (use ra_bwd instead).
 *   - The first call on a device looks up the array's device address (once,
 *     with that device current); make that first call before any stream
 *     capture.
 *   - All calls on a device share the array, which keeps the last call's
 *     contents (the part that must start at zero is cleared by every call).
 *     Calls that overlap on the GPU (unordered streams) race on it.
 */
ra_status ra_bwd_noalloc(const void* q, const void* k, const void* v,
                         const void* out, const float* lse, const void* dout,
                         const int32_t* segment_ids, int causal_block_size,
                         int num_shards, int query_chunk_size, int key_chunk_size,
                         int batch, int seq, int heads, int head_dim, ra_dtype dtype,
                         void* dq, void* dk, void* dv, void* stream);

/* RA_NOALLOC_SCRATCH_BYTES, as built into the library. */
size_t ra_bwd_noalloc_max_scratch(void);

#ifdef __cplusplus
}
#endif

#endif /* RA_H_ */
