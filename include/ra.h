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
 * Debug: record the tiles the tensor-core attention kernels visit, so that the
 * ring order can be checked (the result alone cannot show it: it does not
 * depend on the visit order beyond rounding, paper review page, 排列不变性).
 *   buf : device memory of n int32 words, 16-byte aligned, or NULL to stop
 *         recording.  n >= 16.
 * From this call on, every bf16 ra_fwd, ra_bwd, ra_bwd_noalloc and ring-step
 * call made by the calling thread (until the next ra_debug_visitlog) has its
 * kernels append one entry per visited tile:
 *   buf[0]          entries claimed so far (atomically incremented; it keeps
 *                   counting past the capacity, so an overflow shows).  The
 *                   caller zeroes it before the calls it wants recorded.
 *   buf[1..7]       reserved.
 *   entry e (e < (n - 8) / 8) at buf[8 + 8e .. 8 + 8e + 7]:
 *     [0] kind (0 = forward, 1 = backward) | CTA index << 8
 *     [1] batch index, [2] head
 *     [3] the unit's home shard: the query shard j (forward) or key shard k
 *         (backward) of the unit of work
 *     [4] the unit's tile in that shard: query tile pair (forward: query tiles
 *         2u and 2u+1 of 128 rows) or key tile of 128 rows (backward)
 *     [5] ring step i
 *     [6] visited shard: the key shard (forward, k = (j - i) mod N) or query
 *         shard (backward, (k + i) mod N; paper review page, 环形注意力算法)
 *     [7] visited tile of 128 rows within that shard
 * One unit's entries are claimed in the order it visits its tiles.  Ring-step
 * calls record with shard 0 (each is one block).  Recording costs an atomic
 * per tile; with buf = NULL (the default) the kernels skip it.  The fp32 path
 * records nothing.
 */
ra_status ra_debug_visitlog(int32_t* buf, size_t n);

/*
 * Ring steps across devices (context parallelism; paper review page, 环形通信
 * and 环形注意力算法; code walk-through page, 环形计算模式).  Each device
 * holds one block of `block_len` positions of the sequence: its query block and,
 * at ring step i, the key/value block that has travelled i hops around the
 * ring.  These calls do the device-local work of one step; moving blocks
 * between devices is the caller's (a host ring driver over send/receive).
 *
 * Positions: query i of the block sits at global position q_pos0 + i * pos_stride
 * and key t at k_pos0 + t * pos_stride.  Contiguous blocks (device r holds
 * positions r * block_len ...) use pos_stride 1; striped blocks (device r
 * holds r, r + N, r + 2N, ...) use pos_stride N (paper review page, 相关工作:
 * Striped Attention, which spreads causal work evenly over the ring).  The
 * masks are the forward's, on global positions: causal_block_size c > 0 makes
 * key t visible to query i iff pos_q / c >= pos_k / c; with pos_stride > 1 only
 * c in {0, 1} is supported (RA_ERR_UNSUPPORTED otherwise).  Segment ids come
 * per block: q_segment_ids for the query block and kv_segment_ids for the
 * key/value block ([batch, block_len] int32 each; both or neither).
 * Requirements: as ra_fwd with seq = block_len and one shard, dtype RA_BF16,
 * head_dim 64 or 128, q_pos0, k_pos0 >= 0 and every position < 2^30.
 * Each call is asynchronous on `stream`; the carries are caller-owned device
 * memory that the call reads and updates.
 *
 * ra_ring_fwd_step: merges attention(q block, k/v block) into the running
 * carry: o_carry [batch, block_len, heads, head_dim] float32, the output so far
 * (normalised), and lse_carry [batch, heads, block_len] float32, its natural-log
 * log-sum-exp (-inf = nothing seen yet; start from o = 0, lse = -inf).  The
 * merge is the lazy-softmax update (code walk-through page §2) at block
 * granularity: with l_old, l_blk the two log-sum-exps, the new lse is
 * log(e^l_old + e^l_blk) and the new output the e^l-weighted mean of the old
 * carry and this block's output.  Rows with no visible key in the block keep
 * their carry.  After the last step, ra_ring_finish turns o_carry into the bf16
 * output; lse_carry is the output's lse.
 */
ra_status ra_ring_fwd_step(const void* q, const void* k, const void* v,
                           const int32_t* q_segment_ids, const int32_t* kv_segment_ids,
                           int causal_block_size, long long q_pos0, long long k_pos0, int pos_stride,
                           int batch, int block_len, int heads, int head_dim, ra_dtype dtype,
                           float* o_carry, float* lse_carry, void* stream);

/*
 * Backward ring steps.  The gradients of the query block accumulate on its
 * device; the gradients of a key/value block travel around the ring with it
 * (dK, dV float32 carries, [batch, block_len, heads, head_dim], start at 0):
 *   ra_ring_bwd_begin : once per device, before the steps: from this device's
 *                       final out (bf16), lse (the forward's lse_carry) and dout,
 *                       stores Delta = rowsum(dout * out) and lse in the
 *                       workspace and zeroes its dQ accumulator.
 *   ra_ring_bwd_step  : per ring step: adds dQ of (query block, k/v block) to
 *                       the workspace accumulator and dK, dV of the pair to
 *                       dk_carry, dv_carry (P recomputed from lse, as ra_bwd).
 *   ra_ring_bwd_end   : once, after the steps: dq (bf16) from the accumulator.
 * The workspace holds ra_ring_bwd_workspace_size(...) bytes (16-byte aligned)
 * and must not be shared by two devices' blocks.  When a key/value block is back
 * on its home device after the last step, ra_ring_finish turns its carries into
 * the bf16 dk and dv.
 */
size_t ra_ring_bwd_workspace_size(int batch, int block_len, int heads, int head_dim, ra_dtype dtype);

ra_status ra_ring_bwd_begin(const void* out, const float* lse, const void* dout,
                            int batch, int block_len, int heads, int head_dim, ra_dtype dtype,
                            void* workspace, size_t workspace_bytes, void* stream);

ra_status ra_ring_bwd_step(const void* q, const void* k, const void* v, const void* dout,
                           const int32_t* q_segment_ids, const int32_t* kv_segment_ids,
                           int causal_block_size, long long q_pos0, long long k_pos0, int pos_stride,
                           int batch, int block_len, int heads, int head_dim, ra_dtype dtype,
                           float* dk_carry, float* dv_carry,
                           void* workspace, size_t workspace_bytes, void* stream);

ra_status ra_ring_bwd_end(void* workspace, size_t workspace_bytes,
                          int batch, int block_len, int heads, int head_dim, ra_dtype dtype,
                          void* dq, void* stream);

/*
 * dst[i] = bf16(src[i]) (round to nearest even) for i < count: the last step of
 * a ring, from a float32 carry to the bf16 result.  dtype must be RA_BF16;
 * count a multiple of 4; both pointers 16-byte aligned.  One launch on `stream`.
 */
ra_status ra_ring_finish(const float* src, void* dst, size_t count, ra_dtype dtype, void* stream);

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
 *   - Every call looks up the array's device address with the calling
 *     thread's current device (so a device reset leaves no stale address).
 *     The first call on a device is special: it loads the array onto that
 *     device (64 MiB of device memory, which can fail with an out-of-memory
 *     error or synchronize the device) and, like the first call of any entry
 *     point here, clears the library's device status word with a blocking
 *     memset.  Make that first call at start-up, while allocating and
 *     synchronizing are still allowed, and before any stream capture.
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
