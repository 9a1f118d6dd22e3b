// ra_api.cu — the C ABI (include/ra.h): argument validation, dispatch to the
// kernel launchers, the device status word and per-thread error messages.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "ra.h"
#include "ra_internal.h"

#define RA_API extern "C" __attribute__((visibility("default")))

namespace ra {

__device__ int g_status;  // kernels record a timed-out wait here (one word per device)

namespace {

thread_local char t_msg[512] = "";
thread_local int* t_vlog = nullptr;  // ra_debug_visitlog target of this thread
thread_local int t_vlog_cap = 0;
std::atomic<uint64_t> g_launches{0};
std::mutex g_mu;
int* g_status_ptr[256];  // last status-word address seen per device

ra_status fail(ra_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_msg, sizeof(t_msg), fmt, ap);
  va_end(ap);
  return s;
}

ra_status ok() {
  t_msg[0] = 0;
  return RA_OK;
}

uint64_t limit_ns_from_env() {
  const char* e = getenv("RA_WAIT_LIMIT_NS");
  if (e && *e) {
    long long v = atoll(e);
    if (v > 0 && v <= 10000000000LL) return (uint64_t)v;
  }
  return 2000000000ull;  // 2 s: every legitimate wait is microseconds
}

ra_status make_ctx(void* stream, Ctx* c) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= 256) return fail(RA_ERR_CUDA, "device ordinal %d out of range", dev);
  {
    // The status word's address is looked up on every call: after a device reset
    // the module is loaded again, possibly elsewhere, and a cached address would
    // be stale.  A word at an address not seen before is cleared once.
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_status);
    if (e != cudaSuccess) return fail(RA_ERR_CUDA, "cudaGetSymbolAddress(status): %s", cudaGetErrorString(e));
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_status_ptr[dev] != (int*)p) {
      e = cudaMemset(p, 0, sizeof(int));
      if (e != cudaSuccess) return fail(RA_ERR_CUDA, "cudaMemset(status): %s", cudaGetErrorString(e));
      g_status_ptr[dev] = (int*)p;
    }
    c->status = (int*)p;
  }
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
  c->device = dev;
  c->num_sms = sms;
  c->limit_ns = limit_ns_from_env();
  c->stream = (cudaStream_t)stream;
  return RA_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

ra_status validate(const void* const* ptrs, const char* const* names, int nptr,
                   const int32_t* seg, int causal_block_size, int num_shards, int qc, int kc,
                   int B, int S, int H, int D, ra_dtype dtype, Problem* p) {
  if (dtype != RA_F32 && dtype != RA_BF16) return fail(RA_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
  if (B < 1 || H < 1 || S < 0 || D < 1)
    return fail(RA_ERR_INVALID_ARG, "bad shape B=%d S=%d H=%d D=%d", B, S, H, D);
  if ((long long)B * S * H * D >= (1LL << 31))
    return fail(RA_ERR_INVALID_ARG, "B*S*H*D = %lld must be < 2^31", (long long)B * S * H * D);
  if (num_shards < 1) return fail(RA_ERR_INVALID_ARG, "num_shards=%d must be >= 1", num_shards);
  if (S % num_shards != 0)
    return fail(RA_ERR_INVALID_ARG, "seq=%d not divisible by num_shards=%d", S, num_shards);
  if (qc < 1 || kc < 1)
    return fail(RA_ERR_INVALID_ARG, "chunk sizes must be >= 1 (query %d, key %d)", qc, kc);
  const int Ssh = S / num_shards;
  if (Ssh % qc != 0 || Ssh % kc != 0)
    return fail(RA_ERR_INVALID_ARG, "shard length %d not divisible by query_chunk_size=%d / key_chunk_size=%d",
                Ssh, qc, kc);
  if (causal_block_size < 0)
    return fail(RA_ERR_INVALID_ARG, "causal_block_size=%d must be >= 0", causal_block_size);
  for (int i = 0; i < nptr && S > 0; ++i) {  // an empty problem touches no memory
    if (ptrs[i] == nullptr) return fail(RA_ERR_INVALID_ARG, "%s is NULL", names[i]);
    if (!aligned16(ptrs[i])) return fail(RA_ERR_INVALID_ARG, "%s is not 16-byte aligned", names[i]);
  }
  if (S > 0 && seg != nullptr && !aligned16(seg)) return fail(RA_ERR_INVALID_ARG, "segment_ids is not 16-byte aligned");
  if (dtype == RA_BF16 && D != 64 && D != 128)
    return fail(RA_ERR_UNSUPPORTED, "bf16 path supports head_dim 64 and 128, got %d", D);
  if (dtype == RA_F32 && D > 128) return fail(RA_ERR_UNSUPPORTED, "fp32 path supports head_dim <= 128, got %d", D);
  p->B = B;
  p->S = S;
  p->H = H;
  p->D = D;
  p->N = num_shards;
  p->Ssh = Ssh;
  p->causal = causal_block_size;
  p->seg = seg;
  return RA_OK;
}

// Kernel position offsets for one ring step.  Query i of the block sits at
// global position q_pos0 + i * stride and key t at k_pos0 + t * stride.  With
// stride 1 the kernels compare global positions (offsets q_pos0, k_pos0).  With
// stride > 1 (striped blocks) only causal_block_size 0 or 1 is defined here:
// then key t is visible to query i iff t <= i + delta, delta =
// floor((q_pos0 - k_pos0) / stride), which the kernels see as positions i + m
// and t + m - delta with m = max(0, delta) (both offsets non-negative).
ra_status ring_offsets(int c, long long q_pos0, long long k_pos0, int stride, int S, int* qoff, int* koff) {
  if (q_pos0 < 0 || k_pos0 < 0 || stride < 1)
    return fail(RA_ERR_INVALID_ARG, "positions must be >= 0 and pos_stride >= 1 (got %lld, %lld, %d)", q_pos0, k_pos0,
                stride);
  const long long span = (long long)(S > 0 ? S - 1 : 0) * stride;
  if (q_pos0 + span >= (1LL << 30) || k_pos0 + span >= (1LL << 30))
    return fail(RA_ERR_INVALID_ARG, "positions must stay below 2^30");
  if (stride == 1) {
    *qoff = (int)q_pos0;
    *koff = (int)k_pos0;
    return RA_OK;
  }
  if (c > 1) return fail(RA_ERR_UNSUPPORTED, "strided positions support causal_block_size 0 or 1, got %d", c);
  if (c == 0) {
    *qoff = *koff = 0;
    return RA_OK;
  }
  const long long d = q_pos0 - k_pos0;
  const long long delta = d >= 0 ? d / stride : -((-d + stride - 1) / stride);  // floor division
  const long long m = delta > 0 ? delta : 0;
  *qoff = (int)m;
  *koff = (int)(m - delta);
  return RA_OK;
}

}  // namespace

// Record a message for ra_last_error() on behalf of entry points in other files.
ra_status set_last_error(ra_status s, const char* msg) { return fail(s, "%s", msg); }

}  // namespace ra

using namespace ra;

RA_API ra_status ra_fwd(const void* q, const void* k, const void* v, const int32_t* segment_ids,
                        int causal_block_size, int num_shards, int query_chunk_size, int key_chunk_size,
                        int batch, int seq, int heads, int head_dim, ra_dtype dtype, void* out, float* lse,
                        void* stream) {
  const void* ptrs[] = {q, k, v, out, lse};
  const char* names[] = {"q", "k", "v", "out", "lse"};
  FwdArgs a;
  ra_status s = validate(ptrs, names, 5, segment_ids, causal_block_size, num_shards, query_chunk_size,
                         key_chunk_size, batch, seq, heads, head_dim, dtype, &a.p);
  if (s != RA_OK) return s;
  if (seq == 0) return ok();
  Ctx c;
  if ((s = make_ctx(stream, &c)) != RA_OK) return s;
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.lse = lse;
  a.vlog = t_vlog;
  a.vlog_cap = t_vlog_cap;
  uint64_t n = 0;
  cudaError_t e;
  const char* why = nullptr;
  if (dtype == RA_F32) {
    e = launch_fwd_f32(a, c, &n);
  } else {
    e = launch_fwd_bf16(a, c, &n, &why);
  }
  g_launches += n;
  if (why) return fail(RA_ERR_UNSUPPORTED, "%s", why);
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, "forward launch: %s", cudaGetErrorString(e));
  return ok();
}

RA_API size_t ra_bwd_workspace_size(int batch, int seq, int heads, int head_dim, ra_dtype dtype) {
  if (batch < 1 || seq < 0 || heads < 1 || head_dim < 1) return 0;
  if (dtype == RA_F32) {
    return (((size_t)batch * heads * seq * sizeof(float)) + 255) & ~(size_t)255;  // Delta only
  }
  return bwd_workspace_bytes(batch, seq, heads, head_dim);
}

RA_API ra_status ra_bwd(const void* q, const void* k, const void* v, const void* out, const float* lse,
                        const void* dout, const int32_t* segment_ids, int causal_block_size, int num_shards,
                        int query_chunk_size, int key_chunk_size, int batch, int seq, int heads, int head_dim,
                        ra_dtype dtype, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                        void* stream) {
  const void* ptrs[] = {q, k, v, out, lse, dout, dq, dk, dv, workspace};
  const char* names[] = {"q", "k", "v", "out", "lse", "dout", "dq", "dk", "dv", "workspace"};
  BwdArgs a;
  ra_status s = validate(ptrs, names, 10, segment_ids, causal_block_size, num_shards, query_chunk_size,
                         key_chunk_size, batch, seq, heads, head_dim, dtype, &a.p);
  if (s != RA_OK) return s;
  const size_t need = ra_bwd_workspace_size(batch, seq, heads, head_dim, dtype);
  if (workspace_bytes < need)
    return fail(RA_ERR_INVALID_ARG, "workspace holds %zu bytes, %zu needed", workspace_bytes, need);
  if (seq == 0) return ok();
  Ctx c;
  if ((s = make_ctx(stream, &c)) != RA_OK) return s;
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.lse = lse;
  a.dout = dout;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.vlog = t_vlog;
  a.vlog_cap = t_vlog_cap;
  uint64_t n = 0;
  cudaError_t e;
  const char* why = nullptr;
  if (dtype == RA_F32) {
    a.dq_accum = nullptr;
    a.delta = (float*)workspace;
    e = launch_bwd_f32(a, c, &n);
  } else {
    a.dq_accum = (float*)workspace;
    a.delta = (float*)((char*)workspace + bwd_delta_offset(batch, seq, heads, head_dim));
    a.unit_counter = (int*)((char*)workspace + bwd_counter_offset(batch, seq, heads, head_dim));
    e = launch_bwd_bf16(a, c, &n, &why);
  }
  g_launches += n;
  if (why) return fail(RA_ERR_UNSUPPORTED, "%s", why);
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, "backward launch: %s", cudaGetErrorString(e));
  return ok();
}

RA_API size_t ra_decode_workspace_size(int batch, int new_tokens, int cache_len, int heads, int head_dim,
                                       int num_shards, ra_dtype dtype) {
  (void)dtype;
  if (batch < 1 || new_tokens < 1 || cache_len < 0 || heads < 1 || head_dim < 1 || num_shards < 1) return 0;
  return decode_workspace_bytes(batch, new_tokens, cache_len, heads, head_dim, num_shards);
}

RA_API ra_status ra_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* cache_idx,
                           const int32_t* q_segment_ids, const int32_t* kv_segment_ids, int causal_block_size,
                           int num_shards, int batch, int new_tokens, int cache_len, int heads, int head_dim,
                           ra_dtype dtype, void* out, float* lse, void* workspace, size_t workspace_bytes,
                           void* stream) {
  if (dtype != RA_F32 && dtype != RA_BF16) return fail(RA_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
  if (batch < 1 || batch > 65535 || heads < 1 || heads > 65535 || new_tokens < 0 || cache_len < 0 ||
      head_dim < 1)
    return fail(RA_ERR_INVALID_ARG, "bad shape batch=%d new_tokens=%d cache_len=%d heads=%d head_dim=%d", batch,
                new_tokens, cache_len, heads, head_dim);
  if (num_shards < 1) return fail(RA_ERR_INVALID_ARG, "num_shards=%d must be >= 1", num_shards);
  if (cache_len % num_shards != 0)
    return fail(RA_ERR_INVALID_ARG, "cache_len=%d not divisible by num_shards=%d", cache_len, num_shards);
  if (causal_block_size < 0)
    return fail(RA_ERR_INVALID_ARG, "causal_block_size=%d must be >= 0", causal_block_size);
  if ((q_segment_ids == nullptr) != (kv_segment_ids == nullptr))
    return fail(RA_ERR_INVALID_ARG, "q_segment_ids and kv_segment_ids must be given together");
  if (head_dim != 64 && head_dim != 128)
    return fail(RA_ERR_UNSUPPORTED, "decode supports head_dim 64 and 128, got %d", head_dim);
  if (new_tokens > 64) return fail(RA_ERR_UNSUPPORTED, "decode takes at most 64 new tokens, got %d", new_tokens);
  if (new_tokens == 0) return ok();
  {
    const DecodeSplit sp = decode_split(batch, new_tokens, cache_len, heads, num_shards);
    if ((long long)sp.P * heads * ((new_tokens + 7) / 8) > 0x7fffffffLL)
      return fail(RA_ERR_INVALID_ARG, "cache too long for one decode launch (%d work items per head)", sp.P);
  }
  struct {
    const void* p;
    const char* name;
    bool required;
    uintptr_t align;
  } ptrs[] = {{q, "q", true, 16},
              {k_cache, "k_cache", cache_len > 0, 16},
              {v_cache, "v_cache", cache_len > 0, 16},
              {out, "out", true, 16},
              {lse, "lse", true, 16},
              {cache_idx, "cache_idx", true, 4},
              {q_segment_ids, "q_segment_ids", false, 4},
              {kv_segment_ids, "kv_segment_ids", false, 4}};
  for (const auto& x : ptrs) {
    if (x.p == nullptr) {
      if (x.required) return fail(RA_ERR_INVALID_ARG, "%s is NULL", x.name);
      continue;
    }
    if (((uintptr_t)x.p % x.align) != 0)
      return fail(RA_ERR_INVALID_ARG, "%s is not %d-byte aligned", x.name, (int)x.align);
  }
  const size_t need = decode_workspace_bytes(batch, new_tokens, cache_len, heads, head_dim, num_shards);
  if (workspace_bytes < need)
    return fail(RA_ERR_INVALID_ARG, "workspace holds %zu bytes, %zu needed", workspace_bytes, need);
  if (need > 0 && (workspace == nullptr || !aligned16(workspace)))
    return fail(RA_ERR_INVALID_ARG, "workspace is NULL or not 16-byte aligned");
  Ctx c;
  ra_status s = make_ctx(stream, &c);
  if (s != RA_OK) return s;
  DecodeArgs a;
  a.B = batch;
  a.T = new_tokens;
  a.S = cache_len;
  a.H = heads;
  a.D = head_dim;
  a.N = num_shards;
  a.causal = causal_block_size;
  a.bf16 = dtype == RA_BF16;
  a.q = q;
  a.k = k_cache;
  a.v = v_cache;
  a.cache_idx = cache_idx;
  a.qseg = q_segment_ids;
  a.kseg = kv_segment_ids;
  a.out = out;
  a.lse = lse;
  a.workspace = workspace;
  uint64_t n = 0;
  cudaError_t e = launch_decode(a, c, &n);
  g_launches += n;
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
  return ok();
}

RA_API size_t ra_ffn_workspace_size(int batch, int seq, int ffn_dim, int chunk_size) {
  if (batch < 1 || seq < 0 || ffn_dim < 1 || chunk_size < 1) return 0;
  return ffn_workspace_bytes((long long)batch * seq, chunk_size, ffn_dim);
}

RA_API ra_status ra_blockwise_ffn(const void* x, const void* w1, const float* b1, const void* w2, const float* b2,
                                  int batch, int seq, int model_dim, int ffn_dim, int chunk_size, ra_dtype dtype,
                                  void* out, void* workspace, size_t workspace_bytes, void* stream) {
  if (dtype != RA_F32 && dtype != RA_BF16) return fail(RA_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
  if (batch < 1 || seq < 0 || model_dim < 1 || ffn_dim < 1 || chunk_size < 1)
    return fail(RA_ERR_INVALID_ARG, "bad shape batch=%d seq=%d model_dim=%d ffn_dim=%d chunk_size=%d", batch, seq,
                model_dim, ffn_dim, chunk_size);
  if (model_dim % 8 != 0 || ffn_dim % 8 != 0)
    return fail(RA_ERR_INVALID_ARG, "model_dim (%d) and ffn_dim (%d) must be multiples of 8", model_dim, ffn_dim);
  if ((long long)batch * seq >= (1LL << 31))
    return fail(RA_ERR_INVALID_ARG, "batch * seq must be < 2^31");
  if (dtype != RA_BF16) return fail(RA_ERR_UNSUPPORTED, "the blockwise feed-forward supports bf16 only");
  if (seq == 0) return ok();
  struct {
    const void* p;
    const char* name;
    bool required;
  } ptrs[] = {{x, "x", true}, {w1, "w1", true}, {w2, "w2", true}, {out, "out", true},
              {workspace, "workspace", true}, {b1, "b1", false}, {b2, "b2", false}};
  for (const auto& q : ptrs) {
    if (q.p == nullptr) {
      if (q.required) return fail(RA_ERR_INVALID_ARG, "%s is NULL", q.name);
      continue;
    }
    if (!aligned16(q.p)) return fail(RA_ERR_INVALID_ARG, "%s is not 16-byte aligned", q.name);
  }
  const size_t need = ffn_workspace_bytes((long long)batch * seq, chunk_size, ffn_dim);
  if (workspace_bytes < need)
    return fail(RA_ERR_INVALID_ARG, "workspace holds %zu bytes, %zu needed", workspace_bytes, need);
  Ctx c;
  ra_status s = make_ctx(stream, &c);
  if (s != RA_OK) return s;
  FfnArgs a;
  a.B = batch;
  a.L = seq;
  a.Dm = model_dim;
  a.F = ffn_dim;
  a.chunk = chunk_size;
  a.x = x;
  a.w1 = w1;
  a.b1 = b1;
  a.w2 = w2;
  a.b2 = b2;
  a.out = out;
  a.hidden = workspace;
  uint64_t n = 0;
  const char* why = nullptr;
  cudaError_t e = launch_ffn(a, c, &n, &why);
  g_launches += n;
  if (why) return fail(RA_ERR_UNSUPPORTED, "%s", why);
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, "feed-forward launch: %s", cudaGetErrorString(e));
  return ok();
}

RA_API ra_status ra_sync_check(void* stream) {
  Ctx c;
  ra_status s = make_ctx(stream, &c);
  if (s != RA_OK) return s;
  cudaError_t e = cudaStreamSynchronize(c.stream);
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, "stream synchronize: %s", cudaGetErrorString(e));
  int word = 0;
  e = cudaMemcpy(&word, c.status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, "reading status word: %s", cudaGetErrorString(e));
  if (word != 0) {
    int zero = 0;
    cudaMemcpy(c.status, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (word & 0x20000) return fail(RA_ERR_CUDA, "a kernel found its shared memory misaligned and did nothing");
    return fail(RA_ERR_TIMEOUT, "a device-side wait ran out (site %d)", word & 0xFFFF);
  }
  return ok();
}

RA_API const char* ra_last_error(void) { return t_msg; }

RA_API uint64_t ra_kernel_launches(void) { return g_launches.load(); }

RA_API ra_status ra_selftest_timeout(int64_t limit_ns, void* stream) {
  if (limit_ns < 1 || limit_ns > 1000000000LL)
    return fail(RA_ERR_INVALID_ARG, "limit_ns=%lld must be in [1, 1e9]", (long long)limit_ns);
  Ctx c;
  ra_status s = make_ctx(stream, &c);
  if (s != RA_OK) return s;
  c.limit_ns = (uint64_t)limit_ns;
  uint64_t n = 0;
  cudaError_t e = launch_selftest_timeout(c, &n);
  g_launches += n;
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, "selftest launch: %s", cudaGetErrorString(e));
  return ok();
}

RA_API ra_status ra_debug_visitlog(int32_t* buf, size_t n) {
  if (buf == nullptr) {
    t_vlog = nullptr;
    t_vlog_cap = 0;
    return ok();
  }
  if (!aligned16(buf)) return fail(RA_ERR_INVALID_ARG, "visit log buffer is not 16-byte aligned");
  if (n < 16) return fail(RA_ERR_INVALID_ARG, "visit log needs at least 16 words (8 header + one entry), got %zu", n);
  const size_t cap = (n - 8) / 8;
  t_vlog = buf;
  t_vlog_cap = (int)(cap > 0x7fffffff ? 0x7fffffff : cap);
  return ok();
}

// ----------------------------------------------------------------------------- ring steps

namespace {

ra_status ring_common(const void* const* ptrs, const char* const* names, int nptr, const int32_t* qseg,
                      const int32_t* kseg, int c, long long q_pos0, long long k_pos0, int stride, int B, int S, int H,
                      int D, ra_dtype dtype, Problem* p, CallExtras* x) {
  if ((qseg == nullptr) != (kseg == nullptr))
    return fail(RA_ERR_INVALID_ARG, "q_segment_ids and kv_segment_ids must be given together");
  ra_status s = validate(ptrs, names, nptr, qseg, c, 1, S > 0 ? S : 1, S > 0 ? S : 1, B, S, H, D, dtype, p);
  if (s != RA_OK) return s;
  if (dtype != RA_BF16) return fail(RA_ERR_UNSUPPORTED, "ring steps support bf16 only");
  if (S > 0 && kseg != nullptr && !aligned16(kseg)) return fail(RA_ERR_INVALID_ARG, "kv_segment_ids is not 16-byte aligned");
  if ((s = ring_offsets(c, q_pos0, k_pos0, stride, S, &x->qoff, &x->koff)) != RA_OK) return s;
  if (stride > 1 && c == 1) p->causal = 1;
  x->kseg = kseg;
  x->vlog = t_vlog;
  x->vlog_cap = t_vlog_cap;
  return RA_OK;
}

}  // namespace

RA_API ra_status ra_ring_fwd_step(const void* q, const void* k, const void* v, const int32_t* q_segment_ids,
                                  const int32_t* kv_segment_ids, int causal_block_size, long long q_pos0,
                                  long long k_pos0, int pos_stride, int batch, int block_len, int heads, int head_dim,
                                  ra_dtype dtype, float* o_carry, float* lse_carry, void* stream) {
  const void* ptrs[] = {q, k, v, o_carry, lse_carry};
  const char* names[] = {"q", "k", "v", "o_carry", "lse_carry"};
  FwdArgs a;
  ra_status s = ring_common(ptrs, names, 5, q_segment_ids, kv_segment_ids, causal_block_size, q_pos0, k_pos0,
                            pos_stride, batch, block_len, heads, head_dim, dtype, &a.p, &a);
  if (s != RA_OK) return s;
  if (block_len == 0) return ok();
  Ctx c;
  if ((s = make_ctx(stream, &c)) != RA_OK) return s;
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = nullptr;
  a.lse = nullptr;
  a.o_carry = o_carry;
  a.lse_carry = lse_carry;
  uint64_t n = 0;
  const char* why = nullptr;
  cudaError_t e = launch_fwd_bf16(a, c, &n, &why);
  g_launches += n;
  if (why) return fail(RA_ERR_UNSUPPORTED, "%s", why);
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, "ring forward step launch: %s", cudaGetErrorString(e));
  return ok();
}

RA_API size_t ra_ring_bwd_workspace_size(int batch, int block_len, int heads, int head_dim, ra_dtype dtype) {
  if (dtype != RA_BF16) return 0;
  return ra_bwd_workspace_size(batch, block_len, heads, head_dim, dtype);
}

namespace {

ra_status ring_bwd_launch(BwdArgs& a, void* workspace, size_t workspace_bytes, void* stream) {
  const Problem& p = a.p;
  const size_t need = bwd_workspace_bytes(p.B, p.S, p.H, p.D);
  if (workspace_bytes < need)
    return fail(RA_ERR_INVALID_ARG, "workspace holds %zu bytes, %zu needed", workspace_bytes, need);
  if (p.S == 0) return ok();
  Ctx c;
  ra_status s = make_ctx(stream, &c);
  if (s != RA_OK) return s;
  a.dq_accum = (float*)workspace;
  a.delta = (float*)((char*)workspace + bwd_delta_offset(p.B, p.S, p.H, p.D));
  a.unit_counter = (int*)((char*)workspace + bwd_counter_offset(p.B, p.S, p.H, p.D));
  uint64_t n = 0;
  const char* why = nullptr;
  cudaError_t e = launch_bwd_bf16(a, c, &n, &why);
  g_launches += n;
  if (why) return fail(RA_ERR_UNSUPPORTED, "%s", why);
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, "ring backward launch: %s", cudaGetErrorString(e));
  return ok();
}

}  // namespace

RA_API ra_status ra_ring_bwd_begin(const void* out, const float* lse, const void* dout, int batch, int block_len,
                                   int heads, int head_dim, ra_dtype dtype, void* workspace, size_t workspace_bytes,
                                   void* stream) {
  const void* ptrs[] = {out, lse, dout, workspace};
  const char* names[] = {"out", "lse", "dout", "workspace"};
  BwdArgs a;
  ra_status s = ring_common(ptrs, names, 4, nullptr, nullptr, 0, 0, 0, 1, batch, block_len, heads, head_dim, dtype,
                            &a.p, &a);
  if (s != RA_OK) return s;
  a.stage = kBwdRingBegin;
  a.out = out;
  a.lse = lse;
  a.dout = dout;
  return ring_bwd_launch(a, workspace, workspace_bytes, stream);
}

RA_API ra_status ra_ring_bwd_step(const void* q, const void* k, const void* v, const void* dout,
                                  const int32_t* q_segment_ids, const int32_t* kv_segment_ids, int causal_block_size,
                                  long long q_pos0, long long k_pos0, int pos_stride, int batch, int block_len,
                                  int heads, int head_dim, ra_dtype dtype, float* dk_carry, float* dv_carry,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  const void* ptrs[] = {q, k, v, dout, dk_carry, dv_carry, workspace};
  const char* names[] = {"q", "k", "v", "dout", "dk_carry", "dv_carry", "workspace"};
  BwdArgs a;
  ra_status s = ring_common(ptrs, names, 7, q_segment_ids, kv_segment_ids, causal_block_size, q_pos0, k_pos0,
                            pos_stride, batch, block_len, heads, head_dim, dtype, &a.p, &a);
  if (s != RA_OK) return s;
  a.stage = kBwdRingStep;
  a.q = q;
  a.k = k;
  a.v = v;
  a.dout = dout;
  a.dk_carry = dk_carry;
  a.dv_carry = dv_carry;
  return ring_bwd_launch(a, workspace, workspace_bytes, stream);
}

RA_API ra_status ra_ring_bwd_end(void* workspace, size_t workspace_bytes, int batch, int block_len, int heads,
                                 int head_dim, ra_dtype dtype, void* dq, void* stream) {
  const void* ptrs[] = {workspace, dq};
  const char* names[] = {"workspace", "dq"};
  BwdArgs a;
  ra_status s = ring_common(ptrs, names, 2, nullptr, nullptr, 0, 0, 0, 1, batch, block_len, heads, head_dim, dtype,
                            &a.p, &a);
  if (s != RA_OK) return s;
  a.stage = kBwdRingEnd;
  a.dq = dq;
  return ring_bwd_launch(a, workspace, workspace_bytes, stream);
}

RA_API ra_status ra_ring_finish(const float* src, void* dst, size_t count, ra_dtype dtype, void* stream) {
  if (dtype != RA_BF16) return fail(RA_ERR_UNSUPPORTED, "ra_ring_finish writes bf16 only");
  if (count == 0) return ok();
  if (src == nullptr || dst == nullptr) return fail(RA_ERR_INVALID_ARG, "src or dst is NULL");
  if (!aligned16(src) || !aligned16(dst)) return fail(RA_ERR_INVALID_ARG, "src and dst must be 16-byte aligned");
  if (count % 4 != 0) return fail(RA_ERR_INVALID_ARG, "count must be a multiple of 4, got %zu", count);
  Ctx c;
  ra_status s = make_ctx(stream, &c);
  if (s != RA_OK) return s;
  uint64_t n = 0;
  cudaError_t e = launch_cast_bf16(src, dst, count, 1.0f, c, &n);
  g_launches += n;
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, "ring finish launch: %s", cudaGetErrorString(e));
  return ok();
}
