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
std::atomic<uint64_t> g_launches{0};
std::mutex g_mu;
int* g_status_ptr[256];
bool g_status_init[256];

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
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_init[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_status);
      if (e != cudaSuccess)
        return fail(RA_ERR_CUDA, "cudaGetSymbolAddress(status): %s", cudaGetErrorString(e));
      e = cudaMemset(p, 0, sizeof(int));
      if (e != cudaSuccess) return fail(RA_ERR_CUDA, "cudaMemset(status): %s", cudaGetErrorString(e));
      g_status_ptr[dev] = (int*)p;
      g_status_init[dev] = true;
    }
    c->status = g_status_ptr[dev];
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
