// decode_sm103.cu — decoding T new tokens against a sharded KV cache.
//
// The comparison page "RingAttention与传统注意力机制对比为什么它是大语言模型的
// 终极解决方案" lists `cache_idx` (the inference cache index) among the
// attention's parameters (§关键参数配置) and names incremental decoding with a
// KV cache as a use of the blockwise computation (§推理成本显著降低).  Reading:
// new token t of batch row b sits at position cache_idx[b] + t, its K/V are
// already in the cache, the cache holds L_b = clamp(cache_idx[b] + T, 0, S)
// filled entries, and key j is visible iff j < L_b and the forward's causal
// block and segment masks allow it.  The cache is cut into N contiguous
// virtual shards; each shard's keys are reduced to lazy-softmax partials
// (running max, numerator, denominator; code walk-through page §2) and a
// token merges the shards in ring order k = (j - i) mod N starting from its
// home shard j (paper review page, 环形注意力算法).
//
// The work is a stream over the cache (2 * L_b * H * D elements per batch
// row, each read once) with O(T * D) arithmetic per key row, so it runs on
// the CUDA cores and is bounded by HBM bandwidth:
//   1. partial kernel: one CTA (8 warps) per (batch, head, shard, key
//      chunk).  A warp takes 8-key tiles, staged by cp.async into its own
//      ring in shared memory: every lane reads its D/32 elements of the 8
//      key rows, multiplies by q, and a butterfly of 7 shuffles plus two
//      exchanges between lane groups leaves lanes j, j + 8, ... with the
//      score of key j.  Online softmax in log2 units, then the 8 value rows
//      are accumulated the same way.  The warps' states are merged in shared
//      memory into one partial (m, l, o) per CTA.
//   2. combine kernel: one CTA per (batch, head, token) merges the partials in
//      ring order and writes out = o / l and lse = (m + log2 l) * ln 2.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cuda_bf16.h>

#include "ra_internal.h"

namespace ra {
namespace {

constexpr int kTokGroup = 8;  // new tokens handled per CTA (larger T: more CTAs)
constexpr float kNegInf = -INFINITY;

struct DecParams {
  int B, T, S, H, D, N, Ssh, causal;
  int split_len;        // keys per work item (the last item of a shard may be shorter)
  int items_per_shard;  // ceil(Ssh / split_len)
  int P;                // partials per (b, h, token) = N * items_per_shard
  int tgroups;          // ceil(T / kTokGroup)
  const void* q;
  const void* k;
  const void* v;
  const int32_t* cache_idx;
  const int32_t* qseg;  // [B, T] or nullptr
  const int32_t* kseg;  // [B, S] or nullptr
  float* part_o;        // [B, H, T, P, D]
  float2* part_ml;      // [B, H, T, P]: (m in log2 units, l)
  void* out;            // [B, T, H, D]
  float* lse;           // [B, H, T]
  float scale_log2;     // log2(e) / sqrt(D)
};

// One lane's D/32 elements of a row, kept as raw words until used.
template <typename E, int D>
struct Frag;
template <int D>
struct Frag<__nv_bfloat16, D> {
  static constexpr int DPL = D / 32;
  static constexpr int W = DPL / 2;  // bf16 pairs
  uint32_t w[W];
  __device__ __forceinline__ void load(const __nv_bfloat16* row, int lane) {
    const uint32_t* p = reinterpret_cast<const uint32_t*>(row + lane * DPL);
    if constexpr (W == 2) {
      const uint2 x = __ldg(reinterpret_cast<const uint2*>(p));
      w[0] = x.x;
      w[1] = x.y;
    } else {
      w[0] = __ldg(p);
    }
  }
  __device__ __forceinline__ void load_shared(const __nv_bfloat16* row, int lane) {
    const uint32_t* p = reinterpret_cast<const uint32_t*>(row + lane * DPL);
    if constexpr (W == 2) {
      const uint2 x = *reinterpret_cast<const uint2*>(p);
      w[0] = x.x;
      w[1] = x.y;
    } else {
      w[0] = *p;
    }
  }
  __device__ __forceinline__ void clear() {
#pragma unroll
    for (int i = 0; i < W; ++i) w[i] = 0u;
  }
  __device__ __forceinline__ float get(int i) const {
    const uint32_t x = w[i >> 1];
    return __uint_as_float((i & 1) ? (x & 0xFFFF0000u) : (x << 16));
  }
};
template <int D>
struct Frag<float, D> {
  static constexpr int DPL = D / 32;
  float w[DPL];
  __device__ __forceinline__ void load(const float* row, int lane) {
    const float* p = row + lane * DPL;
    if constexpr (DPL == 4) {
      const float4 x = __ldg(reinterpret_cast<const float4*>(p));
      w[0] = x.x;
      w[1] = x.y;
      w[2] = x.z;
      w[3] = x.w;
    } else {
      const float2 x = __ldg(reinterpret_cast<const float2*>(p));
      w[0] = x.x;
      w[1] = x.y;
    }
  }
  __device__ __forceinline__ void load_shared(const float* row, int lane) {
    const float* p = row + lane * DPL;
    if constexpr (DPL == 4) {
      const float4 x = *reinterpret_cast<const float4*>(p);
      w[0] = x.x;
      w[1] = x.y;
      w[2] = x.z;
      w[3] = x.w;
    } else {
      const float2 x = *reinterpret_cast<const float2*>(p);
      w[0] = x.x;
      w[1] = x.y;
    }
  }
  __device__ __forceinline__ void clear() {
#pragma unroll
    for (int i = 0; i < DPL; ++i) w[i] = 0.f;
  }
  __device__ __forceinline__ float get(int i) const { return w[i]; }
};

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// ---------------------------------------------------------------------------
// 1. partials: grid (H * tgroups * items, B), WARPS warps per CTA.  The head
//    index varies fastest, so the CTAs that run together read the same key
//    rows of all heads: every [H, D] row of the cache is read whole, close in
//    time (DRAM row locality; a head's share of a row is only D elements).
//    Every warp streams its own 16-key tiles (keys kb .. kb+15, tiles of the
//    CTA's range taken round-robin by the warps) through an NST-stage ring in
//    shared memory filled with cp.async: the loads in flight hold no
//    registers, so (NST - 1) tiles per warp are always on their way.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  // src_bytes 0 writes 16 zero bytes and reads nothing
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

constexpr int kTileKeys = 8;

// CTA shape per element type and head dim: WARPS warps, NST ring stages per
// warp.  bf16: 8 warps x 3 stages x 4 KB (D = 128) = 96 KB, two CTAs per SM.
template <typename E, int D>
struct DecShape {
  static constexpr int ROWB = D * (int)sizeof(E);
  static constexpr int TILEB = kTileKeys * ROWB;  // K (or V) of one tile
  static constexpr int STAGEB = 2 * TILEB;
  static constexpr int WARPS = 8;
  static constexpr int NST = STAGEB <= 2048 ? 4 : 3;
  static constexpr int RING = WARPS * NST * STAGEB;
  static constexpr int CPL = TILEB / 16 / 32;  // 16-byte chunks per lane per tile of K (or V)
  static_assert(TILEB % (16 * 32) == 0, "tile must split into whole 16-byte chunks per lane");
};

template <typename E, int D, int TM>
constexpr int dec_smem_bytes() {
  using C = DecShape<E, D>;
  constexpr int merge = C::WARPS * TM * (D + 2) * 4;
  return C::RING > merge ? C::RING : merge;
}

template <typename E, int D, int TM>
__global__ void __launch_bounds__(DecShape<E, D>::WARPS * 32) decode_partial_kernel(DecParams p) {
  using F = Frag<E, D>;
  using C = DecShape<E, D>;
  constexpr int DPL = F::DPL;
  constexpr int WARPS = C::WARPS, NST = C::NST;
  extern __shared__ __align__(128) uint8_t dsm[];
  const int h = blockIdx.x % p.H;
  const int t0 = ((blockIdx.x / p.H) % p.tgroups) * kTokGroup;
  const int item = blockIdx.x / (p.H * p.tgroups);
  const int b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = min(TM, p.T - t0);  // tokens of this CTA

  const int shard = item / p.items_per_shard;
  const int r = item % p.items_per_shard;
  const int lo = shard * p.Ssh + r * p.split_len;
  const int idx = __ldg(p.cache_idx + b);
  const long long filled = min((long long)p.S, max(0LL, (long long)idx + p.T));
  const int hi = (int)min((long long)min(lo + p.split_len, (shard + 1) * p.Ssh), filled);

  float m[TM], l[TM], o[TM][DPL], qv[TM][DPL];
  int qs[TM], kmax[TM];  // kmax: first key the causal block rule hides from the token
#pragma unroll
  for (int t = 0; t < TM; ++t) {
    const long long pos = (long long)idx + t0 + t;
    long long lim = 0x7fffffffLL;
    if (p.causal > 0) lim = pos < 0 ? 0 : (pos / p.causal + 1) * p.causal;
    kmax[t] = (int)min(lim, 0x7fffffffLL);
    m[t] = kNegInf;
    l[t] = 0.f;
#pragma unroll
    for (int i = 0; i < DPL; ++i) o[t][i] = 0.f;
    if (t < nt) {
      F qf;
      qf.load(reinterpret_cast<const E*>(p.q) + (((size_t)b * p.T + t0 + t) * p.H + h) * D, lane);
#pragma unroll
      for (int i = 0; i < DPL; ++i) qv[t][i] = qf.get(i) * p.scale_log2;
      qs[t] = p.qseg ? __ldg(p.qseg + (size_t)b * p.T + t0 + t) : 0;
    } else {
#pragma unroll
      for (int i = 0; i < DPL; ++i) qv[t][i] = 0.f;
      qs[t] = 0;
    }
  }

  const E* kbase = reinterpret_cast<const E*>(p.k) + (size_t)b * p.S * p.H * D + (size_t)h * D;
  const E* vbase = reinterpret_cast<const E*>(p.v) + (size_t)b * p.S * p.H * D + (size_t)h * D;
  const size_t rstride = (size_t)p.H * D;
  uint8_t* ring = dsm + warp * NST * C::STAGEB;

  // tile i of this warp: keys first + i * step .. +15
  const int step = WARPS * kTileKeys;
  const int first = lo + warp * kTileKeys;
  const int ntiles = first < hi ? (hi - first + step - 1) / step : 0;
  // this lane's 16-byte chunks of a tile: the same (row, column) in every tile
  const size_t rbytes = rstride * sizeof(E);
  uint32_t soff[C::CPL];
  size_t goff[C::CPL];
  int crow[C::CPL];
#pragma unroll
  for (int mm = 0; mm < C::CPL; ++mm) {
    const int c = lane + 32 * mm;
    crow[mm] = c / (C::ROWB / 16);
    const int col = c % (C::ROWB / 16);
    soff[mm] = crow[mm] * C::ROWB + col * 16;
    goff[mm] = (size_t)crow[mm] * rbytes + col * 16;
  }
  const uint32_t ring_s = smem_addr(ring);
  const uint8_t* kb8 = reinterpret_cast<const uint8_t*>(kbase);
  const uint8_t* vb8 = reinterpret_cast<const uint8_t*>(vbase);
  auto issue = [&](int i) {
    const int kb = first + i * step;
    const int nk = min(kTileKeys, hi - kb);
    const uint32_t kd = ring_s + (i % NST) * C::STAGEB;
    const size_t tb = (size_t)kb * rbytes;
    if (nk == kTileKeys) {
#pragma unroll
      for (int mm = 0; mm < C::CPL; ++mm) {
        cp_async16(kd + soff[mm], kb8 + tb + goff[mm], 16u);
        cp_async16(kd + C::TILEB + soff[mm], vb8 + tb + goff[mm], 16u);
      }
    } else {  // tail tile: rows past the range are zero-filled, not read
#pragma unroll
      for (int mm = 0; mm < C::CPL; ++mm) {
        const bool ok = crow[mm] < nk;
        const size_t g = ok ? tb + goff[mm] : tb;
        cp_async16(kd + soff[mm], kb8 + g, ok ? 16u : 0u);
        cp_async16(kd + C::TILEB + soff[mm], vb8 + g, ok ? 16u : 0u);
      }
    }
  };
#pragma unroll
  for (int i = 0; i < NST - 1; ++i) {
    if (i < ntiles) issue(i);
    cp_async_commit();
  }
  for (int i = 0; i < ntiles; ++i) {
    if (i + NST - 1 < ntiles) issue(i + NST - 1);
    cp_async_commit();
    if (i + NST < ntiles && lane < kTileKeys) {  // one tile beyond the ring: ask L2 for it
      const int key = first + (i + NST) * step + lane;
      if (key < hi) {
        prefetch_l2(kbase + (size_t)key * rstride, C::ROWB);
        prefetch_l2(vbase + (size_t)key * rstride, C::ROWB);
      }
    }
    cp_async_wait<NST - 1>();  // tile i has landed (this lane's copies) ...
    __syncwarp();               // ... and every lane's
    const int kb = first + i * step;
    const int nk = min(kTileKeys, hi - kb);
    const uint8_t* kt = ring + (i % NST) * C::STAGEB;
    const E* Ks = reinterpret_cast<const E*>(kt);
    const E* Vs = reinterpret_cast<const E*>(kt + C::TILEB);
    const int jk = lane & (kTileKeys - 1);  // lanes j, j + 8, j + 16, j + 24 end up with key j's score
    const int key = kb + jk;
    const int kseg = (p.kseg && jk < nk) ? __ldg(p.kseg + (size_t)b * p.S + key) : 0;
    float pr[TM];
#pragma unroll
    for (int t = 0; t < TM; ++t) {
      // this lane's share of the 8 dot products, then a butterfly over groups
      // of 8 lanes and two exchanges between the groups
      float v[kTileKeys];
#pragma unroll
      for (int j = 0; j < kTileKeys; ++j) {
        F kf;
        kf.load_shared(Ks + j * D, lane);
        float a = 0.f;
#pragma unroll
        for (int i2 = 0; i2 < DPL; ++i2) a = fmaf(qv[t][i2], kf.get(i2), a);
        v[j] = a;
      }
#pragma unroll
      for (int off = kTileKeys / 2, n = kTileKeys; off >= 1; off >>= 1, n >>= 1) {
        const bool up = lane & off;
#pragma unroll
        for (int i2 = 0; i2 < n / 2; ++i2) {
          const float send = up ? v[i2] : v[i2 + n / 2];
          const float keep = up ? v[i2 + n / 2] : v[i2];
          v[i2] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
      }
      float sc = v[0];
#pragma unroll
      for (int off = kTileKeys; off < 32; off <<= 1) sc += __shfl_xor_sync(0xffffffffu, sc, off);
      const bool vis = (t < nt) && (jk < nk) && (key < kmax[t]) && (qs[t] == kseg);
      const float s = vis ? sc : kNegInf;
      const float mn = fmaxf(m[t], warp_max(s));
      if (mn == kNegInf) {  // nothing visible yet for this token
        pr[t] = 0.f;
        continue;
      }
      const float corr = exp2f(m[t] - mn);  // m = -inf -> 0 (o, l are 0 then)
      pr[t] = vis ? exp2f(s - mn) : 0.f;
      l[t] = l[t] * corr + (lane < kTileKeys ? pr[t] : 0.f);
#pragma unroll
      for (int i2 = 0; i2 < DPL; ++i2) o[t][i2] *= corr;
      m[t] = mn;
    }
    // rows past the range are zero in the ring and their weights are zero
#pragma unroll
    for (int j = 0; j < kTileKeys; ++j) {
      F vf;
      vf.load_shared(Vs + j * D, lane);
#pragma unroll
      for (int t = 0; t < TM; ++t) {
        const float pj = __shfl_sync(0xffffffffu, pr[t], j);
#pragma unroll
        for (int i2 = 0; i2 < DPL; ++i2) o[t][i2] = fmaf(pj, vf.get(i2), o[t][i2]);
      }
    }
    __syncwarp();  // the stage is refilled by the next iteration's issue
  }
  cp_async_wait<0>();
  __syncthreads();

  // merge the warps' states into one partial (the ring is free now)
  float* s_m = reinterpret_cast<float*>(dsm);
  float* s_l = s_m + WARPS * TM;
  float* s_o = s_l + WARPS * TM;  // [WARPS][TM][D]
#pragma unroll
  for (int t = 0; t < TM; ++t) {
    const float lt = warp_sum(l[t]);
    if (lane == 0) {
      s_m[warp * TM + t] = m[t];
      s_l[warp * TM + t] = lt;
    }
#pragma unroll
    for (int i = 0; i < DPL; ++i) s_o[(warp * TM + t) * D + lane * DPL + i] = o[t][i];
  }
  __syncthreads();
  for (int e = threadIdx.x; e < nt * D; e += WARPS * 32) {
    const int t = e / D, d = e % D;
    float mx = kNegInf;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) mx = fmaxf(mx, s_m[w * TM + t]);
    float lsum = 0.f, osum = 0.f;
    if (mx != kNegInf) {
#pragma unroll
      for (int w = 0; w < WARPS; ++w) {
        const float f = exp2f(s_m[w * TM + t] - mx);
        lsum += s_l[w * TM + t] * f;
        osum += s_o[(w * TM + t) * D + d] * f;
      }
    }
    const size_t pi = (((size_t)b * p.H + h) * p.T + t0 + t) * p.P + item;
    p.part_o[pi * D + d] = osum;
    if (d == 0) p.part_ml[pi] = make_float2(mx, lsum);
  }
}

// ---------------------------------------------------------------------------
// 2. combine: grid (T, H, B), 8 warps; lane owns D/32 output dimensions
// ---------------------------------------------------------------------------
constexpr int kCombWarps = 8;

template <typename E, int D>
__global__ void __launch_bounds__(kCombWarps * 32) decode_combine_kernel(DecParams p) {
  constexpr int DPL = D / 32;
  const int t = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pos = __ldg(p.cache_idx + b) + t;
  const size_t base = (((size_t)b * p.H + h) * p.T + t) * p.P;
  // The lazy-softmax merge with the running max taken first: pass 1 finds the
  // largest partial max M, pass 2 walks the shards in ring order from the
  // token's home shard (warp w takes every 8th partial of that walk) and sums
  // o_p * 2^(m_p - M) and l_p * 2^(m_p - M); the terms are independent, so
  // their loads overlap.  The warps' sums are added at the end.
  __shared__ float s_red[kCombWarps];
  __shared__ float s_l[kCombWarps];
  __shared__ float s_o[kCombWarps][D];
  float m = kNegInf;
  for (int e = threadIdx.x; e < p.P; e += kCombWarps * 32) {
    const float2 ml = p.part_ml[base + e];
    if (ml.y > 0.f) m = fmaxf(m, ml.x);
  }
  m = warp_max(m);
  if (lane == 0) s_red[warp] = m;
  __syncthreads();
  m = s_red[0];
#pragma unroll
  for (int w = 1; w < kCombWarps; ++w) m = fmaxf(m, s_red[w]);
  float l = 0.f, o[DPL];
#pragma unroll
  for (int i = 0; i < DPL; ++i) o[i] = 0.f;
  if (m != kNegInf) {
    const int home = min(max(pos, 0), p.S - 1) / p.Ssh;
#pragma unroll 4
    for (int e = warp; e < p.P; e += kCombWarps) {
      const int i = e / p.items_per_shard, r = e % p.items_per_shard;
      const int k = ((home - i) % p.N + p.N) % p.N;  // ring order
      const size_t pi = base + (size_t)k * p.items_per_shard + r;
      const float2 ml = p.part_ml[pi];
      const float c = ml.y > 0.f ? exp2f(ml.x - m) : 0.f;
      const float* src = p.part_o + pi * D + lane * DPL;
      if constexpr (DPL == 4) {
        const float4 x = *reinterpret_cast<const float4*>(src);
        o[0] = fmaf(x.x, c, o[0]);
        o[1] = fmaf(x.y, c, o[1]);
        o[2] = fmaf(x.z, c, o[2]);
        o[3] = fmaf(x.w, c, o[3]);
      } else {
        const float2 x = *reinterpret_cast<const float2*>(src);
        o[0] = fmaf(x.x, c, o[0]);
        o[1] = fmaf(x.y, c, o[1]);
      }
      l = fmaf(ml.y, c, l);
    }
  }
  if (lane == 0) s_l[warp] = l;
#pragma unroll
  for (int i = 0; i < DPL; ++i) s_o[warp][lane * DPL + i] = o[i];
  __syncthreads();
  if (threadIdx.x < D) {
    const int d = threadIdx.x;
    float lt = 0.f, ot = 0.f;
#pragma unroll
    for (int w = 0; w < kCombWarps; ++w) {
      lt += s_l[w];
      ot += s_o[w][d];
    }
    const bool has = lt > 0.f;
    E* dst = reinterpret_cast<E*>(p.out) + (((size_t)b * p.T + t) * p.H + h) * D + d;
    if constexpr (sizeof(E) == 2) {
      *dst = __float2bfloat16_rn(has ? ot / lt : 0.f);
    } else {
      *dst = has ? ot / lt : 0.f;
    }
    if (d == 0) p.lse[((size_t)b * p.H + h) * p.T + t] = has ? (m + log2f(lt)) * 0.69314718055994531f : kNegInf;
  }
}

template <typename E, int D, int TM>
cudaError_t launch_partial(const DecParams& p, dim3 grid, const Ctx& c) {
  constexpr int smem = dec_smem_bytes<E, D, TM>();
  static std::atomic<bool> attr_set[256];  // the attribute is per kernel and device, and idempotent
  if (!attr_set[c.device]) {
    cudaError_t e = cudaFuncSetAttribute(decode_partial_kernel<E, D, TM>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set[c.device] = true;
  }
  decode_partial_kernel<E, D, TM><<<grid, DecShape<E, D>::WARPS * 32, smem, c.stream>>>(p);
  return cudaGetLastError();
}

template <typename E, int D>
cudaError_t launch_typed(const DecParams& p, const Ctx& c, uint64_t* launches) {
  const dim3 g1((unsigned)((long long)p.N * p.items_per_shard * p.H * p.tgroups), p.B);
  if (g1.x > 0) {
    cudaError_t e;
    if (p.T == 1) {
      e = launch_partial<E, D, 1>(p, g1, c);
    } else if (p.T == 2) {
      e = launch_partial<E, D, 2>(p, g1, c);
    } else if (p.T <= 4) {
      e = launch_partial<E, D, 4>(p, g1, c);
    } else {
      e = launch_partial<E, D, kTokGroup>(p, g1, c);
    }
    ++*launches;
    if (e != cudaSuccess) return e;
  }
  decode_combine_kernel<E, D><<<dim3(p.T, p.H, p.B), kCombWarps * 32, 0, c.stream>>>(p);
  ++*launches;
  return cudaGetLastError();
}

}  // namespace

DecodeSplit decode_split(int B, int T, int S, int H, int num_shards) {
  DecodeSplit s{};
  const int Ssh = num_shards > 0 ? S / num_shards : 0;
  const long long tg = (T + kTokGroup - 1) / kTokGroup;
  // the largest chunk that still gives >= 4096 CTAs (several waves on 152 SMs)
  int len = 128;
  for (int c : {2048, 1024, 512, 256}) {
    const long long items = (long long)B * H * tg * num_shards * ((Ssh + c - 1) / c);
    if (items >= 4096) {
      len = c;
      break;
    }
  }
  s.split_len = len;
  s.items_per_shard = Ssh > 0 ? (Ssh + len - 1) / len : 0;
  s.P = num_shards * s.items_per_shard;
  return s;
}

size_t decode_workspace_bytes(int B, int T, int S, int H, int D, int num_shards) {
  const DecodeSplit s = decode_split(B, T, S, H, num_shards);
  const size_t n = (size_t)B * H * T * s.P;
  const size_t o = (n * D * sizeof(float) + 255) & ~(size_t)255;
  return o + ((n * sizeof(float2) + 255) & ~(size_t)255);
}

cudaError_t launch_decode(const DecodeArgs& a, const Ctx& c, uint64_t* launches) {
  DecParams p{};
  p.B = a.B;
  p.T = a.T;
  p.S = a.S;
  p.H = a.H;
  p.D = a.D;
  p.N = a.N;
  p.Ssh = a.S / a.N;
  p.causal = a.causal;
  const DecodeSplit s = decode_split(a.B, a.T, a.S, a.H, a.N);
  p.split_len = s.split_len;
  p.items_per_shard = s.items_per_shard;
  p.P = s.P;
  p.tgroups = (a.T + kTokGroup - 1) / kTokGroup;
  p.q = a.q;
  p.k = a.k;
  p.v = a.v;
  p.cache_idx = a.cache_idx;
  p.qseg = a.qseg;
  p.kseg = a.kseg;
  const size_t n = (size_t)a.B * a.H * a.T * s.P;
  p.part_o = reinterpret_cast<float*>(a.workspace);
  p.part_ml = reinterpret_cast<float2*>(reinterpret_cast<char*>(a.workspace) +
                                        ((n * a.D * sizeof(float) + 255) & ~(size_t)255));
  p.out = a.out;
  p.lse = a.lse;
  p.scale_log2 = 1.4426950408889634f / sqrtf((float)a.D);
  if (a.bf16) {
    return a.D == 128 ? launch_typed<__nv_bfloat16, 128>(p, c, launches)
                      : launch_typed<__nv_bfloat16, 64>(p, c, launches);
  }
  return a.D == 128 ? launch_typed<float, 128>(p, c, launches) : launch_typed<float, 64>(p, c, launches);
}

}  // namespace ra
