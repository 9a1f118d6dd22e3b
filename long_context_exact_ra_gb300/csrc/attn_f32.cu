// attn_f32.cu — exact fp32 path on the CUDA cores (FFMA, no tensor cores).
//
// Forward: one warp per query row, 8 rows (one shard) per block.  Each block
// walks the key/value shards in ring order k = (j - i) mod N ("Ring Attention
// with Blockwise Transformers for Near-Infinite Context", paper review page,
// 环形注意力算法), each shard in 32-key tiles staged in shared memory, and
// applies the lazy-softmax update of the code walk-through page
// (§2 数值稳定的注意力计算): running max, correction exp(m_old - m_new) on the
// numerator and denominator, then out = numerator / denominator.
//
// Backward: Delta_i = <dO_i, O_i>; dQ by query rows (ring order of the query's
// shard); dK, dV by key rows, visiting query shards j = k, k+1, ... (mod N),
// i.e. in the order the key block travels around the ring.  P is recomputed
// from the saved lse: P_ij = exp(S_ij - lse_i).
#include <cmath>
#include <cstdint>

#include "ra_internal.h"

namespace ra {
namespace {

constexpr int kRows = 8;   // warps (rows) per block
constexpr int kTile = 32;  // keys (or queries) per shared-memory tile

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ bool causal_ok(int qpos, int kpos, int c) {
  return c == 0 || (qpos / c) >= (kpos / c);
}

// Element (b, s, h, d) of a [B, S, H, D] tensor.
__device__ __forceinline__ size_t at(const Problem& p, int b, int s, int h) {
  return (((size_t)b * p.S + s) * p.H + h) * p.D;
}

template <int DMAX>
__global__ void __launch_bounds__(kRows * 32) fwd_f32_kernel(Problem p, const float* __restrict__ q,
                                                             const float* __restrict__ k,
                                                             const float* __restrict__ v,
                                                             float* __restrict__ out, float* __restrict__ lse) {
  constexpr int E = DMAX / 32;
  __shared__ float sK[kTile][DMAX + 1];
  __shared__ float sV[kTile][DMAX + 1];
  __shared__ float sQ[kRows][DMAX];
  __shared__ int sSegK[kTile];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int j = blockIdx.y;  // query shard
  const int b = blockIdx.z / p.H, h = blockIdx.z % p.H;
  const int row0 = j * p.Ssh + blockIdx.x * kRows;
  const int shard_end = (j + 1) * p.Ssh;
  const int qpos = row0 + warp;
  const bool valid = qpos < shard_end;
  const int last_row = min(row0 + kRows, shard_end) - 1;
  const float scale = 1.0f / sqrtf((float)p.D);
  for (int d = lane; d < DMAX; d += 32) sQ[warp][d] = (valid && d < p.D) ? q[at(p, b, qpos, h) + d] : 0.f;
  const int qseg = (p.seg && valid) ? p.seg[(size_t)b * p.S + qpos] : 0;
  float m = -INFINITY, l = 0.f;
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;

  for (int i = 0; i < p.N; ++i) {
    const int ks = ((j - i) % p.N + p.N) % p.N;  // ring order
    const int kbeg = ks * p.Ssh, kend = kbeg + p.Ssh;
    for (int t0 = kbeg; t0 < kend; t0 += kTile) {
      // block-uniform causal skip: no row of the block sees any key of the tile
      if (p.causal > 0 && (last_row / p.causal) < (t0 / p.causal)) continue;
      __syncthreads();
      for (int idx = threadIdx.x; idx < kTile * DMAX; idx += blockDim.x) {
        const int r = idx / DMAX, d = idx % DMAX;
        const int kp = t0 + r;
        const bool in = kp < kend && d < p.D;
        sK[r][d] = in ? k[at(p, b, kp, h) + d] : 0.f;
        sV[r][d] = in ? v[at(p, b, kp, h) + d] : 0.f;
      }
      if (threadIdx.x < kTile) {
        const int kp = t0 + threadIdx.x;
        sSegK[threadIdx.x] = (p.seg && kp < kend) ? p.seg[(size_t)b * p.S + kp] : 0;
      }
      __syncthreads();
      if (!valid) continue;
      const int kp = t0 + lane;
      const bool vis = kp < kend && causal_ok(qpos, kp, p.causal) && (!p.seg || sSegK[lane] == qseg);
      float s = -INFINITY;
      if (vis) {
        float dot = 0.f;
        for (int d = 0; d < p.D; ++d) dot = fmaf(sQ[warp][d], sK[lane][d], dot);
        s = dot * scale;
      }
      const float m_new = fmaxf(m, warp_max(s));
      if (m_new == -INFINITY) continue;  // nothing visible yet: numerator, denominator stay 0
      const float corr = expf(m - m_new);  // m = -inf -> 0 (numerator is 0 then)
      const float pj = vis ? expf(s - m_new) : 0.f;
      l = l * corr + warp_sum(pj);
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] *= corr;
      for (int jj = 0; jj < kTile; ++jj) {
        const float pjj = __shfl_sync(0xffffffffu, pj, jj);
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = fmaf(pjj, sV[jj][lane + 32 * e], acc[e]);
      }
      m = m_new;
    }
  }
  if (!valid) return;
  const float inv = l > 0.f ? 1.0f / l : 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int d = lane + 32 * e;
    if (d < p.D) out[at(p, b, qpos, h) + d] = acc[e] * inv;
  }
  if (lane == 0) lse[((size_t)b * p.H + h) * p.S + qpos] = l > 0.f ? m + logf(l) : -INFINITY;
}

// Delta_i = sum_d dO_id * O_id (one warp per row)
__global__ void delta_f32_kernel(Problem p, const float* __restrict__ out, const float* __restrict__ dout,
                                 float* __restrict__ delta) {
  const int row = blockIdx.x * kRows + threadIdx.x / 32, lane = threadIdx.x % 32;
  const int total = p.B * p.S * p.H;
  if (row >= total) return;
  const int h = row % p.H, s = (row / p.H) % p.S, b = row / (p.H * p.S);
  const size_t base = (size_t)row * p.D;
  float acc = 0.f;
  for (int d = lane; d < p.D; d += 32) acc = fmaf(dout[base + d], out[base + d], acc);
  acc = warp_sum(acc);
  if (lane == 0) delta[((size_t)b * p.H + h) * p.S + s] = acc;
}

// dQ_i = sum_j P_ij (dP_ij - Delta_i) K_j / sqrt(D),  P_ij = exp(S_ij - lse_i), dP_ij = <dO_i, V_j>
template <int DMAX>
__global__ void __launch_bounds__(kRows * 32) dq_f32_kernel(Problem p, const float* __restrict__ q,
                                                            const float* __restrict__ k,
                                                            const float* __restrict__ v,
                                                            const float* __restrict__ dout,
                                                            const float* __restrict__ lse,
                                                            const float* __restrict__ delta,
                                                            float* __restrict__ dq) {
  constexpr int E = DMAX / 32;
  __shared__ float sK[kTile][DMAX + 1];
  __shared__ float sV[kTile][DMAX + 1];
  __shared__ float sQ[kRows][DMAX];
  __shared__ float sdO[kRows][DMAX];
  __shared__ int sSegK[kTile];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int j = blockIdx.y;
  const int b = blockIdx.z / p.H, h = blockIdx.z % p.H;
  const int row0 = j * p.Ssh + blockIdx.x * kRows;
  const int shard_end = (j + 1) * p.Ssh;
  const int qpos = row0 + warp;
  const bool valid = qpos < shard_end;
  const int last_row = min(row0 + kRows, shard_end) - 1;
  const float scale = 1.0f / sqrtf((float)p.D);
  for (int d = lane; d < DMAX; d += 32) {
    sQ[warp][d] = (valid && d < p.D) ? q[at(p, b, qpos, h) + d] : 0.f;
    sdO[warp][d] = (valid && d < p.D) ? dout[at(p, b, qpos, h) + d] : 0.f;
  }
  const int qseg = (p.seg && valid) ? p.seg[(size_t)b * p.S + qpos] : 0;
  const float lse_i = valid ? lse[((size_t)b * p.H + h) * p.S + qpos] : 0.f;
  const float delta_i = valid ? delta[((size_t)b * p.H + h) * p.S + qpos] : 0.f;
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  for (int i = 0; i < p.N; ++i) {
    const int ks = ((j - i) % p.N + p.N) % p.N;
    const int kbeg = ks * p.Ssh, kend = kbeg + p.Ssh;
    for (int t0 = kbeg; t0 < kend; t0 += kTile) {
      if (p.causal > 0 && (last_row / p.causal) < (t0 / p.causal)) continue;
      __syncthreads();
      for (int idx = threadIdx.x; idx < kTile * DMAX; idx += blockDim.x) {
        const int r = idx / DMAX, d = idx % DMAX;
        const int kp = t0 + r;
        const bool in = kp < kend && d < p.D;
        sK[r][d] = in ? k[at(p, b, kp, h) + d] : 0.f;
        sV[r][d] = in ? v[at(p, b, kp, h) + d] : 0.f;
      }
      if (threadIdx.x < kTile) {
        const int kp = t0 + threadIdx.x;
        sSegK[threadIdx.x] = (p.seg && kp < kend) ? p.seg[(size_t)b * p.S + kp] : 0;
      }
      __syncthreads();
      if (!valid || lse_i == -INFINITY) continue;
      const int kp = t0 + lane;
      const bool vis = kp < kend && causal_ok(qpos, kp, p.causal) && (!p.seg || sSegK[lane] == qseg);
      float ds = 0.f;
      if (vis) {
        float dot = 0.f, dp = 0.f;
        for (int d = 0; d < p.D; ++d) {
          dot = fmaf(sQ[warp][d], sK[lane][d], dot);
          dp = fmaf(sdO[warp][d], sV[lane][d], dp);
        }
        const float pij = expf(dot * scale - lse_i);
        ds = pij * (dp - delta_i);
      }
      for (int jj = 0; jj < kTile; ++jj) {
        const float d_jj = __shfl_sync(0xffffffffu, ds, jj);
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = fmaf(d_jj, sK[jj][lane + 32 * e], acc[e]);
      }
    }
  }
  if (!valid) return;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int d = lane + 32 * e;
    if (d < p.D) dq[at(p, b, qpos, h) + d] = acc[e] * scale;
  }
}

// dV_j = sum_i P_ij dO_i ;  dK_j = sum_i P_ij (dP_ij - Delta_i) Q_i / sqrt(D)
template <int DMAX>
__global__ void __launch_bounds__(kRows * 32) dkdv_f32_kernel(Problem p, const float* __restrict__ q,
                                                              const float* __restrict__ k,
                                                              const float* __restrict__ v,
                                                              const float* __restrict__ dout,
                                                              const float* __restrict__ lse,
                                                              const float* __restrict__ delta,
                                                              float* __restrict__ dk, float* __restrict__ dv) {
  constexpr int E = DMAX / 32;
  __shared__ float sQ[kTile][DMAX + 1];
  __shared__ float sdO[kTile][DMAX + 1];
  __shared__ float sK[kRows][DMAX];
  __shared__ float sV[kRows][DMAX];
  __shared__ int sSegQ[kTile];
  __shared__ float sLse[kTile], sDelta[kTile];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int ksh = blockIdx.y;  // key shard
  const int b = blockIdx.z / p.H, h = blockIdx.z % p.H;
  const int row0 = ksh * p.Ssh + blockIdx.x * kRows;
  const int shard_end = (ksh + 1) * p.Ssh;
  const int kpos = row0 + warp;
  const bool valid = kpos < shard_end;
  const float scale = 1.0f / sqrtf((float)p.D);
  for (int d = lane; d < DMAX; d += 32) {
    sK[warp][d] = (valid && d < p.D) ? k[at(p, b, kpos, h) + d] : 0.f;
    sV[warp][d] = (valid && d < p.D) ? v[at(p, b, kpos, h) + d] : 0.f;
  }
  const int kseg = (p.seg && valid) ? p.seg[(size_t)b * p.S + kpos] : 0;
  float adk[E], adv[E];
#pragma unroll
  for (int e = 0; e < E; ++e) adk[e] = adv[e] = 0.f;
  for (int i = 0; i < p.N; ++i) {
    const int js = (ksh + i) % p.N;  // the ring device that holds this key block at step i
    const int qbeg = js * p.Ssh, qend = qbeg + p.Ssh;
    for (int t0 = qbeg; t0 < qend; t0 += kTile) {
      // block-uniform causal skip: the last query of the tile sees no key of the block
      const int tlast = min(t0 + kTile, qend) - 1;
      if (p.causal > 0 && (tlast / p.causal) < (row0 / p.causal)) continue;
      __syncthreads();
      for (int idx = threadIdx.x; idx < kTile * DMAX; idx += blockDim.x) {
        const int r = idx / DMAX, d = idx % DMAX;
        const int qp = t0 + r;
        const bool in = qp < qend && d < p.D;
        sQ[r][d] = in ? q[at(p, b, qp, h) + d] : 0.f;
        sdO[r][d] = in ? dout[at(p, b, qp, h) + d] : 0.f;
      }
      if (threadIdx.x < kTile) {
        const int qp = t0 + threadIdx.x;
        const bool in = qp < qend;
        sSegQ[threadIdx.x] = (p.seg && in) ? p.seg[(size_t)b * p.S + qp] : 0;
        sLse[threadIdx.x] = in ? lse[((size_t)b * p.H + h) * p.S + qp] : -INFINITY;
        sDelta[threadIdx.x] = in ? delta[((size_t)b * p.H + h) * p.S + qp] : 0.f;
      }
      __syncthreads();
      if (!valid) continue;
      const int qp = t0 + lane;
      const bool vis = qp < qend && sLse[lane] != -INFINITY && causal_ok(qp, kpos, p.causal) &&
                       (!p.seg || sSegQ[lane] == kseg);
      float pij = 0.f, ds = 0.f;
      if (vis) {
        float dot = 0.f, dp = 0.f;
        for (int d = 0; d < p.D; ++d) {
          dot = fmaf(sQ[lane][d], sK[warp][d], dot);
          dp = fmaf(sdO[lane][d], sV[warp][d], dp);
        }
        pij = expf(dot * scale - sLse[lane]);
        ds = pij * (dp - sDelta[lane]);
      }
      for (int ii = 0; ii < kTile; ++ii) {
        const float p_ii = __shfl_sync(0xffffffffu, pij, ii);
        const float ds_ii = __shfl_sync(0xffffffffu, ds, ii);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          adv[e] = fmaf(p_ii, sdO[ii][lane + 32 * e], adv[e]);
          adk[e] = fmaf(ds_ii, sQ[ii][lane + 32 * e], adk[e]);
        }
      }
    }
  }
  if (!valid) return;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int d = lane + 32 * e;
    if (d < p.D) {
      dk[at(p, b, kpos, h) + d] = adk[e] * scale;
      dv[at(p, b, kpos, h) + d] = adv[e];
    }
  }
}

dim3 shard_grid(const Problem& p) {
  return dim3((unsigned)((p.Ssh + kRows - 1) / kRows), (unsigned)p.N, (unsigned)(p.B * p.H));
}

}  // namespace

cudaError_t launch_fwd_f32(const FwdArgs& a, const Ctx& c, uint64_t* launches) {
  const Problem& p = a.p;
  const dim3 grid = shard_grid(p);
  auto q = (const float*)a.q;
  auto k = (const float*)a.k;
  auto v = (const float*)a.v;
  auto o = (float*)a.out;
  if (p.D <= 32)
    fwd_f32_kernel<32><<<grid, kRows * 32, 0, c.stream>>>(p, q, k, v, o, a.lse);
  else if (p.D <= 64)
    fwd_f32_kernel<64><<<grid, kRows * 32, 0, c.stream>>>(p, q, k, v, o, a.lse);
  else
    fwd_f32_kernel<128><<<grid, kRows * 32, 0, c.stream>>>(p, q, k, v, o, a.lse);
  *launches += 1;
  return cudaGetLastError();
}

cudaError_t launch_bwd_f32(const BwdArgs& a, const Ctx& c, uint64_t* launches) {
  const Problem& p = a.p;
  auto q = (const float*)a.q;
  auto k = (const float*)a.k;
  auto v = (const float*)a.v;
  auto o = (const float*)a.out;
  auto dO = (const float*)a.dout;
  const int rows = p.B * p.S * p.H;
  delta_f32_kernel<<<(rows + kRows - 1) / kRows, kRows * 32, 0, c.stream>>>(p, o, dO, a.delta);
  cudaError_t e = cudaGetLastError();
  *launches += 1;
  if (e != cudaSuccess) return e;
  const dim3 grid = shard_grid(p);
#define RA_F32_BWD(DM)                                                                                  \
  dq_f32_kernel<DM><<<grid, kRows * 32, 0, c.stream>>>(p, q, k, v, dO, a.lse, a.delta, (float*)a.dq);    \
  dkdv_f32_kernel<DM><<<grid, kRows * 32, 0, c.stream>>>(p, q, k, v, dO, a.lse, a.delta, (float*)a.dk, \
                                                         (float*)a.dv);
  if (p.D <= 32) {
    RA_F32_BWD(32)
  } else if (p.D <= 64) {
    RA_F32_BWD(64)
  } else {
    RA_F32_BWD(128)
  }
#undef RA_F32_BWD
  *launches += 2;
  return cudaGetLastError();
}

}  // namespace ra
