// ffn_sm103.cu — the blockwise feed-forward network on sm_103a.
//
// FFN(x) = max(0, x W1 + b1) W2 + b2 ("Ring Attention with Blockwise
// Transformers for Near-Infinite Context", paper review page), evaluated
// block by block: the rows of the flattened (batch * sequence) axis are cut
// into chunks of `chunk_size`, each chunk goes through the network, and the
// results land in place ("Blockwise Feedforward网络详解RingAttention如何实现
// 内存高效的前向传播", §核心技术原理, §分块重组机制).  Only one chunk's hidden
// activation [chunk, F] exists at a time (the caller's workspace).
//
// Per chunk, two launches of one GEMM kernel with a fused epilogue:
//   H = relu(X_c W1^T + b1)      (w1 stored [F, Dm], as a linear layer stores it)
//   Y_c = H W2^T + b2            (w2 stored [Dm, F])
// GEMM kernel (persistent, one CTA per SM, 6 warps): 128 x 256 output tiles;
//   warp 4: TMA producer, 4-stage ring of A (128 x 64) and B (256 x 64) bf16
//           tiles with the 128-byte swizzle (K-major);
//   warp 5: tcgen05.mma issuer (M = 128, N = 256, K = 16 per instruction) into
//           one of two 256-column fp32 accumulators in tensor memory, so the
//           epilogue of one tile overlaps the MMAs of the next;
//   warps 0-3: epilogue, one output row per thread: tcgen05.ld, + bias,
//           optional ReLU, round to bf16, 16-byte stores.
// Every wait is bounded; on a timeout the kernel records the site in the
// status word, drains its copies and MMAs, frees tensor memory and returns.
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "ra_internal.h"
#include "sm103.cuh"

namespace ra {
namespace {

constexpr int kGM = 128, kGN = 256, kGK = 64, kGST = 4, kGAcc = 2;
constexpr int kGThreads = 192;
constexpr int kGProdWarp = 4, kGMmaWarp = 5;

struct GCfg {
  static constexpr uint32_t A_BYTES = kGM * kGK * 2;  // 16 KB
  static constexpr uint32_t B_BYTES = kGN * kGK * 2;  // 32 KB
  static constexpr uint32_t OFF_A = 0;
  static constexpr uint32_t OFF_B = OFF_A + kGST * A_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_B + kGST * B_BYTES;
  // full[kGST], empty[kGST], accfull[kGAcc], accempty[kGAcc], done
  static constexpr uint32_t NBAR = 2 * kGST + 2 * kGAcc + 1;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t SMEM = OFF_MISC + 64 + 1024;  // + slack to align the base to 1024 bytes
  static_assert(SMEM <= 232448, "shared memory layout exceeds the per-block limit");
};

struct GemmParams {
  int M, N, K;      // rows of this launch, output columns, reduction length
  int a_row0;       // first row of A inside its tensor map
  int tiles_m, tiles_n;
  int group_n;        // column tiles per raster group (see tile_coords)
  const float* bias;  // [N] or nullptr
  __nv_bfloat16* c;   // row-major, leading dimension ldc
  long long ldc;
  long long c_row0;   // output row of the launch's row 0
  int relu;
  int* status;
  uint64_t limit_ns;
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(map), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

// Tile t -> (first row, first column).  Tiles go in groups of group_n column
// tiles: inside a group the column tile varies fastest and the row tiles follow
// one another, so the group's columns of B (group_n x 256 rows of the weight
// matrix) stay in L2 while the rows of A stream through once per group, and the
// CTAs running at the same time share each A row tile.
__device__ __forceinline__ void tile_coords(const GemmParams& P, int t, int& m0, int& n0) {
  const int per_group = P.tiles_m * P.group_n;
  const int g = t / per_group, w = t - g * per_group;
  const int gn0 = g * P.group_n;
  const int gw = min(P.group_n, P.tiles_n - gn0);  // the last group may be narrower
  m0 = (w / gw) * kGM;
  n0 = (gn0 + w % gw) * kGN;
}

__global__ void __launch_bounds__(kGThreads, 1)
    gemm_bias_act_kernel(const __grid_constant__ CUtensorMap ma, const __grid_constant__ CUtensorMap mb,
                         const GemmParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(sm);
  const uint32_t bar0 = sbase + GCfg::OFF_BAR;
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (kGST + s); };
  auto accfull = [&](int a) { return bar0 + 8u * (2 * kGST + a); };
  auto accempty = [&](int a) { return bar0 + 8u * (2 * kGST + kGAcc + a); };
  const uint32_t done = bar0 + 8u * (2 * kGST + 2 * kGAcc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + GCfg::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + GCfg::OFF_MISC + 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < kGST; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int a = 0; a < kGAcc; ++a) {
      mbar_init(accfull(a), 1);
      mbar_init(accempty(a), 128);
    }
    mbar_init(done, 1);
    fence_mbar_init();
  }
  if (warp == kGMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  WaitCtl ctl{P.status, abort_flag, P.limit_ns};
  const int tiles = P.tiles_m * P.tiles_n;
  const int ksteps = (P.K + kGK - 1) / kGK;

  if (warp == kGProdWarp) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&ma);
      tma_prefetch_desc(&mb);
      int it = 0;
      bool alive = true;
      for (int t = blockIdx.x; t < tiles && alive; t += gridDim.x) {
        int m0, n0;
        tile_coords(P, t, m0, n0);
        for (int kb = 0; kb < ksteps; ++kb) {
          const int s = it % kGST;
          alive = mbar_wait(empty(s), ((it / kGST) & 1) ^ 1, ctl, 80);
          if (!alive) break;
          mbar_arrive_expect_tx(full(s), GCfg::A_BYTES + GCfg::B_BYTES);
          tma_load_2d(sbase + GCfg::OFF_A + s * GCfg::A_BYTES, &ma, full(s), kb * kGK, P.a_row0 + m0);
          tma_load_2d(sbase + GCfg::OFF_B + s * GCfg::B_BYTES, &mb, full(s), kb * kGK, n0);
          ++it;
        }
      }
      for (int s = 0; s < kGST; ++s) {  // let issued copies land (bounded, ignores abort)
        if (it <= s) continue;
        const int last = s + ((it - 1 - s) / kGST) * kGST;
        mbar_drain(full(s), (last / kGST) & 1, ctl, 81);
      }
    }
    __syncwarp();
  } else if (warp == kGMmaWarp) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kGM, kGN, 0, 0);
      const uint64_t da = sdesc_sw128(sbase + GCfg::OFF_A, 16, 1024);
      const uint64_t db = sdesc_sw128(sbase + GCfg::OFF_B, 16, 1024);
      int it = 0, ti = 0;
      bool alive = true;
      for (int t = blockIdx.x; t < tiles && alive; t += gridDim.x, ++ti) {
        const int a = ti & 1;
        alive = mbar_wait(accempty(a), ((ti >> 1) & 1) ^ 1, ctl, 82);
        if (!alive) break;
        tc_fence_after();
        const uint32_t dt = tbase + a * kGN;
        for (int kb = 0; kb < ksteps; ++kb) {
          const int s = it % kGST;
          alive = mbar_wait(full(s), (it / kGST) & 1, ctl, 83);
          if (!alive) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kGK / 16; ++kk)
            mma_ss(dt, sdesc_add(da, s * GCfg::A_BYTES + kk * 32), sdesc_add(db, s * GCfg::B_BYTES + kk * 32), idesc,
                   (kb > 0 || kk > 0) ? 1u : 0u);
          mma_commit(empty(s));
          ++it;
        }
        if (!alive) break;
        mma_commit(accfull(a));
      }
      // every MMA this thread issued has completed before tensor memory is freed
      mma_commit(done);
      mbar_drain(done, 0, ctl, 85);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ epilogue (warps 0-3)
    const int row = warp * 32 + lane;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    int ti = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++ti) {
      const int a = ti & 1;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(accfull(a), (ti >> 1) & 1, ctl, 84));
      if (!ok) break;
      tc_fence_after();
      int m0, n0;
      tile_coords(P, t, m0, n0);
      const bool row_ok = m0 + row < P.M;
      __nv_bfloat16* crow = P.c + (P.c_row0 + m0 + row) * P.ldc;
#pragma unroll 1
      for (int cq = 0; cq < kGN / 32; ++cq) {
        uint32_t v[32];
        tmem_ld32(tbase + lane_off + a * kGN + cq * 32, v);
        tmem_ld_wait(v);
        if (cq == kGN / 32 - 1) {  // the accumulator is free for the tile after next
          tc_fence_before();
          mbar_arrive(accempty(a));
        }
        const int nc = n0 + cq * 32;
        if (nc >= P.N) continue;
        float bias[32];
        if (P.bias && nc + 32 <= P.N) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 b4 = __ldg(reinterpret_cast<const float4*>(P.bias + nc) + q);
            bias[4 * q] = b4.x;
            bias[4 * q + 1] = b4.y;
            bias[4 * q + 2] = b4.z;
            bias[4 * q + 3] = b4.w;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) bias[j] = (P.bias && nc + j < P.N) ? __ldg(P.bias + nc + j) : 0.f;
        }
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float x0 = __uint_as_float(v[2 * j]) + bias[2 * j];
          float x1 = __uint_as_float(v[2 * j + 1]) + bias[2 * j + 1];
          if (P.relu) {
            x0 = fmaxf(x0, 0.f);
            x1 = fmaxf(x1, 0.f);
          }
          w[j] = pack_bf16x2(x0, x1);
        }
        if (row_ok) {
#pragma unroll
          for (int q = 0; q < 4; ++q)  // N is a multiple of 8: every 8-column group is whole or absent
            if (nc + 8 * q < P.N)
              *reinterpret_cast<uint4*>(crow + nc + 8 * q) = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kGMmaWarp) tmem_dealloc(tbase, 512);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_2d_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)f;
  }
  return fn;
}

// Row-major bf16 [rows, cols] with a 64-column x box_rows box, 128B swizzle;
// reads past the edges return zeros.
bool make_2d_map(CUtensorMap* m, const void* ptr, long long rows, long long cols, int box_rows) {
  auto enc = encode_2d_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

cudaError_t launch_gemm(const CUtensorMap& ma, const CUtensorMap& mb, GemmParams P, const Ctx& c,
                        uint64_t* launches) {
  static std::atomic<bool> attr_set[256];  // idempotent attribute; atomic so threads may race
  if (!attr_set[c.device]) {
    cudaError_t e =
        cudaFuncSetAttribute(gemm_bias_act_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)GCfg::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[c.device] = true;
  }
  P.tiles_m = (P.M + kGM - 1) / kGM;
  P.tiles_n = (P.N + kGN - 1) / kGN;
  {  // column tiles whose B rows (256 x K bf16 each) fit in 48 MB of L2 together
    const long long per = (long long)kGN * P.K * 2;
    P.group_n = (int)std::max(1LL, std::min((long long)P.tiles_n, (48LL << 20) / per));
  }
  P.status = c.status;
  P.limit_ns = c.limit_ns;
  const int tiles = P.tiles_m * P.tiles_n;
  const int grid = std::min(c.num_sms, tiles);
  gemm_bias_act_kernel<<<grid, kGThreads, GCfg::SMEM, c.stream>>>(ma, mb, P);
  *launches += 1;
  return cudaGetLastError();
}

}  // namespace

size_t ffn_workspace_bytes(long long rows, int chunk_size, int ffn_dim) {
  const long long r = std::min<long long>(rows, chunk_size);
  return (size_t)r * ffn_dim * sizeof(__nv_bfloat16);
}

cudaError_t launch_ffn(const FfnArgs& a, const Ctx& c, uint64_t* launches, const char** why) {
  const long long rows = (long long)a.B * a.L;
  const long long cap = std::min<long long>(rows, a.chunk);
  CUtensorMap mx, mw1, mh, mw2;
  if (!make_2d_map(&mx, a.x, rows, a.Dm, kGM) || !make_2d_map(&mw1, a.w1, a.F, a.Dm, kGN) ||
      !make_2d_map(&mh, a.hidden, cap, a.F, kGM) || !make_2d_map(&mw2, a.w2, a.Dm, a.F, kGN)) {
    *why = "cuTensorMapEncodeTiled failed (driver entry point unavailable or tensor rejected)";
    return cudaSuccess;
  }
  for (long long lo = 0; lo < rows; lo += a.chunk) {
    const int m = (int)std::min<long long>(a.chunk, rows - lo);
    GemmParams g1{};  // H = relu(X_c W1^T + b1)
    g1.M = m;
    g1.N = a.F;
    g1.K = a.Dm;
    g1.a_row0 = (int)lo;
    g1.bias = a.b1;
    g1.c = reinterpret_cast<__nv_bfloat16*>(a.hidden);
    g1.ldc = a.F;
    g1.c_row0 = 0;
    g1.relu = 1;
    cudaError_t e = launch_gemm(mx, mw1, g1, c, launches);
    if (e != cudaSuccess) return e;
    GemmParams g2{};  // Y_c = H W2^T + b2
    g2.M = m;
    g2.N = a.Dm;
    g2.K = a.F;
    g2.a_row0 = 0;
    g2.bias = a.b2;
    g2.c = reinterpret_cast<__nv_bfloat16*>(a.out);
    g2.ldc = a.Dm;
    g2.c_row0 = lo;
    g2.relu = 0;
    e = launch_gemm(mh, mw2, g2, c, launches);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace ra
