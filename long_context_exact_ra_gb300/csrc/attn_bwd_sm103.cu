// attn_bwd_sm103.cu — bf16 backward of blockwise ring attention on sm_103a.
//
// Gradients of L = sum(dO * out) for out = softmax(Q K^T / sqrt(d)) V with the
// causal / segment masks of the forward, recomputing P from the saved lse
// (no S x S matrix is kept; the code walk-through page of Ring Attention,
// "从论文到代码：深入理解RingAttention的块注意力计算逻辑", names the backward
// among the implementation's parts and recommends recomputation over saving
// intermediates, §性能优化技巧 2):
//   P = exp(S - lse),  Delta_i = <dO_i, O_i>,  dV = P^T dO,
//   dS = P * (dO V^T - Delta),  dK = dS^T Q / sqrt(d),  dQ = dS K / sqrt(d).
//
// Three launches:
//   1. preprocess: Delta = rowsum(dO * O) next to lse * log2(e); zero the fp32 dQ
//      accumulator and the main kernel's unit counter
//   2. main (persistent, one CTA per SM, 10 warps): one unit = one 128-key
//      K/V tile of one (batch, head); CTAs draw units from the counter as they
//      free up.  The unit visits the query tiles in the
//      order the key block travels around the ring: query shards j = k, k+1,
//      ... (mod N) ("Ring Attention with Blockwise Transformers for
//      Near-Infinite Context", paper review page, 环形注意力算法), skipping
//      tiles with no visible element.  Per (key tile, query tile) pair:
//        dP^T = V dO^T, S^T = K Q^T          (tcgen05 SS, fp32 in TMEM)
//        P^T, dS^T by two warpgroups (64 query columns each, one key row per thread)
//        dV += P^T dO, dK += dS^T Q          (tcgen05 TS: P^T / dS^T read from TMEM)
//        dQ^T = K^T dS^T                     (tcgen05 SS: dS^T in smem as an MN-major B)
//      and the same two warpgroups add the dQ tile into the fp32 accumulator.
//   3. finalize: dq = bf16(dQ_accum / sqrt(d)).
// Tensor memory (512 columns): A | B | dK | dV with A = S^T, later P^T, later
// dQ_tile; B = dP^T, later dS^T.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <algorithm>
#include <cudaTypedefs.h>

#include "ra_internal.h"
#include "sm103.cuh"

namespace ra {

bool make_tile_map(CUtensorMap* m, const void* ptr, const Problem& p, int rows);

namespace {

constexpr int kT = 128;  // keys per unit tile, queries per pair tile
constexpr int kNInfo = 8;
constexpr int kThreads = 320;
constexpr int kProdWarp = 8;
constexpr int kMmaWarp = 9;

enum : int { kRecPair = 0, kRecUnitEnd = 1, kRecStop = 2 };
enum : int { kMasked = 1 };

struct __align__(16) BRec {
  int kind;
  int flags;
  int q0;      // first query row of the tile (global)
  int qvalid;  // query rows of the tile inside their shard
  int b, h;
  int k0;      // first key of the unit tile (global)
  int kvalid;  // keys of the unit tile inside their shard
};

template <int D>
struct BCfg {
  static constexpr uint32_t TB = kT * D * 2;  // bytes of one [128 x D] bf16 tile
  static constexpr int QST = 2;               // Q / dO stages
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = OFF_K + TB;
  static constexpr uint32_t OFF_Q = OFF_V + TB;               // QST stages
  static constexpr uint32_t OFF_DO = OFF_Q + QST * TB;        // QST stages
  static constexpr uint32_t OFF_DS = OFF_DO + QST * TB;       // dS^T, 128 x 128 bf16
  static constexpr uint32_t OFF_VEC = OFF_DS + kT * kT * 2;   // per stage: 130 (lse2, delta) pairs
  static constexpr uint32_t VEC_BYTES = kBwdVecEntries * 8;
  static constexpr uint32_t OFF_REC = OFF_VEC + QST * VEC_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_REC + kNInfo * sizeof(BRec);
  // kvfull, kvempty, qfull[2], qempty[2], infofull[8], infoempty[8], spfull, pready,
  // dqfull, dqfree, accdone, accfree
  static constexpr int NBAR = 2 + 2 * QST + 2 * kNInfo + 6;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  // No alignment slack (the D = 128 layout is within a few hundred bytes of the
  // 227 KB limit): the kernel checks that the dynamic base is 1024-byte aligned.
  static constexpr uint32_t SMEM = OFF_MISC + 64;
  static_assert(SMEM <= 232448, "shared memory layout exceeds the per-block limit");
  static constexpr uint32_t TA = 0, TBc = 128, TDK = 256, TDV = 256 + D;  // TMEM columns
};

struct BBars {
  uint32_t base;
  __device__ uint32_t kvfull() const { return base; }
  __device__ uint32_t kvempty() const { return base + 8; }
  __device__ uint32_t qfull(int s) const { return base + 16 + 8 * s; }
  __device__ uint32_t qempty(int s) const { return base + 32 + 8 * s; }
  __device__ uint32_t infofull(int i) const { return base + 48 + 8 * i; }
  __device__ uint32_t infoempty(int i) const { return base + 48 + 8 * (kNInfo + i); }
  __device__ uint32_t spfull() const { return base + 48 + 16 * kNInfo; }
  __device__ uint32_t pready() const { return base + 56 + 16 * kNInfo; }
  __device__ uint32_t dqfull() const { return base + 64 + 16 * kNInfo; }
  __device__ uint32_t dqfree() const { return base + 72 + 16 * kNInfo; }
  __device__ uint32_t accdone() const { return base + 80 + 16 * kNInfo; }
  __device__ uint32_t accfree() const { return base + 88 + 16 * kNInfo; }
};

struct BwdParams {
  Problem p;
  const float2* ld2;  // (lse * log2(e), Delta) per (b, h, s), row pitch Sp
  int Sp;
  float* dq_accum;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int* status;
  uint64_t limit_ns;
  int tiles_per_shard;
  int num_units;
  float scale;       // 1 / sqrt(D)
  float scale_log2;  // log2(e) / sqrt(D)
  int* unit_counter; // zeroed by the preprocess kernel: CTAs draw tickets as they free up
  int group_heads;   // (b, h) heads per ticket group (their Q, dO, dQ accumulator fit in part of L2)
  // Positions and key segment ids: query row r sits at position r + qoff, key row
  // x at x + koff (0 and 0 for one sequence cut into virtual shards); kseg holds
  // the key rows' segment ids (p.seg for one sequence).
  int qoff, koff;
  const int32_t* kseg;
  // Ring-step carries (kCarry kernels only): fp32 dK, dV [B, S, H, D] that this
  // call's key-block gradients are added to.
  float* dk_carry;
  float* dv_carry;
  int* vlog;     // visit log (see visit_log), or null
  int vlog_cap;
};

__device__ __forceinline__ bool mbar_poll(uint32_t bar, uint32_t parity) {  // non-suspending test
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void red_add_v2(float* addr, float a, float b) {
  asm volatile("red.global.add.v2.f32 [%0], {%1, %2};" ::"l"(addr), "f"(a), "f"(b) : "memory");
}
__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

// ---------------------------------------------------------------------------
// 1. preprocess: Delta_i = sum_d dO_id O_id (bf16 inputs, fp32) stored next to
//    lse_i * log2(e), and the dQ accumulator zeroed
// ---------------------------------------------------------------------------
__global__ void bwd_pre_kernel(Problem p, const __nv_bfloat16* __restrict__ out,
                               const __nv_bfloat16* __restrict__ dout, const float* __restrict__ lse,
                               float2* __restrict__ ld2, int Sp, float* __restrict__ dq_accum,
                               int* __restrict__ unit_counter) {
  if (blockIdx.x == 0 && threadIdx.x == 0) *unit_counter = 0;
  const int warps = blockDim.x / 32;
  const long long row = (long long)blockIdx.x * warps + threadIdx.x / 32;  // (b, s, h) row
  const int lane = threadIdx.x & 31;
  const long long total = (long long)p.B * p.S * p.H;
  if (row >= total) return;
  const int h = (int)(row % p.H), s = (int)((row / p.H) % p.S), b = (int)(row / ((long long)p.H * p.S));
  const size_t base = (size_t)row * p.D;
  float acc = 0.f;
  for (int d = lane * 4; d < p.D; d += 128) {
    const uint2 o = *reinterpret_cast<const uint2*>(out + base + d);
    const uint2 g = *reinterpret_cast<const uint2*>(dout + base + d);
    const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&o);
    const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&g);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float2 of = __bfloat1622float2(o2[i]);
      const float2 gf = __bfloat1622float2(g2[i]);
      acc = fmaf(of.x, gf.x, acc);
      acc = fmaf(of.y, gf.y, acc);
    }
    *reinterpret_cast<float4*>(dq_accum + base + d) = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) {
    const size_t bh = (size_t)b * p.H + h;
    ld2[bh * Sp + s] = make_float2(lse[bh * p.S + s] * 1.4426950408889634f, acc);
  }
}

// ---------------------------------------------------------------------------
// 3. finalize: dq = bf16(dq_accum * scale)
// ---------------------------------------------------------------------------
__global__ void bwd_fin_kernel(size_t n4, const float4* __restrict__ acc, uint2* __restrict__ dq, float scale) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
    const float4 a = acc[i];
    uint2 o;
    o.x = pack_bf16x2(a.x * scale, a.y * scale);
    o.y = pack_bf16x2(a.z * scale, a.w * scale);
    dq[i] = o;
  }
}

// Unit u -> (b, h, key shard k, tile t).  Units are numbered head-major, and
// within a head by increasing key position (rank 0 = longest causal work); the
// order in which CTAs take them is set by bticket_unit.
__device__ __forceinline__ void bunit_coords(const BwdParams& P, int u, int& b, int& h, int& k, int& t) {
  const int per_head = P.p.N * P.tiles_per_shard;
  const int bh = u / per_head, rank = u % per_head;
  k = rank / P.tiles_per_shard;
  t = rank % P.tiles_per_shard;
  b = bh / P.p.H;
  h = bh % P.p.H;
}

// Ticket t -> unit.  The (b, h) heads form groups of group_heads whose Q, dO and
// dQ accumulator fit in L2 together; a group's tickets go rank-major (key tile 0
// of every head of the group, the longest causal work, then key tile 1, ...), so
// the last tickets of a group are its shortest units and the CTAs finish together.
__device__ __forceinline__ int bticket_unit(const BwdParams& P, int t) {
  const int per_head = P.p.N * P.tiles_per_shard;
  const int bh_total = P.p.B * P.p.H;
  const int G = P.group_heads;
  const int g = t / (G * per_head);
  const int g0 = g * G;
  const int gh = min(G, bh_total - g0);
  const int w = t - g * G * per_head;
  const int rank = w / gh;
  return (g0 + (w - rank * gh)) * per_head + rank;
}

// ---------------------------------------------------------------------------
// 2. main kernel
// ---------------------------------------------------------------------------
template <int D, bool kCarry, bool kLog>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_bf16_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                    const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
                    const BwdParams P) {
  using C = BCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if ((smem_u32(smem_raw) & 1023u) != 0) {  // swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) atomicCAS(P.status, 0, kDevBadSmem);
    return;
  }
  uint8_t* sm = smem_raw;
  const uint32_t sbase = smem_u32(sm);
  BRec* recs = reinterpret_cast<BRec*>(sm + C::OFF_REC);
  BBars bars{sbase + C::OFF_BAR};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::OFF_MISC + 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Problem& pb = P.p;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bars.kvfull(), 1);
    mbar_init(bars.kvempty(), 1);
    for (int s = 0; s < C::QST; ++s) {
      mbar_init(bars.qfull(s), 1);
      mbar_init(bars.qempty(s), 1);
    }
    for (int i = 0; i < kNInfo; ++i) {
      mbar_init(bars.infofull(i), 1);
      mbar_init(bars.infoempty(i), 1 + 8);  // MMA thread + one lane per P/dS warp
    }
    mbar_init(bars.spfull(), 1);
    mbar_init(bars.pready(), 256);
    mbar_init(bars.dqfull(), 1);
    mbar_init(bars.dqfree(), 256);
    mbar_init(bars.accdone(), 1);
    mbar_init(bars.accfree(), 256);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  WaitCtl ctl{P.status, abort_flag, P.limit_ns};

  if (warp == kProdWarp) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&mq);
      tma_prefetch_desc(&mk);
      tma_prefetch_desc(&mv);
      tma_prefetch_desc(&mdo);
    }
    int rec_n = 0, pair_n = 0, unit_n = 0, kv_loads = 0;
    bool alive = true;
    const int c = pb.causal;
    const int qo = kCarry ? P.qoff : 0, ko = kCarry ? P.koff : 0;
    auto publish = [&](const BRec& r) -> bool {
      const int slot = rec_n % kNInfo;
      if (!mbar_wait(bars.infoempty(slot), ((rec_n / kNInfo) & 1) ^ 1, ctl, 40)) return false;
      recs[slot] = r;
      mbar_arrive(bars.infofull(slot));
      ++rec_n;
      return true;
    };
    // CTAs draw tickets (bticket_unit: L2-sized head groups, longest units first)
    // as they become free, so uneven unit costs even out and all CTAs move through
    // one group of heads together; the next ticket is drawn one unit ahead so its
    // latency hides behind the current unit.
    auto ticket = [&]() -> int {  // lane 0 draws, the warp gets the unit (or -1)
      int tk = 0;
      if (lane == 0) tk = atomicAdd(P.unit_counter, 1);
      tk = __shfl_sync(0xffffffffu, tk, 0);
      return tk < P.num_units ? bticket_unit(P, tk) : -1;
    };
    int u = ticket();
    while (u >= 0 && alive) {
      int ahead = 0;
      if (lane == 0) ahead = atomicAdd(P.unit_counter, 1);
      int b, h, k, t;
      bunit_coords(P, u, b, h, k, t);
      const int k0 = k * pb.Ssh + t * kT;
      const int kvalid = min(kT, (k + 1) * pb.Ssh - k0);
      const int klast = k0 + kvalid - 1;
      int kmn = 0, kmx = 0;
      if (pb.seg) {
        int mn = INT_MAX, mx = INT_MIN;
        for (int r = lane; r < kvalid; r += 32) {
          const int sv = __ldg((kCarry ? P.kseg : pb.seg) + (size_t)b * pb.S + k0 + r);
          mn = min(mn, sv);
          mx = max(mx, sv);
        }
        for (int o = 16; o > 0; o >>= 1) {
          mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
          mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        }
        kmn = mn;
        kmx = mx;
      }
      if (lane == 0) {
        alive = mbar_wait(bars.kvempty(), (unit_n & 1) ^ 1, ctl, 41);
        if (alive) {
          ++kv_loads;
          mbar_arrive_expect_tx(bars.kvfull(), 2 * C::TB);
          for (int cb = 0; cb < D / 64; ++cb) {
            tma_load_4d(sbase + C::OFF_K + cb * 16384, &mk, bars.kvfull(), cb * 64, h, k0, b);
            tma_load_4d(sbase + C::OFF_V + cb * 16384, &mv, bars.kvfull(), cb * 64, h, k0, b);
          }
        }
      }
      alive = __shfl_sync(0xffffffffu, alive, 0);
      for (int i = 0; i < pb.N && alive; ++i) {
        const int js = (k + i) % pb.N;  // the ring device holding this key block at step i
        const int qbeg = js * pb.Ssh, qend = qbeg + pb.Ssh;
        if (c > 0 && (qend - 1 + qo) / c < (k0 + ko) / c) continue;  // every query of the shard precedes the keys
        for (int t0 = 0; t0 < P.tiles_per_shard && alive; t0 += 32) {
          int qmn = 0, qmx = 0;
          const int my_t = t0 + lane;
          if (pb.seg && my_t < P.tiles_per_shard) {
            const int qa = qbeg + my_t * kT;
            const int qb = min(qend, qa + kT);
            int mn = INT_MAX, mx = INT_MIN;
            if (!(c > 0 && (qb - 1 + qo) / c < (k0 + ko) / c)) {
              const int* sp = pb.seg + (size_t)b * pb.S;
              for (int x = qa; x < qb; ++x) {
                const int sv = __ldg(sp + x);
                mn = min(mn, sv);
                mx = max(mx, sv);
              }
            }
            qmn = mn;
            qmx = mx;
          }
          const int tend = min(32, P.tiles_per_shard - t0);
          for (int tt = 0; tt < tend && alive; ++tt) {
            const int qa = qbeg + (t0 + tt) * kT;
            const int qvalid = min(kT, qend - qa);
            const int ql = qa + qvalid - 1;
            const int tmn = __shfl_sync(0xffffffffu, qmn, tt);
            const int tmx = __shfl_sync(0xffffffffu, qmx, tt);
            bool skip = false, full = true;
            if (c > 0) {
              if ((ql + qo) / c < (k0 + ko) / c) skip = true;
              else if (!((qa + qo) / c >= (klast + ko) / c)) full = false;
            }
            if (!skip && pb.seg) {
              if (tmx < kmn || tmn > kmx) skip = true;
              else if (!(kmn == kmx && tmn == kmx && tmx == kmx)) full = false;
            }
            if (qvalid < kT || kvalid < kT) full = false;
            if (skip) continue;
            // stage s: Q and dO tiles (TMA) and the (lse2, delta) pairs of the tile (bulk copy)
            const int s = pair_n % C::QST;
            const uint32_t par = ((pair_n / C::QST) & 1) ^ 1;
            if (lane == 0) alive = mbar_wait(bars.qempty(s), par, ctl, 42);
            alive = __shfl_sync(0xffffffffu, alive, 0);
            if (!alive) break;
            if (lane == 0) {
              mbar_arrive_expect_tx(bars.qfull(s), 2 * C::TB + C::VEC_BYTES);
              for (int cb = 0; cb < D / 64; ++cb) {
                tma_load_4d(sbase + C::OFF_Q + s * C::TB + cb * 16384, &mq, bars.qfull(s), cb * 64, h, qa, b);
                tma_load_4d(sbase + C::OFF_DO + s * C::TB + cb * 16384, &mdo, bars.qfull(s), cb * 64, h, qa, b);
              }
              bulk_g2s(sbase + C::OFF_VEC + s * C::VEC_BYTES, P.ld2 + ((size_t)b * pb.H + h) * P.Sp + (qa & ~1),
                       C::VEC_BYTES, bars.qfull(s));
              BRec r;
              r.kind = kRecPair;
              r.flags = full ? 0 : kMasked;
              r.q0 = qa;
              r.qvalid = qvalid;
              r.b = b;
              r.h = h;
              r.k0 = k0;
              r.kvalid = kvalid;
              alive = publish(r);
              if constexpr (kLog) visit_log(P.vlog, P.vlog_cap, 1, b, h, k, t, i, js, t0 + tt);
            }
            alive = __shfl_sync(0xffffffffu, alive, 0);
            ++pair_n;
          }
        }
      }
      if (lane == 0 && alive) {
        BRec r;
        r.kind = kRecUnitEnd;
        r.flags = 0;
        r.q0 = 0;
        r.qvalid = 0;
        r.b = b;
        r.h = h;
        r.k0 = k0;
        r.kvalid = kvalid;
        alive = publish(r);
      }
      alive = __shfl_sync(0xffffffffu, alive, 0);
      ++unit_n;
      const int tk = __shfl_sync(0xffffffffu, ahead, 0);
      u = tk < P.num_units ? bticket_unit(P, tk) : -1;
    }
    if (lane == 0 && alive) {
      BRec r;
      r.kind = kRecStop;
      publish(r);
    }
    if (lane == 0) {  // let issued copies land (bounded, ignores abort)
      for (int s = 0; s < C::QST; ++s) {
        if (pair_n <= s) continue;
        const int last = s + ((pair_n - 1 - s) / C::QST) * C::QST;
        mbar_drain(bars.qfull(s), (last / C::QST) & 1, ctl, 43);
      }
      if (kv_loads > 0) mbar_drain(bars.kvfull(), (kv_loads - 1) & 1, ctl, 44);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idSP = idesc_bf16_f32(kT, kT, 0, 0);  // S^T, dP^T: K-major A and B
      constexpr uint32_t idKV = idesc_bf16_f32(kT, D, 0, 1);   // dV, dK: A in TMEM, B MN-major
      // dQ^T (D = 128): A = K^T, B = dS^T; dQ (D = 64): A = dS, B = K; all MN-major
      constexpr uint32_t idQ = idesc_bf16_f32(D == 128 ? D : kT, D == 128 ? kT : D, 1, 1);
      int rec_n = 0, pair_n = 0, unit_n = 0, dq_n = 0, unit_pairs = 0;
      uint32_t pready_ph = 0;
      bool alive = true, in_unit = false;
      const uint32_t tA = tbase + C::TA, tB = tbase + C::TBc;
      // Shared-memory descriptors built once; each MMA adds a compile-time byte offset.
      const uint64_t kdK = sdesc_sw128(sbase + C::OFF_K, 16, 1024);     // K, K-major
      const uint64_t kdV = sdesc_sw128(sbase + C::OFF_V, 16, 1024);     // V, K-major
      const uint64_t kdQ = sdesc_sw128(sbase + C::OFF_Q, 16, 1024);     // Q stage 0, K-major
      const uint64_t kdO = sdesc_sw128(sbase + C::OFF_DO, 16, 1024);    // dO stage 0, K-major
      const uint64_t mdK = sdesc_sw128(sbase + C::OFF_K, 16384, 1024);  // K, MN-major
      const uint64_t mdQ = sdesc_sw128(sbase + C::OFF_Q, 16384, 1024);  // Q stage 0, MN-major
      const uint64_t mdO = sdesc_sw128(sbase + C::OFF_DO, 16384, 1024); // dO stage 0, MN-major
      const uint64_t mdS = sdesc_sw128(sbase + C::OFF_DS, 16384, 1024); // dS^T, MN-major
      // This thread needs only each record's kind.  It reads the next record while
      // the P/dS warpgroups work on the current pair (and frees its slot at once),
      // so that the next pair's MMAs follow the current pair's without a gap.
      auto fetch_kind = [&](int& kind) -> bool {
        const int slot = rec_n % kNInfo;
        if (!mbar_wait(bars.infofull(slot), (rec_n / kNInfo) & 1, ctl, 50)) return false;
        kind = recs[slot].kind;
        mbar_arrive(bars.infoempty(slot));
        ++rec_n;
        return true;
      };
      int kind = kRecStop;
      alive = fetch_kind(kind);
      while (alive) {
        if (kind == kRecStop) break;
        if (!in_unit) {  // first record of a unit: its K/V tiles must be resident
          if (!mbar_wait(bars.kvfull(), unit_n & 1, ctl, 51)) break;
          in_unit = true;
          unit_pairs = 0;
        }
        if (kind == kRecUnitEnd) {
          mma_commit(bars.accdone());
          mma_commit(bars.kvempty());
          ++unit_n;
          in_unit = false;
          alive = fetch_kind(kind);
          continue;
        }
        const bool first = unit_pairs == 0;
        const int s = pair_n % C::QST;
        if (!mbar_wait(bars.qfull(s), (pair_n / C::QST) & 1, ctl, 52)) break;
        tc_fence_after();
        // dP^T = V dO^T into B (B was last read by the previous pair's dK MMA: in order)
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss(tB, sdesc_add(kdV, off), sdesc_add(kdO, s * C::TB + off), idSP, kk > 0);
        }
        // S^T = K Q^T into A, once the previous dQ tile has been read out of A
        if (dq_n > 0 && !mbar_wait(bars.dqfree(), (dq_n - 1) & 1, ctl, 53)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss(tA, sdesc_add(kdK, off), sdesc_add(kdQ, s * C::TB + off), idSP, kk > 0);
        }
        mma_commit(bars.spfull());
        // the record after this pair (a pair or the unit's end: the producer
        // publishes either without waiting for this pair)
        int next_kind = kRecStop;
        if (!fetch_kind(next_kind)) break;
        // wait for P^T, dS^T (TMEM) and dS^T (smem)
        {  // spin (no suspend) for up to 4096 polls, then the bounded wait
          bool got = false;
          for (int n = 0; n < 4096 && !got; ++n) got = mbar_poll(bars.pready(), pready_ph);
          if (!got && !mbar_wait(bars.pready(), pready_ph, ctl, 54)) break;
        }
        pready_ph ^= 1;
        // the previous unit's dK / dV must have been read out before they are overwritten
        if (first && unit_n > 0 && !mbar_wait(bars.accfree(), (unit_n - 1) & 1, ctl, 55)) break;
        tc_fence_after();
        // dQ tile into A (S^T there has been consumed by the softmax warpgroups)
        if constexpr (D == 128) {
          // dQ^T = K^T dS^T: TMEM lanes = head dim, columns = queries
#pragma unroll
          for (int kk = 0; kk < kT / 16; ++kk)
            mma_ss(tA, sdesc_add(mdK, kk * 2048), sdesc_add(mdS, kk * 2048), idQ,
                   kk > 0);
        } else {
          // dQ = dS K: TMEM lanes = queries, columns = head dim
#pragma unroll
          for (int kk = 0; kk < kT / 16; ++kk)
            mma_ss(tA, sdesc_add(mdS, kk * 2048), sdesc_add(mdK, kk * 2048), idQ,
                   kk > 0);
        }
        mma_commit(bars.dqfull());
        // dV += P^T dO ; dK += dS^T Q.  In B the 16 columns of query group kk hold
        // dS^T (8 columns of bf16 pairs) then P^T (8 columns).
#pragma unroll
        for (int kk = 0; kk < kT / 16; ++kk) {
          const uint32_t col = kk * 16 + 8;
          mma_ts(tbase + C::TDV, tB + col, sdesc_add(mdO, s * C::TB + kk * 2048), idKV,
                 (first && kk == 0) ? 0 : 1);
        }
#pragma unroll
        for (int kk = 0; kk < kT / 16; ++kk) {
          const uint32_t col = kk * 16;
          mma_ts(tbase + C::TDK, tB + col, sdesc_add(mdQ, s * C::TB + kk * 2048), idKV,
                 (first && kk == 0) ? 0 : 1);
        }
        mma_commit(bars.qempty(s));
        ++dq_n;
        ++pair_n;
        ++unit_pairs;
        kind = next_kind;
      }
      // drain every MMA before TMEM is freed
      mma_commit(bars.kvempty());
      mbar_drain(bars.kvempty(), unit_n & 1, ctl, 56);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ P / dS warpgroups
    const int wg = warp >> 2;              // query columns 64*wg .. +63
    const int r4 = warp & 3;
    const int kr = r4 * 32 + lane;         // key row within the unit tile
    const uint32_t lane_off = (uint32_t)(r4 * 32) << 16;
    const uint32_t tA = tbase + C::TA + lane_off, tB = tbase + C::TBc + lane_off;
    const float sl2 = P.scale_log2;
    int rec_n = 0, pair_n = 0, unit_pairs = 0;
    uint32_t sp_ph = 0, acc_ph = 0, dq_ph = 0;
    bool alive = true;
    uint8_t* dsT = sm + C::OFF_DS + wg * 16384;  // this warpgroup's 64-query block of dS^T
    while (alive) {
      const int slot = rec_n % kNInfo;
      alive = __all_sync(0xffffffffu, mbar_wait(bars.infofull(slot), (rec_n / kNInfo) & 1, ctl, 70));
      if (!alive) break;
      const BRec r = recs[slot];
      if (r.kind == kRecStop) {
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.infoempty(slot));
        break;
      }
      if (r.kind == kRecPair) {
        const int s = pair_n % C::QST;
        // (lse2, delta) of query column c is vec[c]; the copy started at an even row
        const float2* vec = reinterpret_cast<const float2*>(sm + C::OFF_VEC + s * C::VEC_BYTES) + (r.q0 & 1);
        const int* qsegp = pb.seg ? pb.seg + (size_t)r.b * pb.S : nullptr;
        alive = __all_sync(0xffffffffu, mbar_wait(bars.spfull(), sp_ph, ctl, 71));
        if (!alive) break;
        sp_ph ^= 1;
        tc_fence_after();
        const bool masked = r.flags & kMasked;
        const int kidx = r.k0 + kr;
        const int cb = pb.causal;
        const int kblk = cb > 0 ? (kidx + (kCarry ? P.koff : 0)) / cb : 0;
        const int kseg = (pb.seg && kr < r.kvalid) ? __ldg((kCarry ? P.kseg : pb.seg) + (size_t)r.b * pb.S + kidx) : 0;
        // this warpgroup's 64 query columns in quarters of 16: S^T from A, dP^T from B;
        // each quarter's 16 B columns become 8 columns of dS^T then 8 of P^T (bf16 pairs)
        uint32_t sv[16], dp[16];
        tmem_ld16(tA + wg * 64, sv);
        tmem_ld16(tB + wg * 64, dp);
        tmem_ld_wait16(sv);
        tmem_ld_wait16(dp);
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          const int c0 = wg * 64 + qq * 16;
          // branch-free exponentials for the whole quarter (one basic block, so the
          // independent per-element chains interleave), then the mask, then dS
          float pq[16], dq16[16];
#pragma unroll
          for (int y = 0; y < 16; y += 2) {
            const float2 va = vec[c0 + y], vb = vec[c0 + y + 1];
            float a0, a1;
            fma_f32x2(a0, a1, __uint_as_float(sv[y]), __uint_as_float(sv[y + 1]), sl2, sl2, -va.x, -vb.x);
            pq[y] = ex2_approx(a0);
            pq[y + 1] = ex2_approx(a1);
            add_f32x2(dq16[y], dq16[y + 1], __uint_as_float(dp[y]), __uint_as_float(dp[y + 1]), -va.y, -vb.y);
          }
          if (masked) {  // one uniform branch around the whole quarter; selects inside
#pragma unroll
            for (int y = 0; y < 16; ++y) {
              const int cc = c0 + y;
              const int qidx = r.q0 + cc;
              bool vis = (kr < r.kvalid) & (cc < r.qvalid);
              vis &= (cb <= 0) | ((qidx + (kCarry ? P.qoff : 0)) / max(cb, 1) >= kblk);
              const int qs = qsegp ? __ldg(qsegp + min(qidx, pb.S - 1)) : kseg;
              vis &= (qs == kseg);
              // masked: P = 0 and dS = 0 (dS by a select too, not 0 * (dP - Delta): the
              // (lse, Delta) entries of columns past the sequence end are not written)
              pq[y] = vis ? pq[y] : 0.f;
              dq16[y] = vis ? dq16[y] : 0.f;
            }
          }
          uint32_t pk[8], dk[8];
#pragma unroll
          for (int x = 0; x < 8; ++x) {
            pk[x] = pack_bf16x2(pq[2 * x], pq[2 * x + 1]);
            float d0, d1;
            mul_f32x2(d0, d1, pq[2 * x], pq[2 * x + 1], dq16[2 * x], dq16[2 * x + 1]);
            dk[x] = pack_bf16x2(d0, d1);
          }
          if (qq < 3) {  // next quarter's loads fly while this one is stored
            tmem_ld16(tA + c0 + 16, sv);
            tmem_ld16(tB + c0 + 16, dp);
          }
          tmem_st8(tB + c0, dk);
          tmem_st8(tB + c0 + 8, pk);
          // dS^T into smem: row kr, queries c0..c0+15 = 16-byte chunks 2qq, 2qq+1 (128B swizzle)
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            const int chunk = 2 * qq + ch;
            *reinterpret_cast<uint4*>(dsT + kr * 128 + ((chunk ^ (kr & 7)) * 16)) =
                make_uint4(dk[ch * 4], dk[ch * 4 + 1], dk[ch * 4 + 2], dk[ch * 4 + 3]);
          }
          if (qq < 3) {
            tmem_ld_wait16(sv);
            tmem_ld_wait16(dp);
          }
        }
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bars.pready());
        // dQ tile (written by the first MMA after pready) -> fp32 accumulator.  Each
        // warpgroup takes half of the tile's columns; tensor memory is released
        // before the adds are issued.
        alive = __all_sync(0xffffffffu, mbar_wait(bars.dqfull(), dq_ph, ctl, 73));
        if (!alive) break;
        dq_ph ^= 1;
        tc_fence_after();
        if constexpr (D == 128) {
          // dQ^T: lanes = head-dim index d, columns = queries.  Neighbouring lanes
          // (d even, d + 1) swap one value per query pair so that the even lane adds
          // (d, d + 1) of query i and the odd lane (d - 1, d) of query i + 1: one
          // 8-byte add per lane, and a warp-level add covers 128 bytes of two rows.
          uint32_t v[64];
          tmem_ld32(tA + wg * 64, v);
          tmem_ld32(tA + wg * 64 + 32, v + 32);
          tmem_ld_wait(v);
          tmem_ld_wait(v + 32);
          tc_fence_before();
          mbar_arrive(bars.dqfree());
          const size_t qstride = (size_t)pb.H * D;
          const int odd = lane & 1;
          // even lane: row i, columns d, d + 1; odd lane: row i + 1, columns d - 1, d
          float* base = P.dq_accum + (((size_t)r.b * pb.S + r.q0 + wg * 64) * pb.H + r.h) * D + kr - odd +
                        odd * qstride;
          const int nq = r.qvalid - wg * 64 - odd;
#pragma unroll
          for (int i = 0; i < 64; i += 2) {
            const float lo = __uint_as_float(v[i]), hi = __uint_as_float(v[i + 1]);
            const float got = __shfl_xor_sync(0xffffffffu, odd ? lo : hi, 1);
            if (i < nq) red_add_v2(base + (size_t)i * qstride, odd ? got : lo, odd ? hi : got);
          }
        } else {
          // dQ: lanes = query rows, columns = head dim (32 per warpgroup); 16-byte adds
          uint32_t v[32];
          tmem_ld32(tA + wg * 32, v);
          tmem_ld_wait(v);
          tc_fence_before();
          mbar_arrive(bars.dqfree());
          if (kr < r.qvalid) {
            float* dst = P.dq_accum + (((size_t)r.b * pb.S + r.q0 + kr) * pb.H + r.h) * D + wg * 32;
#pragma unroll
            for (int x = 0; x < 32; x += 4)
              red_add_v4(dst + x, __uint_as_float(v[x]), __uint_as_float(v[x + 1]), __uint_as_float(v[x + 2]),
                         __uint_as_float(v[x + 3]));
          }
        }
        ++pair_n;
        ++unit_pairs;
      } else if (r.kind == kRecUnitEnd) {
        // dK (warpgroup 0) or dV (warpgroup 1) rows -> bf16
        alive = __all_sync(0xffffffffu, mbar_wait(bars.accdone(), acc_ph, ctl, 72));
        if (!alive) break;
        acc_ph ^= 1;
        tc_fence_after();
        const uint32_t tacc = tbase + (wg == 0 ? C::TDK : C::TDV) + lane_off;
        const float mul = wg == 0 ? P.scale : 1.f;
        const size_t row = ((size_t)r.b * pb.S + r.k0 + kr) * pb.H + r.h;
#pragma unroll
        for (int cq = 0; cq < D / 32; ++cq) {
          uint32_t o[32];
          tmem_ld32(tacc + cq * 32, o);
          tmem_ld_wait(o);
          if constexpr (!kCarry) {
            __nv_bfloat16* dst = (wg == 0 ? P.dk : P.dv) + row * D;
            if (unit_pairs == 0) {  // no visible query: the gradient is zero
#pragma unroll
              for (int x = 0; x < 32; ++x) o[x] = 0u;
            }
            if (kr < r.kvalid) {
              uint4* d4 = reinterpret_cast<uint4*>(dst + cq * 32);
#pragma unroll
              for (int v4 = 0; v4 < 4; ++v4) {
                uint4 val;
                val.x = pack_bf16x2(__uint_as_float(o[v4 * 8 + 0]) * mul, __uint_as_float(o[v4 * 8 + 1]) * mul);
                val.y = pack_bf16x2(__uint_as_float(o[v4 * 8 + 2]) * mul, __uint_as_float(o[v4 * 8 + 3]) * mul);
                val.z = pack_bf16x2(__uint_as_float(o[v4 * 8 + 4]) * mul, __uint_as_float(o[v4 * 8 + 5]) * mul);
                val.w = pack_bf16x2(__uint_as_float(o[v4 * 8 + 6]) * mul, __uint_as_float(o[v4 * 8 + 7]) * mul);
                d4[v4] = val;
              }
            }
          } else {
            // Ring step: this key block's gradients from this query block are added
            // to the carries that travel around the ring with K and V.  Each unit
            // owns its key rows, so the read-modify-write does not race.
            if (unit_pairs > 0 && kr < r.kvalid) {
              float4* d4 = reinterpret_cast<float4*>((wg == 0 ? P.dk_carry : P.dv_carry) + row * D + cq * 32);
#pragma unroll
              for (int v4 = 0; v4 < 8; ++v4) {
                float4 c4 = d4[v4];
                c4.x += __uint_as_float(o[v4 * 4 + 0]) * mul;
                c4.y += __uint_as_float(o[v4 * 4 + 1]) * mul;
                c4.z += __uint_as_float(o[v4 * 4 + 2]) * mul;
                c4.w += __uint_as_float(o[v4 * 4 + 3]) * mul;
                d4[v4] = c4;
              }
            }
          }
        }
        tc_fence_before();
        mbar_arrive(bars.accfree());
        unit_pairs = 0;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.infoempty(slot));
      ++rec_n;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tbase, 512);
}

}  // namespace

// Stages of the backward (BwdArgs::stage): the whole backward on one sequence,
// or one of the three parts a ring of separate blocks runs (begin once,
// one step per key/value block, end once).
template <int D, bool kCarry, bool kLog>
static cudaError_t launch_bwd_main(const BwdArgs& a, const Ctx& c, uint64_t* launches, const char** why) {
  using Cf = BCfg<D>;
  const Problem& p = a.p;
  CUtensorMap mq, mk, mv, mdo;
  if (!make_tile_map(&mq, a.q, p, kT) || !make_tile_map(&mk, a.k, p, kT) || !make_tile_map(&mv, a.v, p, kT) ||
      !make_tile_map(&mdo, a.dout, p, kT)) {
    *why = "cuTensorMapEncodeTiled failed (driver entry point unavailable or tensor rejected)";
    return cudaSuccess;
  }
  BwdParams P;
  P.p = p;
  P.ld2 = (const float2*)a.delta;
  P.Sp = bwd_row_pitch(p.S);
  P.dq_accum = a.dq_accum;
  P.dk = (__nv_bfloat16*)a.dk;
  P.dv = (__nv_bfloat16*)a.dv;
  P.status = c.status;
  P.limit_ns = c.limit_ns;
  P.tiles_per_shard = (p.Ssh + kT - 1) / kT;
  P.num_units = p.B * p.H * p.N * P.tiles_per_shard;
  P.scale = (float)(1.0 / sqrt((double)p.D));
  P.scale_log2 = (float)(1.4426950408889634 / sqrt((double)p.D));
  P.unit_counter = a.unit_counter;
  P.qoff = a.qoff;
  P.koff = a.koff;
  P.kseg = a.kseg ? a.kseg : p.seg;
  P.dk_carry = a.dk_carry;
  P.dv_carry = a.dv_carry;
  P.vlog = a.vlog;
  P.vlog_cap = a.vlog_cap;
  {  // heads whose Q, dO (bf16) and dQ accumulator (fp32), 8 * S * D bytes, fit in
     // 48 MB of L2 together, or in 128 MB when one head's take 16 MB or less (the
     // forward's rule: balance for short heads, no DRAM re-reads for long ones)
    const long long per = 8LL * p.S * p.D;
    const long long budget = per <= (16LL << 20) ? (128LL << 20) : (48LL << 20);
    P.group_heads = (int)std::max(1LL, std::min((long long)p.B * p.H, budget / per));
  }
  static std::atomic<bool> attr_set[256];  // idempotent attribute; atomic so threads may race
  if (!attr_set[c.device]) {
    cudaError_t e = cudaFuncSetAttribute(bwd_bf16_kernel<D, kCarry, kLog>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)Cf::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[c.device] = true;
  }
  const int grid = std::min(c.num_sms, P.num_units);
  bwd_bf16_kernel<D, kCarry, kLog><<<grid, kThreads, Cf::SMEM, c.stream>>>(mq, mk, mv, mdo, P);
  *launches += 1;
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_bwd_bf16_d(const BwdArgs& a, const Ctx& c, uint64_t* launches, const char** why) {
  const Problem& p = a.p;
  const long long rows = (long long)p.B * p.S * p.H;
  cudaError_t e;
  if (a.stage == kBwdWhole || a.stage == kBwdRingBegin) {
    bwd_pre_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, c.stream>>>(
        p, (const __nv_bfloat16*)a.out, (const __nv_bfloat16*)a.dout, a.lse, (float2*)a.delta, bwd_row_pitch(p.S),
        a.dq_accum, a.unit_counter);
    *launches += 1;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (a.stage == kBwdWhole) {
    e = a.vlog ? launch_bwd_main<D, false, true>(a, c, launches, why)
               : launch_bwd_main<D, false, false>(a, c, launches, why);
    if (e != cudaSuccess || *why) return e;
  } else if (a.stage == kBwdRingStep) {
    // every launch of the main kernel starts from a zero unit counter
    if ((e = cudaMemsetAsync(a.unit_counter, 0, sizeof(int), c.stream)) != cudaSuccess) return e;
    e = a.vlog ? launch_bwd_main<D, true, true>(a, c, launches, why)
               : launch_bwd_main<D, true, false>(a, c, launches, why);
    if (e != cudaSuccess || *why) return e;
  }
  if (a.stage == kBwdWhole || a.stage == kBwdRingEnd) {
    const size_t n4 = (size_t)rows * p.D / 4;
    bwd_fin_kernel<<<c.num_sms * 8, 256, 0, c.stream>>>(n4, (const float4*)a.dq_accum, (uint2*)a.dq,
                                                        (float)(1.0 / sqrt((double)p.D)));
    *launches += 1;
    return cudaGetLastError();
  }
  return cudaSuccess;
}

cudaError_t launch_cast_bf16(const float* src, void* dst, size_t count, float scale, const Ctx& c,
                             uint64_t* launches) {
  bwd_fin_kernel<<<c.num_sms * 8, 256, 0, c.stream>>>(count / 4, (const float4*)src, (uint2*)dst, scale);
  *launches += 1;
  return cudaGetLastError();
}

cudaError_t launch_bwd_bf16(const BwdArgs& a, const Ctx& c, uint64_t* launches, const char** why) {
  if (a.p.D == 64) return launch_bwd_bf16_d<64>(a, c, launches, why);
  if (a.p.D == 128) return launch_bwd_bf16_d<128>(a, c, launches, why);
  *why = "bf16 head_dim must be 64 or 128";
  return cudaSuccess;
}

}  // namespace ra
