// attn_fwd_sm103.cu — bf16 forward of blockwise ring attention on sm_103a.
//
// What it computes: per (batch, head), out = softmax(Q K^T / sqrt(d)) V and the
// natural-log lse of each row ("Ring Attention with Blockwise Transformers for
// Near-Infinite Context", paper review page, §三 核心公式), with the sequence
// split into N contiguous virtual shards and each query shard j visiting the
// KV shards in ring order k = (j - i) mod N (same page, 环形注意力算法).  The
// running max / numerator / denominator update is the lazy softmax of the code
// walk-through page ("从论文到代码：深入理解RingAttention的块注意力计算逻辑",
// §2 数值稳定的注意力计算); tiles with no visible element are skipped (§3,
// below_or_on_diag), and segment ids mask across documents.
//
// How (one persistent CTA per SM, 10 warps; 11 at D = 64):
//   warps 0-3  softmax warpgroup for Q tile 0 (TMEM lanes 0-127, one row per thread)
//   warps 4-7  softmax warpgroup for Q tile 1
//   warp 8     producer: takes query-tile-pair units (from a per-call counter,
//              or a fixed schedule under stream capture), walks the ring
//              schedule, classifies 32 key tiles at once (one per lane: skip /
//              full / needs a mask; at D = 64 from a per-tile segment-id
//              summary that all warps build in smem at kernel start), publishes
//              a record per visible tile and TMA-loads K and V into a smem ring
//              (128B swizzle)
//   warp 9     MMA issuer: S_w = Q_w K^T (SS, fp32 in TMEM), then
//              O_w += P_w V with P_w read from TMEM (TS), ping-ponging the two
//              Q tiles so the tensor pipe runs one tile's MMAs while the other
//              tile's softmax runs.  At D = 64 warps 9 and 10 each issue one Q
//              tile's MMAs instead (Cfg::ISSUERS).
// Tensor memory (512 columns): S0 | S1 | O0 | O1.  P_w is written as packed
// bf16 pairs over the first 64 columns of S_w at D = 128; at D = 64 it has
// columns of its own (S0 | S1 | O0 | O1 | P0 | P1), so S_w(t + 1) can be issued
// once the softmax has read S_w(t), ahead of PV_w(t).
// The running max is only moved (and O, l rescaled) when a row's tile max
// exceeds it by more than 2^8; in exact arithmetic the result is unchanged
// (numerator and denominator carry the same factor), and the exponentials
// stay <= 256.  Every mbarrier wait is bounded (see sm103.cuh).
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <cudaTypedefs.h>

#include "ra_internal.h"
#include "sm103.cuh"

namespace ra {
namespace {

constexpr int kBM = 128;  // rows per Q tile
constexpr int kBN = 128;  // keys per KV tile
constexpr int kNInfo = 8; // schedule-record ring depth
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

enum : int { kRecTile = 0, kRecUnitEnd = 1, kRecStop = 2 };
enum : int { kSkip0 = 1, kSkip1 = 2, kMask0 = 4, kMask1 = 8, kKeyUni = 16 };  // kKeyUni: every key id of the tile is kseg

struct __align__(16) Rec {
  int kind;
  int flags;
  int kstart;   // first key (global sequence index) of the tile
  int kvalid;   // keys of the tile that lie inside the shard (1..128)
  int b, h;
  int q0;       // first row of Q tile 0 (global); tile 1 starts at q0 + 128
  int qvalid0, qvalid1;  // rows of each Q tile inside the shard (0 = tile absent)
  int kseg;              // with kKeyUni: the segment id of every key of the tile
  int pad[2];
};

template <int D>
struct Cfg {
  // MMA issuers: at D = 128 one thread issues both Q tiles' MMAs in the order
  // PV0, S0, PV1, S1, which keeps one tile's MMAs under the other tile's softmax.
  // At D = 64 the MMAs are short, and one issuer per Q tile (warps 9 and 10) lets
  // each tile's chain run without waiting on the other's softmax.
  static constexpr int ISSUERS = (D == 64) ? 2 : 1;
  static constexpr int THREADS = 32 * (9 + ISSUERS);     // softmax 0-7, producer 8, MMA 9 (and 10)
  static constexpr int KST = (D == 64) ? 4 : 2;          // K/V ring stages
  static constexpr uint32_t QT = kBM * D * 2;            // bytes of one Q tile
  static constexpr uint32_t KVT = kBN * D * 2;           // bytes of one K or V tile
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + 2 * QT;
  static constexpr uint32_t OFF_V = OFF_K + KST * KVT;
  static constexpr uint32_t OFF_REC = OFF_V + KST * KVT;
  static constexpr uint32_t OFF_BAR = OFF_REC + kNInfo * sizeof(Rec);
  // barriers: qfull, qempty, kfull[KST], kempty[KST], vfull[KST], vempty[KST],
  //           infofull[8], infoempty[8], sfull[2], pready[2], odone[2], ofree[2]
  static constexpr int NBAR = 2 + 4 * KST + 2 * kNInfo + 8 + ((D == 64) ? 4 : 0);  // + sread[2], pfree[2]
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  // Segment-id (min, max) of every key tile (b, shard, tile), built at kernel
  // start when segment ids are given and the tiles fit (else the producer reads
  // each tile's ids itself).  D = 64 only, the head size of the packed-document
  // workloads: at D = 128 the extra code cost the unsegmented forward ~0.5 %.
  static constexpr int SUMCAP = (D == 64) ? 4096 : 0;
  static constexpr uint32_t OFF_SUM = OFF_MISC + 64;
  static constexpr uint32_t SMEM = OFF_SUM + SUMCAP * 8 + 1024;  // + alignment slack
  static constexpr uint32_t TCOL_O = 256;                 // O0 at 256, O1 at 256 + D
  // D = 64: P_w in columns of its own (384 + 64 w), so S_w(t + 1) can be written
  // as soon as the softmax has read S_w(t), ahead of PV_w(t).
  static constexpr bool PSEP = (D == 64);
  static constexpr uint32_t TCOL_P = 256 + 2 * D;
};

struct Bars {
  uint32_t base;
  int kst;
  __device__ uint32_t qfull() const { return base; }
  __device__ uint32_t qempty() const { return base + 8; }
  __device__ uint32_t kfull(int s) const { return base + 16 + 8 * s; }
  __device__ uint32_t kempty(int s) const { return base + 16 + 8 * (kst + s); }
  __device__ uint32_t vfull(int s) const { return base + 16 + 8 * (2 * kst + s); }
  __device__ uint32_t vempty(int s) const { return base + 16 + 8 * (3 * kst + s); }
  __device__ uint32_t infofull(int i) const { return base + 16 + 8 * (4 * kst + i); }
  __device__ uint32_t infoempty(int i) const { return base + 16 + 8 * (4 * kst + kNInfo + i); }
  __device__ uint32_t sfull(int w) const { return base + 16 + 8 * (4 * kst + 2 * kNInfo + w); }
  __device__ uint32_t pready(int w) const { return base + 16 + 8 * (4 * kst + 2 * kNInfo + 2 + w); }
  __device__ uint32_t odone(int w) const { return base + 16 + 8 * (4 * kst + 2 * kNInfo + 4 + w); }
  __device__ uint32_t ofree(int w) const { return base + 16 + 8 * (4 * kst + 2 * kNInfo + 6 + w); }
  __device__ uint32_t sread(int w) const { return base + 16 + 8 * (4 * kst + 2 * kNInfo + 8 + w); }
  __device__ uint32_t pfree(int w) const { return base + 16 + 8 * (4 * kst + 2 * kNInfo + 10 + w); }
};

struct FwdParams {
  Problem p;
  __nv_bfloat16* out;
  float* lse;
  // Positions and key segment ids.  Query row r sits at position r + qoff and key
  // row x at x + koff (both 0 for one sequence cut into virtual shards; a ring
  // step between two separate blocks passes their global offsets).  kseg holds the
  // key rows' segment ids (the same array as p.seg for one sequence).
  int qoff, koff;
  const int32_t* kseg;
  // Ring-step carry (kCarry kernels only): fp32 running output [B, S, H, D] and
  // natural-log lse [B, H, S] that this call's result is merged into.
  float* o_carry;
  float* lse_carry;
  int* vlog;            // visit log (see visit_log), or null
  int vlog_cap;         // entries the log holds
  int* status;
  uint64_t limit_ns;
  int tiles_per_shard;  // ceil(Ssh / 128)
  int pairs_per_shard;  // ceil(tiles_per_shard / 2)
  int num_units;        // B * H * N * pairs_per_shard
  float scale_log2;     // log2(e) / sqrt(D)
  int* unit_counter;    // zeroed per call: CTAs draw tickets as they free up; null: static pairs
  int group_heads;      // (b, h) heads per ticket group (their K and V fit in part of L2)
};

__device__ __forceinline__ int floordiv_pos(int a, int c) { return a / c; }  // a >= 0

// Unit u -> (b, h, query shard j, pair index).  Units are numbered head-major,
// and within a head by decreasing query position (rank 0 = longest causal work).
// The order in which CTAs take them is set by ticket_unit (dynamic) or by the
// static pairs in the producer.
__device__ __forceinline__ void unit_coords(const FwdParams& P, int u, int& b, int& h, int& j, int& pr) {
  const int per_head = P.p.N * P.pairs_per_shard;
  const int bh = u / per_head;
  const int g = per_head - 1 - (u % per_head);
  j = g / P.pairs_per_shard;
  pr = g % P.pairs_per_shard;
  b = bh / P.p.H;
  h = bh % P.p.H;
}

// Ticket t -> unit.  The (b, h) heads form groups of group_heads whose K and V
// fit in L2 together; a group's tickets go rank-major (the longest causal unit of
// every head of the group, then the next longest, ...), so the last tickets of a
// group are its shortest units and the CTAs finish together.
__device__ __forceinline__ int ticket_unit(const FwdParams& P, int t) {
  const int per_head = P.p.N * P.pairs_per_shard;
  const int bh_total = P.p.B * P.p.H;
  const int G = P.group_heads;
  const int g = t / (G * per_head);
  const int g0 = g * G;                     // first head of the group
  const int gh = min(G, bh_total - g0);     // heads in the group (the last may be short)
  const int w = t - g * G * per_head;       // ticket within the group, < gh * per_head
  const int rank = w / gh;                  // 0 = longest causal work
  return (g0 + (w - rank * gh)) * per_head + rank;
}

template <int D, bool kCarry, bool kLog>
__global__ void __launch_bounds__(Cfg<D>::THREADS, 1)  // 10-11 warps: 3 on some SM sub-partitions -> <= 168 registers
    fwd_bf16_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                    const __grid_constant__ CUtensorMap mv, const FwdParams P) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* sm = smem_raw + ((1024 - (raw & 1023)) & 1023);
  const uint32_t sbase = smem_u32(sm);
  Rec* recs = reinterpret_cast<Rec*>(sm + C::OFF_REC);
  Bars bars{sbase + C::OFF_BAR, C::KST};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::OFF_MISC + 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bars.qfull(), 1);
    mbar_init(bars.qempty(), C::ISSUERS);  // one commit per MMA issuer
    for (int s = 0; s < C::KST; ++s) {
      mbar_init(bars.kfull(s), 1);
      mbar_init(bars.kempty(s), C::ISSUERS);
      mbar_init(bars.vfull(s), 1);
      mbar_init(bars.vempty(s), C::ISSUERS);
    }
    for (int i = 0; i < kNInfo; ++i) {
      mbar_init(bars.infofull(i), 1);
      mbar_init(bars.infoempty(i), C::ISSUERS + 8);  // MMA threads + one lane per softmax warp
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(bars.sfull(w), 1);
      mbar_init(bars.pready(w), 4);  // one arrival per softmax warp
      mbar_init(bars.odone(w), 1);
      mbar_init(bars.ofree(w), 4);
      if constexpr (C::PSEP) {
        mbar_init(bars.sread(w), 4);  // one arrival per softmax warp: S_w read into registers
        mbar_init(bars.pfree(w), 1);  // MMA commit after PV_w: P_w and O_w may be written
      }
    }
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  // Key segment summary: warp-per-tile, 4 ids per lane, 8 tiles in flight.
  const int nsum = (C::SUMCAP > 0 && P.p.seg) ? P.p.B * P.p.N * P.tiles_per_shard : 0;
  const bool use_sum = C::SUMCAP > 0 && nsum > 0 && nsum <= C::SUMCAP;
  int2* ksum = reinterpret_cast<int2*>(sm + C::OFF_SUM);
  if constexpr (C::SUMCAP > 0) if (use_sum) {
    const int* kids = kCarry ? P.kseg : P.p.seg;
    const int nwarps = C::THREADS / 32;
    for (int e0 = warp * 8; e0 < nsum; e0 += nwarps * 8) {
      int mn[8], mx[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        mn[u] = INT_MAX;
        mx[u] = INT_MIN;
        const int e = e0 + u;
        if (e < nsum) {
          const int t = e % P.tiles_per_shard, bk = e / P.tiles_per_shard;
          const int k = bk % P.p.N, bb = bk / P.p.N;
          const int ka = k * P.p.Ssh + t * kBN;
          const int n = min(kBN, (k + 1) * P.p.Ssh - ka);
          const int* sp = kids + (size_t)bb * P.p.S + ka;
          if (n == kBN && ((reinterpret_cast<uintptr_t>(sp) & 15u) == 0)) {
            const int4 v4 = __ldg(reinterpret_cast<const int4*>(sp) + lane);
            mn[u] = min(min(v4.x, v4.y), min(v4.z, v4.w));
            mx[u] = max(max(v4.x, v4.y), max(v4.z, v4.w));
          } else {
            for (int x = lane; x < n; x += 32) {
              const int v = __ldg(sp + x);
              mn[u] = min(mn[u], v);
              mx[u] = max(mx[u], v);
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          mn[u] = min(mn[u], __shfl_xor_sync(0xffffffffu, mn[u], o));
          mx[u] = max(mx[u], __shfl_xor_sync(0xffffffffu, mx[u], o));
        }
        if (lane == 0 && e0 + u < nsum) ksum[e0 + u] = make_int2(mn[u], mx[u]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  WaitCtl ctl{P.status, abort_flag, P.limit_ns};
  const Problem& pb = P.p;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------------
    // Producer: ring schedule + TMA
    // ------------------------------------------------------------------
    if (lane == 0) {
      tma_prefetch_desc(&mq);
      tma_prefetch_desc(&mk);
      tma_prefetch_desc(&mv);
    }
    int rec_n = 0, tile_n = 0, unit_n = 0, q_loads = 0;
    bool alive = true;
    const int c = pb.causal;
    const int qo = kCarry ? P.qoff : 0, ko = kCarry ? P.koff : 0;
    // publish a record (lane 0 only); returns false on abort
    auto publish = [&](const Rec& r) -> bool {
      const int slot = rec_n % kNInfo;
      if (!mbar_wait(bars.infoempty(slot), ((rec_n / kNInfo) & 1) ^ 1, ctl, 10)) return false;
      recs[slot] = r;
      mbar_arrive(bars.infofull(slot));
      ++rec_n;
      return true;
    };
    // Unit order.  With a unit counter, CTAs draw tickets (ticket_unit: L2-sized head
    // groups, longest units first) as they become free, so uneven unit costs
    // (packed documents, few units per SM) even out; the next ticket is drawn one
    // unit ahead so its latency hides behind the current unit.  Without one,
    // units go out in balanced pairs: within a head, unit r (long causal work) with
    // unit per_head - 1 - r (short), CTA c taking pairs c, c + G, ...  Either way all
    // CTAs move through one or two heads together, keeping those heads' operands
    // resident in L2.
    const int per_head = pb.N * P.pairs_per_shard;
    const int pairs_per_head = (per_head + 1) / 2;
    const int num_super = (P.num_units / per_head) * pairs_per_head;
    int st_su = blockIdx.x, st_half = 0;
    auto static_next = [&]() -> int {
      while (st_su < num_super) {
        const int su = st_su, half = st_half;
        if (++st_half == 2) {
          st_half = 0;
          st_su += gridDim.x;
        }
        const int rr = su % pairs_per_head;
        const int rank = half == 0 ? rr : per_head - 1 - rr;
        if (half == 1 && rank == rr) continue;  // odd count: the middle unit has no partner
        return (su / pairs_per_head) * per_head + rank;
      }
      return -1;
    };
    auto ticket = [&]() -> int {  // lane 0 draws, the warp gets the unit (or -1)
      int t = 0;
      if (lane == 0) t = atomicAdd(P.unit_counter, 1);
      t = __shfl_sync(0xffffffffu, t, 0);
      return t < P.num_units ? ticket_unit(P, t) : -1;
    };
    int u = P.unit_counter ? ticket() : static_next();
    while (u >= 0 && alive) {
      int ahead = 0;
      if (P.unit_counter && lane == 0) ahead = atomicAdd(P.unit_counter, 1);
      int b, h, j, pr;
      unit_coords(P, u, b, h, j, pr);
      const int shard0 = j * pb.Ssh;
      const int q0 = shard0 + pr * 2 * kBM;
      const int qv0 = max(0, min(kBM, shard0 + pb.Ssh - q0));
      const int qv1 = max(0, min(kBM, shard0 + pb.Ssh - (q0 + kBM)));
      // segment range of each Q tile
      int qmin[2] = {0, 0}, qmax[2] = {0, 0};
      if (pb.seg && use_sum && !kCarry) {
        for (int w = 0; w < 2; ++w) {
          const int tq = pr * 2 + w;
          const int nv = w == 0 ? qv0 : qv1;
          qmin[w] = INT_MAX;
          qmax[w] = INT_MIN;
          if (nv > 0 && tq < P.tiles_per_shard) {
            const int2 mm = ksum[((size_t)b * pb.N + j) * P.tiles_per_shard + tq];
            qmin[w] = mm.x;
            qmax[w] = mm.y;
          }
        }
      } else if (pb.seg) {
        for (int w = 0; w < 2; ++w) {
          const int nv = w == 0 ? qv0 : qv1;
          int mn = INT_MAX, mx = INT_MIN;
          for (int r = lane; r < nv; r += 32) {
            const int sv = __ldg(pb.seg + (size_t)b * pb.S + q0 + w * kBM + r);
            mn = min(mn, sv);
            mx = max(mx, sv);
          }
          for (int o = 16; o > 0; o >>= 1) {
            mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
            mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          }
          qmin[w] = mn;
          qmax[w] = mx;
        }
      }
      // Q tiles (wait until the previous unit's S MMAs have finished with Q smem)
      if (lane == 0) {
        alive = mbar_wait(bars.qempty(), (unit_n & 1) ^ 1, ctl, 11);
        if (alive) {
          ++q_loads;
          mbar_arrive_expect_tx(bars.qfull(), 2 * C::QT);
          for (int w = 0; w < 2; ++w)
            for (int cb = 0; cb < D / 64; ++cb)
              tma_load_4d(sbase + C::OFF_Q + w * C::QT + cb * 16384, &mq, bars.qfull(), cb * 64, h,
                          q0 + w * kBM, b);
        }
      }
      alive = __shfl_sync(0xffffffffu, alive, 0);
      const int qlast0 = q0 + max(qv0, 1) - 1;
      const int qlast1 = q0 + kBM + max(qv1, 1) - 1;
      const int qlast = qv1 > 0 ? qlast1 : qlast0;
      for (int i = 0; i < pb.N && alive; ++i) {
        const int ks = ((j - i) % pb.N + pb.N) % pb.N;  // ring order
        const int kbeg = ks * pb.Ssh, kend = kbeg + pb.Ssh;
        if (c > 0 && floordiv_pos(qlast + qo, c) < floordiv_pos(kbeg + ko, c)) continue;  // whole shard in the future
        for (int t0 = 0; t0 < P.tiles_per_shard && alive; t0 += 32) {
          // tile segment ranges, one tile per lane
          int kmn = 0, kmx = 0;
          const int my_t = t0 + lane;
          if (pb.seg && my_t < P.tiles_per_shard) {
            const int ka = kbeg + my_t * kBN;
            const int kb = min(kend, ka + kBN);
            bool needed = !(c > 0 && floordiv_pos(qlast + qo, c) < floordiv_pos(ka + ko, c));
            int mn = INT_MAX, mx = INT_MIN;
            if (needed && use_sum) {
              const int2 mm = ksum[((size_t)b * pb.N + ks) * P.tiles_per_shard + my_t];
              mn = mm.x;
              mx = mm.y;
            } else if (needed) {
              const int* sp = (kCarry ? P.kseg : pb.seg) + (size_t)b * pb.S + ka;
              if (kb - ka == kBN && ((reinterpret_cast<uintptr_t>(sp) & 15u) == 0)) {
#pragma unroll 8
                for (int x4 = 0; x4 < kBN / 4; ++x4) {
                  const int4 sv = __ldg(reinterpret_cast<const int4*>(sp) + x4);
                  mn = min(mn, min(min(sv.x, sv.y), min(sv.z, sv.w)));
                  mx = max(mx, max(max(sv.x, sv.y), max(sv.z, sv.w)));
                }
              } else {
                for (int x = 0; x < kb - ka; ++x) {
                  const int sv = __ldg(sp + x);
                  mn = min(mn, sv);
                  mx = max(mx, sv);
                }
              }
            }
            kmn = mn;
            kmx = mx;
          }
          // Each lane classifies its own tile; the warp then walks the visible ones
          // only, so skipped positions cost nothing serial.
          const int tend = min(32, P.tiles_per_shard - t0);
          int my_flags = kSkip0 | kSkip1;
          if (lane < tend) {
            const int ka = kbeg + my_t * kBN;
            const int kb = ka + min(kBN, kend - ka) - 1;
            my_flags = 0;
            for (int w = 0; w < 2; ++w) {
              const int qv = w == 0 ? qv0 : qv1;
              const int qa = q0 + w * kBM, ql = qa + qv - 1;
              bool skip = qv == 0, full = true;
              if (!skip && c > 0) {
                if (floordiv_pos(ql + qo, c) < floordiv_pos(ka + ko, c)) skip = true;
                else if (!(floordiv_pos(qa + qo, c) >= floordiv_pos(kb + ko, c))) full = false;
              }
              if (!skip && pb.seg) {
                if (kmx < qmin[w] || kmn > qmax[w]) skip = true;
                else if (!(qmin[w] == qmax[w] && kmn == qmax[w] && kmx == qmax[w])) full = false;
              }
              if (kb - ka + 1 < kBN) full = false;
              if (skip) my_flags |= (w == 0 ? kSkip0 : kSkip1);
              else if (!full) my_flags |= (w == 0 ? kMask0 : kMask1);
            }
            if constexpr (D == 64) {  // a masked row then needs one id compare (see the softmax)
              if (pb.seg && kmn == kmx) my_flags |= kKeyUni;
            }
          }
          uint32_t todo = __ballot_sync(0xffffffffu, (my_flags & (kSkip0 | kSkip1)) != (kSkip0 | kSkip1));
          while (todo != 0u && alive) {
            const int tt = __ffs(todo) - 1;
            todo &= todo - 1u;
            const int flags = __shfl_sync(0xffffffffu, my_flags, tt);
            int kseg = 0;
            if constexpr (D == 64) kseg = __shfl_sync(0xffffffffu, kmn, tt);
            const int ka = kbeg + (t0 + tt) * kBN;
            const int kvalid = min(kBN, kend - ka);
            if (lane == 0) {
              Rec r;
              r.kind = kRecTile;
              r.flags = flags;
              r.kstart = ka;
              r.kvalid = kvalid;
              r.b = b;
              r.h = h;
              r.q0 = q0;
              r.qvalid0 = qv0;
              r.qvalid1 = qv1;
              if constexpr (D == 64) r.kseg = kseg;
              alive = publish(r);
              if constexpr (kLog) visit_log(P.vlog, P.vlog_cap, 0, b, h, j, pr, i, ks, t0 + tt);
              const int s = tile_n % C::KST;
              const uint32_t par = ((tile_n / C::KST) & 1) ^ 1;
              if (alive) alive = mbar_wait(bars.kempty(s), par, ctl, 12);
              if (alive) {
                mbar_arrive_expect_tx(bars.kfull(s), C::KVT);
                for (int cb = 0; cb < D / 64; ++cb)
                  tma_load_4d(sbase + C::OFF_K + s * C::KVT + cb * 16384, &mk, bars.kfull(s), cb * 64, h, ka, b);
              }
              if (alive) alive = mbar_wait(bars.vempty(s), par, ctl, 13);
              if (alive) {
                mbar_arrive_expect_tx(bars.vfull(s), C::KVT);
                for (int cb = 0; cb < D / 64; ++cb)
                  tma_load_4d(sbase + C::OFF_V + s * C::KVT + cb * 16384, &mv, bars.vfull(s), cb * 64, h, ka, b);
              }
              ++tile_n;
            }
            alive = __shfl_sync(0xffffffffu, alive, 0);
          }
        }
      }
      if (lane == 0 && alive) {
        Rec r;
        r.kind = kRecUnitEnd;
        r.flags = 0;
        r.kstart = 0;
        r.kvalid = 0;
        r.b = b;
        r.h = h;
        r.q0 = q0;
        r.qvalid0 = qv0;
        r.qvalid1 = qv1;
        alive = publish(r);
      }
      alive = __shfl_sync(0xffffffffu, alive, 0);
      ++unit_n;
      if (P.unit_counter) {
        const int t = __shfl_sync(0xffffffffu, ahead, 0);
        u = t < P.num_units ? ticket_unit(P, t) : -1;
      } else {
        u = static_next();
      }
    }
    if (lane == 0 && alive) {
      Rec r;
      r.kind = kRecStop;
      publish(r);
    }
    // Let every issued copy land before the CTA can exit (bounded, ignores abort).
    if (lane == 0) {
      for (int s = 0; s < C::KST; ++s) {
        if (tile_n <= s) continue;
        const int last = s + ((tile_n - 1 - s) / C::KST) * C::KST;  // last tile that used stage s
        const uint32_t par = (last / C::KST) & 1;
        mbar_drain(bars.kfull(s), par, ctl, 14);
        mbar_drain(bars.vfull(s), par, ctl, 15);
      }
      if (q_loads > 0) mbar_drain(bars.qfull(), (q_loads - 1) & 1, ctl, 16);
    }
  } else if (warp == kMmaWarp || (C::ISSUERS == 2 && warp == kMmaWarp + 1)) {
    // ------------------------------------------------------------------
    // MMA issuer(s) (lane 0): both Q tiles, or (two issuers) the warp's own
    // ------------------------------------------------------------------
    // Q tiles this thread issues: w = 0, 1 with one issuer; w = mw with two.  The
    // loop bounds below fold to exactly those two forms at compile time (written
    // any other way, the generated code of both instances ran slower).
    const int mw = warp - kMmaWarp;
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(kBM, kBN, 0, 0);
      constexpr uint32_t idO = idesc_bf16_f32(kBM, D, 0, 1);
      int tile_n = 0, unit_n = 0;
      uint32_t ofree_ph[2] = {1, 1}, pready_ph[2] = {0, 0};
      bool alive = true;
      int s_n[2] = {0, 0};  // S issued per Q tile (PSEP: the softmax reads each once)
      // Shared-memory descriptors of every operand buffer, built once; each MMA
      // adds a compile-time byte offset.
      const uint64_t dQ0 = sdesc_sw128(sbase + C::OFF_Q, 16, 1024);
      const uint64_t dK0 = sdesc_sw128(sbase + C::OFF_K, 16, 1024);
      const uint64_t dV0 = sdesc_sw128(sbase + C::OFF_V, 16384, 1024);
      auto dQ = [&](int w) { return sdesc_add(dQ0, w * C::QT); };
      auto dK = [&](int s) { return sdesc_add(dK0, s * C::KVT); };
      auto dV = [&](int s) { return sdesc_add(dV0, s * C::KVT); };
      struct MRec {  // the two record fields the MMA warp needs
        int kind, flags;
      };
      auto release = [&](int n) { mbar_arrive(bars.infoempty(n % kNInfo)); };
      auto issue_S = [&](const MRec& r, int stage) -> bool {
        if (!mbar_wait(bars.kfull(stage), (tile_n / C::KST) & 1, ctl, 21)) return false;
        tc_fence_after();
        for (int w = C::ISSUERS == 2 ? mw : 0; C::ISSUERS == 2 ? w == mw : w < 2; ++w) {
          if (r.flags & (w == 0 ? kSkip0 : kSkip1)) continue;
          if constexpr (C::PSEP) {
            if (s_n[w] > 0 && !mbar_wait(bars.sread(w), (s_n[w] - 1) & 1, ctl, 28)) return false;
            ++s_n[w];
            tc_fence_after();
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_ss(tbase + w * 128, sdesc_add(dQ(w), off), sdesc_add(dK(stage), off), idS, kk > 0);
          }
          mma_commit(bars.sfull(w));
        }
        mma_commit(bars.kempty(stage));
        return true;
      };
      // Record i of the ring: wait until published, read its kind and flags.
      auto take_at = [&](MRec& r, int i) -> bool {
        if (!mbar_wait(bars.infofull(i % kNInfo), (i / kNInfo) & 1, ctl, 20)) return false;
        const int2 kf = *reinterpret_cast<const int2*>(&recs[i % kNInfo]);
        r.kind = kf.x;
        r.flags = kf.y;
        return true;
      };
      MRec rec, nxt;
      int rec_i = 0;
      alive = take_at(rec, rec_i);
      while (alive && rec.kind != kRecStop) {
        // rec is the first record of a unit
        alive = mbar_wait(bars.qfull(), unit_n & 1, ctl, 22);
        if (alive && rec.kind == kRecUnitEnd) {  // a unit without visible tiles
          mma_commit(bars.qempty());
          release(rec_i);
          ++rec_i;
          ++unit_n;
          alive = take_at(rec, rec_i);
          continue;
        }
        int stage = tile_n % C::KST;
        if (alive) alive = issue_S(rec, stage);
        bool first[2] = {true, true};
        bool any_pv[2] = {false, false};
        while (alive) {
          // rec: tile t (record rec_i); nxt: record t + 1 (a tile or the unit end).
          // Order on the tensor pipe: PV0(t), S0(t+1), PV1(t), S1(t+1) with one
          // issuer; with P in columns of its own (PSEP), each issuer sends
          // S_w(t+1) once its softmax has read S_w(t), then PV_w(t).
          const int nxt_i = rec_i + 1;
          if (!take_at(nxt, nxt_i)) { alive = false; break; }
          if (!mbar_wait(bars.vfull(stage), (tile_n / C::KST) & 1, ctl, 23)) { alive = false; break; }
          const int nstage = (tile_n + 1) % C::KST;
          bool nxt_k_ready = false;
          // The unit's last tile: every S (the only MMAs that read Q) is already
          // issued, so at D = 64 (short packed-document units) Q's buffer is
          // released before the last PVs and the next unit's Q tiles load under them.
          if (C::ISSUERS == 2 && nxt.kind != kRecTile) mma_commit(bars.qempty());
          if constexpr (C::PSEP) {
            const int w = mw;
            if (nxt.kind == kRecTile && !(nxt.flags & (w == 0 ? kSkip0 : kSkip1))) {
              if (!mbar_wait(bars.kfull(nstage), ((tile_n + 1) / C::KST) & 1, ctl, 26)) { alive = false; break; }
              if (s_n[w] > 0 && !mbar_wait(bars.sread(w), (s_n[w] - 1) & 1, ctl, 28)) { alive = false; break; }
              ++s_n[w];
              tc_fence_after();
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                mma_ss(tbase + w * 128, sdesc_add(dQ(w), off), sdesc_add(dK(nstage), off), idS, kk > 0);
              }
              mma_commit(bars.sfull(w));
            }
            if (!(rec.flags & (w == 0 ? kSkip0 : kSkip1))) {
              if (first[w]) {
                if (!mbar_wait(bars.ofree(w), ofree_ph[w], ctl, 24)) { alive = false; break; }
                ofree_ph[w] ^= 1;
              }
              if (!mbar_wait(bars.pready(w), pready_ph[w], ctl, 25)) { alive = false; break; }
              pready_ph[w] ^= 1;
              tc_fence_after();
#pragma unroll
              for (int kk = 0; kk < kBN / 16; ++kk)
                mma_ts(tbase + C::TCOL_O + w * D, tbase + C::TCOL_P + w * 64 + kk * 8, sdesc_add(dV(stage), kk * 2048),
                       idO, first[w] ? (kk > 0) : 1);
              mma_commit(bars.pfree(w));
              first[w] = false;
              any_pv[w] = true;
            }
          } else
          for (int w = C::ISSUERS == 2 ? mw : 0; (C::ISSUERS == 2 ? w == mw : w < 2) && alive; ++w) {
            if (!(rec.flags & (w == 0 ? kSkip0 : kSkip1))) {
              if (first[w]) {
                if (!mbar_wait(bars.ofree(w), ofree_ph[w], ctl, 24)) { alive = false; break; }
                ofree_ph[w] ^= 1;
              }
              if (!mbar_wait(bars.pready(w), pready_ph[w], ctl, 25)) { alive = false; break; }
              pready_ph[w] ^= 1;
              tc_fence_after();
#pragma unroll
              for (int kk = 0; kk < kBN / 16; ++kk)
                mma_ts(tbase + C::TCOL_O + w * D, tbase + w * 128 + kk * 8, sdesc_add(dV(stage), kk * 2048), idO,
                       first[w] ? (kk > 0) : 1);
              first[w] = false;
              any_pv[w] = true;
            }
            if (nxt.kind == kRecTile && !(nxt.flags & (w == 0 ? kSkip0 : kSkip1))) {
              if (!nxt_k_ready) {
                if (!mbar_wait(bars.kfull(nstage), ((tile_n + 1) / C::KST) & 1, ctl, 26)) { alive = false; break; }
                tc_fence_after();
                nxt_k_ready = true;
              }
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                mma_ss(tbase + w * 128, sdesc_add(dQ(w), off), sdesc_add(dK(nstage), off), idS, kk > 0);
              }
              mma_commit(bars.sfull(w));
            }
          }
          if (!alive) break;
          mma_commit(bars.vempty(stage));
          if (nxt.kind == kRecTile) mma_commit(bars.kempty(nstage));
          release(rec_i);
          ++tile_n;
          stage = nstage;
          if (nxt.kind != kRecTile) {  // unit end
            for (int w = C::ISSUERS == 2 ? mw : 0; C::ISSUERS == 2 ? w == mw : w < 2; ++w)
              if (any_pv[w]) mma_commit(bars.odone(w));
            if (C::ISSUERS == 1) mma_commit(bars.qempty());
            release(nxt_i);
            rec_i = nxt_i + 1;
            ++unit_n;
            break;
          }
          rec = nxt;
          rec_i = nxt_i;
        }
        if (!alive) break;
        alive = take_at(rec, rec_i);
      }
      if (alive && rec.kind == kRecStop) release(rec_i);
      // Drain: wait for every MMA issued by this thread before TMEM is freed.
      mma_commit(bars.qempty());
      mbar_drain(bars.qempty(), (unit_n & 1), ctl, 27);
    }
    __syncwarp();
  } else if (C::ISSUERS == 1 || warp < 8) {  // with one issuer, every remaining warp (0-7)
    // ------------------------------------------------------------------
    // Softmax warpgroups: w = Q tile, one row per thread
    // ------------------------------------------------------------------
    const int w = warp >> 2;
    const int rl = (warp & 3) * 32 + lane;              // row within the tile
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tbase + lane_base + w * 128;
    const uint32_t tO = tbase + lane_base + C::TCOL_O + w * D;
    const uint32_t tP = C::PSEP ? tbase + lane_base + C::TCOL_P + w * 64 : tS;  // where P_w goes
    int p_n = 0;  // P stores so far (PSEP: each waits for the previous PV_w)
    const float sl2 = P.scale_log2;
    float m_use = -INFINITY, l = 0.f;
    int processed = 0;
    uint32_t sfull_ph = 0, odone_ph = 0;
    int rec_n = 0;
    bool alive = true;
    while (alive) {
      const int slot = rec_n % kNInfo;
      alive = mbar_wait(bars.infofull(slot), (rec_n / kNInfo) & 1, ctl, 30);
      alive = __all_sync(0xffffffffu, alive);
      if (!alive) break;
      const Rec r = recs[slot];
      if (r.kind == kRecStop) {
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.infoempty(slot));
        break;
      }
      const int qrow = r.q0 + w * kBM + rl;
      if (r.kind == kRecTile && !(r.flags & (w == 0 ? kSkip0 : kSkip1))) {
        alive = mbar_wait(bars.sfull(w), sfull_ph, ctl, 31);
        alive = __all_sync(0xffffffffu, alive);
        if (!alive) break;
        sfull_ph ^= 1;
        tc_fence_after();
        uint32_t sr[128];
#pragma unroll
        for (int cq = 0; cq < 4; ++cq) tmem_ld32(tS + cq * 32, sr + cq * 32);
#pragma unroll
        for (int cq = 0; cq < 4; ++cq) tmem_ld_wait(sr + cq * 32);
        if constexpr (C::PSEP) {  // S_w is in registers: its columns may take S_w(t + 1)
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bars.sread(w));
        }
        if (r.flags & (w == 0 ? kMask0 : kMask1)) {
          // keys x < nvis of the tile pass the range and causal rules: the causal
          // block of key kstart + x must not exceed the row's block
          long long lim = r.kvalid;
          if (pb.causal > 0)
            lim = min(lim, ((long long)(qrow + (kCarry ? P.qoff : 0)) / pb.causal + 1) * pb.causal - (r.kstart + (kCarry ? P.koff : 0)));
          int nvis = (int)max(lim, 0LL);
          // With one segment id across the tile's keys (packed documents: the causal
          // diagonal tiles), a row sees all of the tile or none of it, and the 128 key
          // ids need not be read.  Only at D = 64: at D = 128 the extra branch in this
          // 168-register kernel cost ~1 % of the unmasked forward.
          bool uni = false;
          if constexpr (D == 64) uni = pb.seg != nullptr && (r.flags & kKeyUni) != 0;
          if (uni) {
            if (__ldg(pb.seg + (size_t)r.b * pb.S + min(qrow, pb.S - 1)) != r.kseg) nvis = 0;
          }
          if (pb.seg && !uni) {
            const int* ks = (kCarry ? P.kseg : pb.seg) + (size_t)r.b * pb.S + r.kstart;
            const int qseg = __ldg(pb.seg + (size_t)r.b * pb.S + min(qrow, pb.S - 1));
            if (r.kvalid == 128 && ((reinterpret_cast<uintptr_t>(ks) & 15u) == 0)) {
              // the tile's 128 key ids in 16-byte loads (the same addresses for every row: L1 broadcast)
#pragma unroll
              for (int x4 = 0; x4 < 32; ++x4) {
                const int4 sv = __ldg(reinterpret_cast<const int4*>(ks) + x4);
                const int e[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const int x = 4 * x4 + i;
                  if (!(x < nvis && e[i] == qseg)) sr[x] = __float_as_uint(-INFINITY);
                }
              }
            } else {
#pragma unroll
              for (int x = 0; x < 128; ++x) {
                const bool vis = x < nvis && __ldg(ks + min(x, r.kvalid - 1)) == qseg;
                if (!vis) sr[x] = __float_as_uint(-INFINITY);
              }
            }
          } else {
#pragma unroll
            for (int x = 0; x < 128; ++x)
              if (!(x < nvis)) sr[x] = __float_as_uint(-INFINITY);
          }
        }
        // row max: eight independent chains of three-input max
        float mx8[8];
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) mx8[c8] = fmaxf(__uint_as_float(sr[c8]), __uint_as_float(sr[c8 + 8]));
#pragma unroll
        for (int x = 16; x < 128; x += 16) {
#pragma unroll
          for (int c8 = 0; c8 < 8; ++c8)
            mx8[c8] = fmax3(mx8[c8], __uint_as_float(sr[x + c8]), __uint_as_float(sr[x + 8 + c8]));
        }
        const float mx = fmaxf(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(fmax3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
        const float m_tile = mx * sl2;
        float corr = 1.f;
        bool resc = false;
        if (m_tile > m_use + kRescaleThreshold) {
          if (m_use != -INFINITY) {
            corr = ex2_approx(m_use - m_tile);
            resc = true;
          }
          m_use = m_tile;
        }
        const float mb = (m_use == -INFINITY) ? 0.f : m_use;
        if constexpr (C::PSEP) {  // the previous PV_w has read P_w and written O_w
          if (p_n > 0) {
            alive = __all_sync(0xffffffffu, mbar_wait(bars.pfree(w), (p_n - 1) & 1, ctl, 33));
            if (!alive) break;
          }
          ++p_n;
          tc_fence_after();
        }
        float rs[4] = {0.f, 0.f, 0.f, 0.f};  // two packed accumulators
        uint32_t pk[64];
#pragma unroll
        for (int x = 0; x < 64; ++x) {
          float a0, a1;
          fma_f32x2(a0, a1, __uint_as_float(sr[2 * x]), __uint_as_float(sr[2 * x + 1]), sl2, sl2, -mb, -mb);
          const float p0 = ex2_approx(a0);
          const float p1 = ex2_approx(a1);
          const int acc = (x & 1) * 2;
          add_f32x2(rs[acc], rs[acc + 1], rs[acc], rs[acc + 1], p0, p1);
          pk[x] = pack_bf16x2(p0, p1);
          if (x == 31) tmem_st32(tP, pk);  // first half of P goes out while the rest is computed
        }
        tmem_st32(tP + 32, pk + 32);
        l = l * corr + ((rs[0] + rs[1]) + (rs[2] + rs[3]));
        if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
          for (int cq = 0; cq < D / 32; ++cq) {
            uint32_t o[32];
            tmem_ld32(tO + cq * 32, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * corr);
            tmem_st32(tO + cq * 32, o);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.pready(w));
        ++processed;
      } else if (r.kind == kRecUnitEnd) {
        if (processed > 0) {
          alive = mbar_wait(bars.odone(w), odone_ph, ctl, 32);
          alive = __all_sync(0xffffffffu, alive);
          if (!alive) break;
          odone_ph ^= 1;
          tc_fence_after();
          const int qv = w == 0 ? r.qvalid0 : r.qvalid1;
          const bool store = rl < qv;
          if constexpr (!kCarry) {
            const float inv = l > 0.f ? 1.f / l : 0.f;
            __nv_bfloat16* orow = P.out + (((size_t)r.b * pb.S + qrow) * pb.H + r.h) * D;
#pragma unroll
            for (int cq = 0; cq < D / 32; ++cq) {
              uint32_t o[32];
              tmem_ld32(tO + cq * 32, o);
              tmem_ld_wait(o);
              if (store) {
                uint4* dst = reinterpret_cast<uint4*>(orow + cq * 32);
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4) {
                  uint4 val;
                  val.x = pack_bf16x2(__uint_as_float(o[v4 * 8 + 0]) * inv, __uint_as_float(o[v4 * 8 + 1]) * inv);
                  val.y = pack_bf16x2(__uint_as_float(o[v4 * 8 + 2]) * inv, __uint_as_float(o[v4 * 8 + 3]) * inv);
                  val.z = pack_bf16x2(__uint_as_float(o[v4 * 8 + 4]) * inv, __uint_as_float(o[v4 * 8 + 5]) * inv);
                  val.w = pack_bf16x2(__uint_as_float(o[v4 * 8 + 6]) * inv, __uint_as_float(o[v4 * 8 + 7]) * inv);
                  dst[v4] = val;
                }
              }
            }
            if (store)
              P.lse[((size_t)r.b * pb.H + r.h) * pb.S + qrow] =
                  l > 0.f ? (m_use + __log2f(l)) * 0.69314718055994531f : -INFINITY;
          } else {
            // Ring step: merge this block's (out, lse) into the running carry, the
            // lazy-softmax update at block granularity (code walk-through page §2):
            // with L the log2-sum-exp of the carry and of this block and M their
            // max, carry = carry * 2^(L_old - M) / Z + out_blk * 2^(L_blk - M) / Z,
            // Z = 2^(L_old - M) + 2^(L_blk - M), lse = (M + log2 Z) ln 2.  A row
            // with no visible key in this block leaves its carry unchanged.
            const bool merge = store && l > 0.f;
            float wo = 0.f, wn = 0.f;
            const size_t lidx = ((size_t)r.b * pb.H + r.h) * pb.S + qrow;
            if (merge) {
              const float L_blk = m_use + __log2f(l);
              const float L_old = P.lse_carry[lidx] * 1.4426950408889634f;  // -inf stays -inf
              const float M = fmaxf(L_old, L_blk);
              const float a = ex2_approx(L_old - M);  // 0 for an empty carry
              const float bb = ex2_approx(L_blk - M);
              const float z = a + bb;
              wo = a / z;
              wn = bb / (z * l);
              P.lse_carry[lidx] = (M + __log2f(z)) * 0.69314718055994531f;
            }
            float* oc = P.o_carry + (((size_t)r.b * pb.S + qrow) * pb.H + r.h) * D;
#pragma unroll
            for (int cq = 0; cq < D / 32; ++cq) {
              uint32_t o[32];
              tmem_ld32(tO + cq * 32, o);
              tmem_ld_wait(o);
              if (merge) {
                float4* dst = reinterpret_cast<float4*>(oc + cq * 32);
#pragma unroll
                for (int v4 = 0; v4 < 8; ++v4) {
                  float4 c4 = dst[v4];
                  c4.x = c4.x * wo + __uint_as_float(o[v4 * 4 + 0]) * wn;
                  c4.y = c4.y * wo + __uint_as_float(o[v4 * 4 + 1]) * wn;
                  c4.z = c4.z * wo + __uint_as_float(o[v4 * 4 + 2]) * wn;
                  c4.w = c4.w * wo + __uint_as_float(o[v4 * 4 + 3]) * wn;
                  dst[v4] = c4;
                }
              }
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bars.ofree(w));
        }
        m_use = -INFINITY;
        l = 0.f;
        processed = 0;
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

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

}  // namespace

// [B, S, H, D] bf16 tensor map with a 64-element x 128-row box, 128B swizzle.
bool make_tile_map(CUtensorMap* m, const void* ptr, const Problem& p, int rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[4] = {(cuuint64_t)p.D, (cuuint64_t)p.H, (cuuint64_t)p.S, (cuuint64_t)p.B};
  cuuint64_t strides[3] = {(cuuint64_t)p.D * 2, (cuuint64_t)p.H * p.D * 2, (cuuint64_t)p.S * p.H * p.D * 2};
  cuuint32_t box[4] = {64, 1, (cuuint32_t)rows, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// A zeroed 4-byte counter for one call, or null (stream capture, or no pool).
static int* take_unit_counter(const Ctx& c) {
  static std::mutex mu;
  static cudaMemPool_t pools[256];
  static bool tried[256];
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(c.stream, &cs) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  if (cs != cudaStreamCaptureStatusNone || c.device < 0 || c.device >= 256) return nullptr;
  cudaMemPool_t pool = nullptr;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!tried[c.device]) {
      tried[c.device] = true;
      cudaMemPoolProps props = {};
      props.allocType = cudaMemAllocationTypePinned;
      props.handleTypes = cudaMemHandleTypeNone;
      props.location.type = cudaMemLocationTypeDevice;
      props.location.id = c.device;
      if (cudaMemPoolCreate(&pools[c.device], &props) == cudaSuccess) {
        uint64_t keep = UINT64_MAX;  // keep the pool's few bytes reserved between calls
        cudaMemPoolSetAttribute(pools[c.device], cudaMemPoolAttrReleaseThreshold, &keep);
      } else {
        pools[c.device] = nullptr;
      }
      (void)cudaGetLastError();
    }
    pool = pools[c.device];
  }
  if (!pool) return nullptr;
  void* p = nullptr;
  if (cudaMallocFromPoolAsync(&p, 16, pool, c.stream) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  if (cudaMemsetAsync(p, 0, 16, c.stream) != cudaSuccess) {
    (void)cudaGetLastError();
    cudaFreeAsync(p, c.stream);
    (void)cudaGetLastError();
    return nullptr;
  }
  return static_cast<int*>(p);
}

template <int D, bool kCarry, bool kLog>
static cudaError_t launch_fwd_bf16_d(const FwdArgs& a, const Ctx& c, uint64_t* launches, const char** why) {
  using Cf = Cfg<D>;
  const Problem& p = a.p;
  CUtensorMap mq, mk, mv;
  if (!make_tile_map(&mq, a.q, p, kBM) || !make_tile_map(&mk, a.k, p, kBN) || !make_tile_map(&mv, a.v, p, kBN)) {
    *why = "cuTensorMapEncodeTiled failed (driver entry point unavailable or tensor rejected)";
    return cudaSuccess;
  }
  FwdParams P;
  P.p = p;
  P.out = (__nv_bfloat16*)a.out;
  P.lse = a.lse;
  P.qoff = a.qoff;
  P.koff = a.koff;
  P.kseg = a.kseg ? a.kseg : p.seg;
  P.o_carry = a.o_carry;
  P.lse_carry = a.lse_carry;
  P.vlog = a.vlog;
  P.vlog_cap = a.vlog_cap;
  P.status = c.status;
  P.limit_ns = c.limit_ns;
  P.tiles_per_shard = (p.Ssh + kBN - 1) / kBN;
  P.pairs_per_shard = (P.tiles_per_shard + 1) / 2;
  P.num_units = p.B * p.H * p.N * P.pairs_per_shard;
  P.scale_log2 = (float)(1.4426950408889634 / sqrt((double)p.D));
  static std::atomic<bool> attr_set[256];  // idempotent attribute; atomic so threads may race
  if (!attr_set[c.device]) {
    cudaError_t e = cudaFuncSetAttribute(fwd_bf16_kernel<D, kCarry, kLog>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)Cf::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[c.device] = true;
  }
  const int per_head = p.N * P.pairs_per_shard;
  const int num_super = (P.num_units / per_head) * ((per_head + 1) / 2);  // balanced unit pairs
  // A unit counter of this call's own, from a stream-ordered pool on the caller's
  // stream, so that calls running at the same time never share one.  Under stream
  // capture the static pairs are used instead (same results: each unit is computed
  // whole by one CTA either way).
  P.unit_counter = take_unit_counter(c);
  {  // heads whose K and V (2 * S * D bf16 each) fit in 48 MB of L2 together, or in
     // 128 MB when one head's take 16 MB or less: short heads have few units each,
     // and a small last group cannot balance its longest units, so the SMs idle at
     // the end of the launch; long heads past 48 MB only re-read K and V from DRAM
    const long long kv = 2LL * p.S * p.D * 2;
    const long long budget = kv <= (16LL << 20) ? (128LL << 20) : (48LL << 20);
    P.group_heads = (int)std::max(1LL, std::min((long long)p.B * p.H, budget / kv));
  }
  const int grid = std::min(c.num_sms, P.unit_counter ? P.num_units : num_super);
  fwd_bf16_kernel<D, kCarry, kLog><<<grid, Cf::THREADS, Cf::SMEM, c.stream>>>(mq, mk, mv, P);
  *launches += 1;
  cudaError_t e = cudaGetLastError();
  if (P.unit_counter) {
    cudaError_t ef = cudaFreeAsync(P.unit_counter, c.stream);
    if (e == cudaSuccess) e = ef;
  }
  return e;
}

template <int D>
static cudaError_t launch_fwd_bf16_dd(const FwdArgs& a, const Ctx& c, uint64_t* launches, const char** why) {
  // separate kernels with and without the ring-step carry and the visit log, so
  // that the plain forward carries no code of either
  const bool carry = a.o_carry != nullptr, log = a.vlog != nullptr;
  if (carry) return log ? launch_fwd_bf16_d<D, true, true>(a, c, launches, why)
                        : launch_fwd_bf16_d<D, true, false>(a, c, launches, why);
  return log ? launch_fwd_bf16_d<D, false, true>(a, c, launches, why)
             : launch_fwd_bf16_d<D, false, false>(a, c, launches, why);
}

cudaError_t launch_fwd_bf16(const FwdArgs& a, const Ctx& c, uint64_t* launches, const char** why) {
  if (a.p.D == 64) return launch_fwd_bf16_dd<64>(a, c, launches, why);
  if (a.p.D == 128) return launch_fwd_bf16_dd<128>(a, c, launches, why);
  *why = "bf16 head_dim must be 64 or 128";
  return cudaSuccess;
}

}  // namespace ra
