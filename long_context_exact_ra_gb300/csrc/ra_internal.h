// ra_internal.h — argument bundles shared by the C ABI layer and the kernel launchers.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "ra.h"

namespace ra {

// One attention problem: [B, S, H, D] tensors split into N contiguous virtual shards.
struct Problem {
  int B, S, H, D;
  int N;       // num_shards
  int Ssh;     // S / N
  int causal;  // causal_block_size (0 = non-causal)
  const int32_t* seg;  // [B, S] or nullptr
};

// Optional extras shared by the forward and backward calls.
struct CallExtras {
  // Positions: query row r sits at r + qoff, key row x at x + koff (see the
  // ring-step entry points); kseg = key rows' segment ids (null: p.seg).
  int qoff = 0, koff = 0;
  const int32_t* kseg = nullptr;
  int* vlog = nullptr;  // debug visit log (ra_debug_visitlog), or null
  int vlog_cap = 0;     // entries it holds
};

struct FwdArgs : CallExtras {
  Problem p;
  const void* q;
  const void* k;
  const void* v;
  void* out;
  float* lse;
  float* o_carry = nullptr;    // ring step: fp32 running output (then out/lse are unused)
  float* lse_carry = nullptr;  // ring step: running lse
};

// What a backward call runs.
enum BwdStage : int {
  kBwdWhole = 0,      // preprocess, main kernel, finalize (ra_bwd)
  kBwdRingBegin = 1,  // preprocess only (Delta, lse*log2(e); dQ accumulator zeroed)
  kBwdRingStep = 2,   // main kernel with fp32 dK/dV carries
  kBwdRingEnd = 3,    // finalize only (dq from the accumulator)
};

struct BwdArgs : CallExtras {
  Problem p;
  int stage = kBwdWhole;
  const void* q;
  const void* k;
  const void* v;
  const void* out;
  const float* lse;
  const void* dout;
  void* dq;
  void* dk;
  void* dv;
  float* dq_accum;  // [B, S, H, D] fp32 scratch (bf16 path)
  float* delta;     // fp32 path: [B, H, S] Delta; bf16 path: float2 (lse*log2(e), Delta) rows of bwd_row_pitch
  int* unit_counter;  // bf16 path: the main kernel's unit counter (in the workspace)
  float* dk_carry = nullptr;  // ring step: fp32 dK accumulator of the key/value block
  float* dv_carry = nullptr;  // ring step: fp32 dV accumulator
};

// Launch context: device facts and the device status word.
struct Ctx {
  int device;
  int num_sms;
  int* status;        // device address of the status word
  uint64_t limit_ns;  // bounded-wait limit
  cudaStream_t stream;
};

// Decoding T new tokens against a [B, S, H, D] KV cache.
struct DecodeArgs {
  int B, T, S, H, D, N, causal;
  bool bf16;
  const void* q;             // [B, T, H, D]
  const void* k;             // [B, S, H, D]
  const void* v;             // [B, S, H, D]
  const int32_t* cache_idx;  // [B]
  const int32_t* qseg;       // [B, T] or nullptr
  const int32_t* kseg;       // [B, S] or nullptr
  void* out;                 // [B, T, H, D]
  float* lse;                // [B, H, T]
  void* workspace;           // decode_workspace_bytes(...)
};

// How the cache is cut into work items (a function of the shape only, so that
// the workspace size does not depend on the device).
struct DecodeSplit {
  int split_len;        // keys per work item
  int items_per_shard;  // ceil((S / N) / split_len)
  int P;                // partials per (b, h, token) = N * items_per_shard
};
DecodeSplit decode_split(int B, int T, int S, int H, int num_shards);
size_t decode_workspace_bytes(int B, int T, int S, int H, int D, int num_shards);
cudaError_t launch_decode(const DecodeArgs& a, const Ctx& c, uint64_t* launches);

// Blockwise feed-forward: out = max(0, x w1^T + b1) w2^T + b2, chunk by chunk.
struct FfnArgs {
  int B, L, Dm, F, chunk;
  const void* x;    // [B, L, Dm] bf16
  const void* w1;   // [F, Dm] bf16
  const float* b1;  // [F] or nullptr
  const void* w2;   // [Dm, F] bf16
  const float* b2;  // [Dm] or nullptr
  void* out;        // [B, L, Dm] bf16
  void* hidden;     // [min(B*L, chunk), F] bf16 scratch
};
size_t ffn_workspace_bytes(long long rows, int chunk_size, int ffn_dim);
cudaError_t launch_ffn(const FfnArgs& a, const Ctx& c, uint64_t* launches, const char** why);

// Launchers.  Each returns the CUDA error of its launch(es) and adds the
// number of kernels it launched to *launches.
cudaError_t launch_fwd_f32(const FwdArgs& a, const Ctx& c, uint64_t* launches);
cudaError_t launch_bwd_f32(const BwdArgs& a, const Ctx& c, uint64_t* launches);
cudaError_t launch_fwd_bf16(const FwdArgs& a, const Ctx& c, uint64_t* launches, const char** why);
cudaError_t launch_bwd_bf16(const BwdArgs& a, const Ctx& c, uint64_t* launches, const char** why);
cudaError_t launch_selftest_timeout(const Ctx& c, uint64_t* launches);
// dst[i] = bf16(src[i] * scale), i < count (count a multiple of 4, both 16-byte aligned).
cudaError_t launch_cast_bf16(const float* src, void* dst, size_t count, float scale, const Ctx& c,
                             uint64_t* launches);

// Sets the calling thread's ra_last_error() message and returns s.
ra_status set_last_error(ra_status s, const char* msg);

// Scratch layout of the bf16 backward (byte offsets into the caller's workspace):
// the fp32 dQ accumulator, then (lse*log2(e), Delta) float2 pairs per (b, h) row
// with an even row pitch (16-byte aligned pairs of entries) and a tail pad so
// that a 130-entry bulk copy starting at any even index stays inside ...
constexpr int kBwdVecEntries = 130;
inline int bwd_row_pitch(int S) { return S + (S & 1); }
inline size_t bwd_delta_offset(int B, int S, int H, int D) {
  size_t dq = (size_t)B * S * H * D * sizeof(float);
  return (dq + 255) & ~(size_t)255;
}
// ... and last a 256-byte slot whose first word is the main kernel's unit counter
// (zeroed by the preprocess kernel).
inline size_t bwd_counter_offset(int B, int S, int H, int D) {
  const size_t vec = ((size_t)B * H * bwd_row_pitch(S) + kBwdVecEntries) * 2 * sizeof(float);
  return bwd_delta_offset(B, S, H, D) + ((vec + 255) & ~(size_t)255);
}
inline size_t bwd_workspace_bytes(int B, int S, int H, int D) { return bwd_counter_offset(B, S, H, D) + 256; }

}  // namespace ra
