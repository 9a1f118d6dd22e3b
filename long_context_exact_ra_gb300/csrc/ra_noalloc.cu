// ra_noalloc.cu — ra_bwd_noalloc: the backward for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the point
// where they run the backward: code inside a memory-capped or pre-planned
// arena, host runtimes that forbid allocation after start-up, or callers that
// must not synchronize the device (cudaMalloc and cudaFree can).  ra_bwd needs
// a scratch workspace from its caller; this entry point instead uses a fixed
// scratch array that lives in the library's device image.  It is allocated
// when this file's device code is first loaded on a device and held by every
// GPU that uses it until the process exits.
//
// The array is shared by every call on a device and keeps the last call's
// contents; the backward's preprocess kernel clears the part that must start
// at zero (the fp32 dQ accumulator) on every call.  Calls whose work overlaps
// on the GPU (different streams, no ordering between them) race on the array.
#include <cstdio>

#include "ra.h"
#include "ra_internal.h"

#define RA_API extern "C" __attribute__((visibility("default")))

namespace ra {
namespace {

static __device__ __align__(256) unsigned char g_bwd_scratch[RA_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array on the current device, looked up on every
// call with that device current.  In host code `g_bwd_scratch` names a host
// stand-in, not device memory, so only this address may be passed to kernels.
// The lookup is not cached: after a device reset the array is loaded again at
// a new address, and a cached one would point at memory the library no longer
// owns.  Once the array is loaded the lookup allocates nothing.
ra_status scratch_address(void** out) {
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_bwd_scratch);
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof(msg), "cudaGetSymbolAddress(no-alloc scratch): %s", cudaGetErrorString(e));
    return set_last_error(RA_ERR_CUDA, msg);
  }
  *out = p;
  return RA_OK;
}

}  // namespace
}  // namespace ra

using namespace ra;

RA_API size_t ra_bwd_noalloc_max_scratch(void) { return (size_t)RA_NOALLOC_SCRATCH_BYTES; }

RA_API ra_status ra_bwd_noalloc(const void* q, const void* k, const void* v, const void* out, const float* lse,
                                const void* dout, const int32_t* segment_ids, int causal_block_size,
                                int num_shards, int query_chunk_size, int key_chunk_size, int batch, int seq,
                                int heads, int head_dim, ra_dtype dtype, void* dq, void* dk, void* dv,
                                void* stream) {
  const size_t need = ra_bwd_workspace_size(batch, seq, heads, head_dim, dtype);
  if (need > (size_t)RA_NOALLOC_SCRATCH_BYTES) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "problem needs %zu bytes of backward scratch; the built-in array holds %zu "
             "(use ra_bwd with a caller-provided workspace)",
             need, (size_t)RA_NOALLOC_SCRATCH_BYTES);
    return set_last_error(RA_ERR_INVALID_ARG, msg);
  }
  void* scratch = nullptr;
  if (seq > 0) {
    ra_status s = scratch_address(&scratch);
    if (s != RA_OK) return s;
  }
  return ra_bwd(q, k, v, out, lse, dout, segment_ids, causal_block_size, num_shards, query_chunk_size,
                key_chunk_size, batch, seq, heads, head_dim, dtype, dq, dk, dv, scratch,
                (size_t)RA_NOALLOC_SCRATCH_BYTES, stream);
}
