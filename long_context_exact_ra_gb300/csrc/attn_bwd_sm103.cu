// attn_bwd_sm103.cu — bf16 backward (placeholder until the tensor-core kernel lands).
#include "ra_internal.h"

namespace ra {
cudaError_t launch_bwd_bf16(const BwdArgs&, const Ctx&, uint64_t*, const char** why) {
  *why = "bf16 backward is not built yet";
  return cudaSuccess;
}
}  // namespace ra
