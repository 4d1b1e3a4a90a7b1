// attn_tc.cu -- tensor-core chunk attention (tcgen05).  Placeholder until the kernel lands.
#include "internal.cuh"

namespace lsh {
bool attn_tc_supported(const Problem &) { return false; }
cudaError_t attn_tc(const Problem &, const void *, const void *, const int32_t *, const int32_t *,
                    const int32_t *, const float *, void *, float *, StatusBlock *, cudaStream_t)
{ return cudaErrorNotSupported; }
}  // namespace lsh
