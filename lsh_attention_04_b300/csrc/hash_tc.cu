// hash_tc.cu -- tensor-core angular LSH (tcgen05).  Placeholder until the kernel lands.
#include "internal.cuh"

namespace lsh {
bool hash_tc_supported(const Problem &) { return false; }
size_t hash_tc_pack_bytes(const Problem &) { return 0; }
int hash_tc_launches(const Problem &) { return 0; }
cudaError_t hash_tc(const Problem &, const void *, const void *, void *, int32_t *, float *,
                    StatusBlock *, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace lsh
