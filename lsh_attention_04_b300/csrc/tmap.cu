// tmap.cu -- host-side encoding of TMA tensor maps through the driver entry point
// (the library does not link libcuda directly; the runtime hands out the driver symbol).
#include <mutex>

#include "sm100.cuh"

namespace lsh {
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver function pointer, looked up once per process (read-only afterwards).
EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeTiledFn)p;
    });
    return fn;
}

}  // namespace

bool make_tmap_2d_bf16(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                       uint32_t box_cols, uint32_t box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace lsh

#ifdef LSH_WAIT_PROF
namespace lsh {
namespace sm100 {
__device__ unsigned long long g_wait_cycles[4096];
__device__ unsigned long long g_wait_count[4096];
}  // namespace sm100
}  // namespace lsh
// Profiling build only: copy (and clear) the per-code wait cycles and counts.
extern "C" int lsh_debug_wait_profile(unsigned long long *cycles, unsigned long long *counts)
{
    cudaDeviceSynchronize();
    if (cudaMemcpyFromSymbol(cycles, lsh::sm100::g_wait_cycles, sizeof(unsigned long long) * 4096) != cudaSuccess) return 1;
    if (cudaMemcpyFromSymbol(counts, lsh::sm100::g_wait_count, sizeof(unsigned long long) * 4096) != cudaSuccess) return 1;
    static unsigned long long zero[4096];
    cudaMemcpyToSymbol(lsh::sm100::g_wait_cycles, zero, sizeof(zero));
    cudaMemcpyToSymbol(lsh::sm100::g_wait_count, zero, sizeof(zero));
    return 0;
}
#endif
