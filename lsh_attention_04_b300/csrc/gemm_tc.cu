// gemm_tc.cu -- the dense projections of the reversible block on the tcgen05 tensor cores:
// C = epilogue(A W^T) with A [M][K] and W [N][K] bf16 (both K contiguous), fp32
// accumulation in tensor memory.
//
// Persistent CTAs walk 128 x 256 output tiles (tile t = m_block * n_blocks + n_block, so
// neighbouring CTAs share A's row block in L2; a last tile 128 columns wide when
// N % 256 = 128 reads zeros past W's last row and stores only its live columns).  Warp
// roles (6 warps):
//   0-3  epilogue: warp w reads TMEM lanes 32w .. 32w+31 (one output row per thread),
//        32 columns at a time, and applies bias, ReLU and a residual (out = res + s * x),
//        writing fp32 and/or bf16, row-major or split into heads [B][H][L][d];
//   4    producer: TMA loads of 64-column tiles of A (128 rows) and W (256 rows),
//        128-byte swizzle, into a 4-stage ring of 48 KB stages;
//   5    MMA issuer and TMEM owner: 4 tcgen05.mma (M=128, N=256, K=16) per stage into one
//        of two 256-column accumulators (all 512 columns), so the epilogue of a tile
//        overlaps the MMAs of the next one.  At N = 256 an MMA reads 12 KB of operands in
//        128 cycles, inside the shared-memory bandwidth (N = 128 would need all of it).
// Every wait is bounded (sm100::wait); on a timeout the kernel records where in the
// workspace status block and winds down.
#include "sm100.cuh"

namespace lsh {
namespace {

using namespace sm100;

constexpr int kTM = 128, kTN = 256, kTK = 64;
constexpr int kStages = 4;
constexpr int kStageBytes = (kTM + kTN) * kTK * 2;   // 48 KB
constexpr int kGemmThreads = 6 * 32;

struct __align__(8) GemmBarriers {
    uint64_t full[kStages], empty[kStages];
    uint64_t acc_full[2], acc_empty[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
};

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__global__ void __launch_bounds__(kGemmThreads, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap amap, const __grid_constant__ CUtensorMap wmap,
               GemmArgs g, StatusBlock *status)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ GemmBarriers sb;
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int *abort_flag = &sb.abort_flag;
    const int m_blocks = (g.M + kTM - 1) / kTM, n_blocks = (g.N + kTN - 1) / kTN, k_steps = g.K / kTK;
    const int n_tiles = m_blocks * n_blocks;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sb.full[s], 1);
            mbar_init(&sb.empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sb.acc_full[b], 1);
            mbar_init(&sb.acc_empty[b], 128);
        }
        mbar_init(&sb.mma_done, 1);
        sb.abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 5) tmem_alloc(&sb.tmem_base, 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = sb.tmem_base;

    if (warp == 4) {
        // ---------------- producer
        if (lane == 0) {
            prefetch_tmap(&amap);
            prefetch_tmap(&wmap);
            int it = 0;
            for (int t = blockIdx.x; t < n_tiles; t += gridDim.x) {
                const int m0 = (t / n_blocks) * kTM, n0 = (t % n_blocks) * kTN;
                bool ok = true;
                for (int kb = 0; kb < k_steps; ++kb, ++it) {
                    const int s = it % kStages;
                    if (!(ok = wait(&sb.empty[s], ((it / kStages) & 1) ^ 1, abort_flag, status, 0x801)))
                        break;
                    uint8_t *st = smem + s * kStageBytes;
                    mbar_expect_tx(&sb.full[s], kStageBytes);
                    tma_load_2d(st, &amap, kb * kTK, m0, &sb.full[s]);
                    tma_load_2d(st + kTM * kTK * 2, &wmap, kb * kTK, n0, &sb.full[s]);
                }
                if (!ok) break;
            }
            // wind-down: the last fills have landed before the CTA exits
            for (int k = 1; k <= kStages && it - k >= 0; ++k) {
                const int i2 = it - k, s = i2 % kStages;
                int dummy = 0;
                wait(&sb.full[s], (i2 / kStages) & 1, &dummy, status, 0x802);
            }
        }
    } else if (warp == 5) {
        // ---------------- MMA issuer (whole converged warp; one lane elected per MMA)
        const uint32_t idesc = idesc_bf16(kTM, kTN, 0, 0);
        const uint32_t sbase = smem_u32(smem);
        int it = 0, tc = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x, ++tc) {
            const int b = tc & 1;
            if (!(ok = wait_w(&sb.acc_empty[b], ((tc >> 1) & 1) ^ 1, abort_flag, status, 0x803))) break;
            fence_after_sync();
            for (int kb = 0; kb < k_steps; ++kb, ++it) {
                const int s = it % kStages;
                if (!(ok = wait_w(&sb.full[s], (it / kStages) & 1, abort_flag, status, 0x804))) break;
                fence_after_sync();
                const uint32_t sa = sbase + s * kStageBytes, sw = sa + kTM * kTK * 2;
#pragma unroll
                for (int ks = 0; ks < kTK / 16; ++ks)
                    mma_ss(tmem + b * kTN, smem_desc(sa + 32 * ks, 16, 1024),
                           smem_desc(sw + 32 * ks, 16, 1024), idesc, (kb | ks) != 0);
                mma_commit(smem_u32(&sb.empty[s]));
            }
            if (!ok) break;
            mma_commit(smem_u32(&sb.acc_full[b]));
        }
        mma_commit(smem_u32(&sb.mma_done));
        int dummy = 0;
        wait_w(&sb.mma_done, 0, &dummy, status, 0x805);
    } else {
        // ---------------- epilogue: thread = output row (TMEM lane)
        const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
        int tc = 0;
        for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++tc) {
            const int b = tc & 1;
            const int m0 = (t / n_blocks) * kTM, n0 = (t % n_blocks) * kTN;
            const bool w_ok = wait(&sb.acc_full[b], (tc >> 1) & 1, abort_flag, status, 0x806);
            if (!__all_sync(0xffffffffu, w_ok)) break;
            fence_after_sync();
            const int m = m0 + warp * 32 + lane;
            const bool live = m < g.M;
            for (int q = 0; q < kTN / 32; ++q) {
                if (n0 + 32 * q >= g.N) break;               // past N: a half-width last tile
                uint32_t v[32];
                tmem_ld32(tl + b * kTN + 32 * q, v);
                tmem_wait_ld(v);
                const int n = n0 + 32 * q;
                float x[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    float y = __uint_as_float(v[j]);
                    if (g.bias) y += __ldg(g.bias + n + j);
                    if (g.relu) y = fmaxf(y, 0.f);
                    x[j] = y;
                }
                if (!live) continue;
                if (g.res) {
                    const float4 *r = reinterpret_cast<const float4 *>(g.res + (size_t)m * g.N + n);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float4 rv = __ldg(r + j);
                        x[4 * j] = rv.x + g.res_sign * x[4 * j];
                        x[4 * j + 1] = rv.y + g.res_sign * x[4 * j + 1];
                        x[4 * j + 2] = rv.z + g.res_sign * x[4 * j + 2];
                        x[4 * j + 3] = rv.w + g.res_sign * x[4 * j + 3];
                    }
                }
                if (g.out_f32) {
                    float4 *o = reinterpret_cast<float4 *>(g.out_f32 + (size_t)m * g.N + n);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        o[j] = make_float4(x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
                }
                if (g.out_bf16) {
                    // row-major, or head-split: row m = (b, l), column n = (h, c) goes to
                    // [b][h][l][c] (a 32-column batch stays inside one head)
                    size_t base;
                    if (g.split_heads) {
                        const int bb = m / g.split_L, l = m % g.split_L;
                        const int h = n / g.split_d, c = n % g.split_d;
                        base = (((size_t)bb * (g.N / g.split_d) + h) * g.split_L + l) * g.split_d + c;
                    } else {
                        base = (size_t)m * g.N + n;
                    }
                    uint4 *o = reinterpret_cast<uint4 *>(g.out_bf16 + base);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        o[j] = make_uint4(pack2(x[8 * j], x[8 * j + 1]), pack2(x[8 * j + 2], x[8 * j + 3]),
                                          pack2(x[8 * j + 4], x[8 * j + 5]), pack2(x[8 * j + 6], x[8 * j + 7]));
                }
            }
            fence_before_sync();
            mbar_arrive(&sb.acc_empty[b]);
        }
    }

    fence_before_sync();
    __syncthreads();
    if (warp == 5) {
        __syncwarp();
        fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

bool gemm_tc_supported(int M, int N, int K)
{
    return M > 0 && N > 0 && K > 0 && N % 128 == 0 && K % kTK == 0;
}

cudaError_t gemm_tc(const GemmArgs &g, StatusBlock *status, cudaStream_t st)
{
    if (!gemm_tc_supported(g.M, g.N, g.K)) return cudaErrorInvalidValue;
    CUtensorMap amap, wmap;
    if (!make_tmap_2d_bf16(&amap, g.A, (uint64_t)g.M, (uint64_t)g.K, kTK, kTM) ||
        !make_tmap_2d_bf16(&wmap, g.W, (uint64_t)g.N, (uint64_t)g.K, kTK, kTN))
        return cudaErrorNotSupported;
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int tiles = ((g.M + kTM - 1) / kTM) * ((g.N + kTN - 1) / kTN);
    const int grid = tiles < sms ? tiles : sms;
    const size_t smem = 1024 + (size_t)kStages * kStageBytes;
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    gemm_tc_kernel<<<grid, kGemmThreads, smem, st>>>(amap, wmap, g, status);
    return cudaGetLastError();
}

}  // namespace lsh

extern "C" lsh_status_t lsh_gemm_bf16(const void *A, const void *W, int M, int N, int K,
                                      const float *bias, int relu, const float *res,
                                      float res_sign, float *out_f32, void *out_bf16,
                                      int split_L, int split_d, void *workspace,
                                      size_t workspace_bytes, void *stream)
{
    using namespace lsh;
    const auto a16 = [](const void *p) { return ((uintptr_t)p) % 16 == 0; };
    if (!A || !W || !a16(A) || !a16(W) || (!out_f32 && !out_bf16)) return LSH_ERR_INVALID_ARGUMENT;
    if (!a16(res) || !a16(out_f32) || !a16(out_bf16) || ((uintptr_t)bias) % 4 != 0)
        return LSH_ERR_INVALID_ARGUMENT;
    if (M <= 0 || N <= 0 || K <= 0 || (relu != 0 && relu != 1)) return LSH_ERR_INVALID_ARGUMENT;
    if (split_L < 0 || split_d < 0 || (split_L == 0) != (split_d == 0)) return LSH_ERR_INVALID_ARGUMENT;
    if (split_L > 0 && (!out_bf16 || M % split_L != 0 || N % split_d != 0 || split_d % 32 != 0))
        return LSH_ERR_INVALID_ARGUMENT;
    if (!workspace || ((uintptr_t)workspace) % 256 != 0) return LSH_ERR_INVALID_ARGUMENT;
    if (!gemm_tc_supported(M, N, K)) return LSH_ERR_UNSUPPORTED;
    if (workspace_bytes < sizeof(StatusBlock)) return LSH_ERR_WORKSPACE_TOO_SMALL;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaMemsetAsync(workspace, 0, sizeof(StatusBlock), st) != cudaSuccess) return LSH_ERR_CUDA;
    GemmArgs g;
    g.A = (const __nv_bfloat16 *)A; g.W = (const __nv_bfloat16 *)W;
    g.M = M; g.N = N; g.K = K;
    g.bias = bias; g.relu = relu; g.res = res; g.res_sign = res_sign;
    g.out_f32 = out_f32; g.out_bf16 = (__nv_bfloat16 *)out_bf16;
    g.split_heads = split_L > 0; g.split_L = split_L; g.split_d = split_d;
    return gemm_tc(g, (StatusBlock *)workspace, st) == cudaSuccess ? LSH_OK : LSH_ERR_CUDA;
}
