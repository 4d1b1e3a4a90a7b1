// combine_tma.cu -- round combination over token-ordered per-round rows, fed by TMA bulk
// copies.
//
// Inside the fused forward the attention step writes round r's row of token i at position
// i of plane r (o_r [B][H][R][L][d] bf16, lse_r [B][H][R][L]).  Then for a tile of 16
// consecutive tokens of one head, each round's rows are one contiguous 16*d*2-byte block
// and its log-normalisers one 64-byte block.  One producer lane moves these blocks into
// a 3-stage shared-memory ring with cp.async.bulk (large contiguous transfers, which the
// copy engine streams at full rate; a warp gathering the same rows token by token touches
// R DRAM pages per token instead).  Eight consumer warps then combine two tokens each:
//   lse_i = logsumexp_r lse_r(i),   out_i = sum_r exp(lse_r(i) - lse_i) * o_r(i)
// (rounds weighted by their share of the softmax mass, as in combine.cu), and stream the
// fp32 outputs.  Persistent CTAs, two per SM (two independent copy pipelines keep more
// DRAM reads in flight than one CTA with a deeper ring); every wait is bounded
// (sm100::wait).
#include <math.h>

#include "sm100.cuh"

namespace lsh {
namespace {

using namespace sm100;

constexpr int kT = 16;            // tokens per tile
constexpr int kStages = 3;
constexpr int kMaxR = 8;          // rounds this kernel takes
constexpr int kCWarps = 8;        // consumer warps, kT / kCWarps tokens each
constexpr int kThreads = (kCWarps + 1) * 32;
constexpr int kCtasPerSm = 2;

struct __align__(8) CombineBars {
    uint64_t full[kStages], empty[kStages];
    int abort_flag;
};

__host__ __device__ constexpr size_t stage_bytes(int d) {
    return (size_t)kMaxR * kT * d * 2 + (size_t)kMaxR * kT * 4;
}

template <int D>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
combine_tma_kernel(const __nv_bfloat16 *__restrict__ o_r, const float *__restrict__ lse_r,
                   long n_tiles, int L, int R, float *__restrict__ out, float *__restrict__ lse,
                   StatusBlock *status)
{
    constexpr int EPL = D / 32;                       // elements per lane
    constexpr uint32_t kOBytes = (uint32_t)kT * D * 2;
    extern __shared__ uint8_t smem_raw[];
    __shared__ CombineBars sb;
    uint8_t *smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int *abort_flag = &sb.abort_flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sb.full[s], 1);
            mbar_init(&sb.empty[s], kCWarps);
        }
        sb.abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();

    if (warp == kCWarps) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            int it = 0;
            for (long u = blockIdx.x; u < n_tiles; u += gridDim.x, ++it) {
                const int s = it % kStages;
                if (!wait(&sb.empty[s], ((it / kStages) & 1) ^ 1, abort_flag, status, 0x901)) break;
                const long tok0 = u * kT;
                const long bh = tok0 / L;
                const int i0 = (int)(tok0 - bh * L);
                uint8_t *so = smem + s * stage_bytes(D);
                uint8_t *sl = so + (size_t)kMaxR * kOBytes;
                mbar_expect_tx(&sb.full[s], (uint32_t)R * (kOBytes + kT * 4));
                for (int r = 0; r < R; ++r) {
                    const size_t row0 = ((size_t)bh * R + r) * L + i0;
                    bulk_g2s(so + r * kOBytes, o_r + row0 * D, kOBytes, &sb.full[s]);
                    bulk_g2s(sl + r * kT * 4, lse_r + row0, kT * 4, &sb.full[s]);
                }
            }
            // wind-down: the last fills land before the CTA exits
            const int n_it = it;
            for (int k = 1; k <= kStages && n_it - k >= 0; ++k) {
                const int i2 = n_it - k;
                int dummy = 0;
                wait(&sb.full[i2 % kStages], (i2 / kStages) & 1, &dummy, nullptr, 0x902);
            }
        }
        return;
    }

    // -------------------------------------------------------------------- consumers
    constexpr int kPerWarp = kT / kCWarps;
    int it = 0;
    for (long u = blockIdx.x; u < n_tiles; u += gridDim.x, ++it) {
        const int s = it % kStages;
        const bool ok = wait(&sb.full[s], (it / kStages) & 1, abort_flag, status, 0x903);
        if (!__all_sync(0xffffffffu, ok)) break;
        const uint8_t *so = smem + s * stage_bytes(D);
        const float *sl = reinterpret_cast<const float *>(so + (size_t)kMaxR * kOBytes);
#pragma unroll
        for (int k = 0; k < kPerWarp; ++k) {
            const int tl = warp * kPerWarp + k;
            const float lr = lane < R ? sl[lane * kT + tl] : -INFINITY;
            const float mx = warp_max(lr);
            const float w = lane < R ? expf(lr - mx) : 0.f;
            const float sum = warp_sum(w);
            float acc[EPL];
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
#pragma unroll
            for (int r = 0; r < kMaxR; ++r) {
                const float wr = __shfl_sync(0xffffffffu, w, r);
                if (r < R) {
                    const __nv_bfloat16 *row =
                        reinterpret_cast<const __nv_bfloat16 *>(so + r * kOBytes) + (size_t)tl * D + lane * EPL;
                    if constexpr (EPL == 4) {
                        const uint2 t = *reinterpret_cast<const uint2 *>(row);
                        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&t.x));
                        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&t.y));
                        acc[0] = fmaf(wr, a.x, acc[0]);
                        acc[1] = fmaf(wr, a.y, acc[1]);
                        acc[2] = fmaf(wr, b.x, acc[2]);
                        acc[3] = fmaf(wr, b.y, acc[3]);
                    } else {
                        const uint32_t t = *reinterpret_cast<const uint32_t *>(row);
                        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&t));
                        acc[0] = fmaf(wr, a.x, acc[0]);
                        acc[1] = fmaf(wr, a.y, acc[1]);
                    }
                }
            }
            const long tok = u * kT + tl;
            const float rs = 1.0f / sum;
            float *dst = out + (size_t)tok * D + lane * EPL;
            if constexpr (EPL == 4) {
                __stcs(reinterpret_cast<float4 *>(dst), make_float4(acc[0] * rs, acc[1] * rs, acc[2] * rs, acc[3] * rs));
            } else {
                __stcs(reinterpret_cast<float2 *>(dst), make_float2(acc[0] * rs, acc[1] * rs));
            }
            if (lane == 0) lse[tok] = mx + logf(sum);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sb.empty[s]);
    }
}

template <int D>
cudaError_t launch(const Problem &p, const void *o_r, const float *lse_r, float *out, float *lse,
                   StatusBlock *status, cudaStream_t st)
{
    const long n_tiles = p.n_tok() / kT;
    const size_t smem = 128 + kStages * stage_bytes(D);
    cudaError_t e = cudaFuncSetAttribute(combine_tma_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long grid = n_tiles < (long)kCtasPerSm * sms ? n_tiles : (long)kCtasPerSm * sms;
    combine_tma_kernel<D><<<(unsigned)grid, kThreads, smem, st>>>(
        (const __nv_bfloat16 *)o_r, lse_r, n_tiles, p.L, p.n_rounds, out, lse, status);
    return cudaGetLastError();
}

}  // namespace

bool combine_tma_supported(const Problem &p)
{
    return p.token_order && is16(p.dtype) && p.n_rounds <= kMaxR && p.L % kT == 0 &&
           (p.d == 64 || p.d == 128);
}

cudaError_t combine_tma(const Problem &p, const void *o_r, const float *lse_r, float *out, float *lse,
                        StatusBlock *status, cudaStream_t st)
{
    return p.d == 64 ? launch<64>(p, o_r, lse_r, out, lse, status, st)
                     : launch<128>(p, o_r, lse_r, out, lse, status, st);
}

}  // namespace lsh
