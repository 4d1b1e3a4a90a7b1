// attn_simt.cu -- chunked look-one-back LSH attention on CUDA cores (fp32 path).
//
// "Reformer" glossary (ultralytics.com), section "Atencion LSH": the sorted sequence is
// cut into equal chunks and each token attends only to its own chunk and the previous
// one.  modulabs-hub notes, section "LSH attention": keys outside the query's bucket are
// masked with -infinity, the token itself is removed (under shared QK it would always
// score highest), and in the causal case only earlier positions are kept.
//
// One CTA = one chunk of one (b, h, r) segment.  The window (previous + own chunk) is
// gathered through perm into shared memory once; each warp then handles queries of the
// chunk.  Because sorted order groups each bucket into one run and keeps position order
// inside it, the keys a query may see are one interval of sorted indices:
//   [max(window_lo, bucket_lo), causal ? s : min(window_hi, bucket_hi))  minus s itself.
// Scores use scale * (q . k) * |k|^-1; softmax and the value sum run in fp32.
#include <math.h>

#include <type_traits>

#include "internal.cuh"

namespace lsh {
namespace {

constexpr int kWarps = 16;

// T: input element type; TO: per-round row type (fp32 for fp32 inputs, bf16 for both
// 16-bit input types)
// Shared-memory element of the staged window rows: fp32, except 16-bit inputs at chunk
// 128 and d = 128, whose rows stay 16-bit so the 256-row window fits.
template <typename T, int D, int C>
using Stage = typename std::conditional<(C == 128 && D == 128 && sizeof(T) == 2), T, float>::type;
__device__ __forceinline__ float tof(float x) { return x; }
__device__ __forceinline__ float tof(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float tof(__half x) { return __half2float(x); }
template <typename E> __device__ __forceinline__ E fromf(float x);
template <> __device__ __forceinline__ float fromf<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 fromf<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }
template <> __device__ __forceinline__ __half fromf<__half>(float x) { return __float2half_rn(x); }

template <typename T, typename TO, int D, int C>
__global__ void __launch_bounds__(kWarps * 32)
attn_simt_kernel(const T *__restrict__ qk, const T *__restrict__ v,
                 const int32_t *__restrict__ buckets, const int32_t *__restrict__ perm,
                 const int32_t *__restrict__ bstart, const float *__restrict__ inv_norm, int L,
                 int n_rounds, int nb, int causal, float scale, int token_order,
                 TO *__restrict__ o_r, float *__restrict__ lse_r)
{
    using E = Stage<T, D, C>;
    constexpr int KS = D + (sizeof(E) == 4 ? 1 : 2);  // padded key row: lanes reading
                                                      // different rows hit different banks
    extern __shared__ float smem[];
    float *kin = smem;                     // [2C]  |k|^-1
    int *kb = (int *)(kin + 2 * C);        // [2C]  bucket
    E *Ks = reinterpret_cast<E *>(kb + 2 * C);   // [2C][KS]
    E *Vs = Ks + 2 * C * KS;               // [2C][D]

    const int chunk_id = blockIdx.x;
    const long seg = blockIdx.y;
    const long bh = seg / n_rounds;
    const int lo = max(0, (chunk_id - 1) * C);
    const int hi = (chunk_id + 1) * C;
    const int nwin = hi - lo;
    const int32_t *P = perm + seg * L;
    const T *qkh = qk + (size_t)bh * L * D;
    const T *vh = v + (size_t)bh * L * D;

    for (int idx = threadIdx.x; idx < nwin * D; idx += blockDim.x) {
        const int t = idx / D, e = idx % D;
        const int j = P[lo + t];
        Ks[t * KS + e] = fromf<E>(ld_f32(qkh, (size_t)j * D + e));
        Vs[t * D + e] = fromf<E>(ld_f32(vh, (size_t)j * D + e));
    }
    for (int t = threadIdx.x; t < nwin; t += blockDim.x) {
        const int j = P[lo + t];
        kin[t] = inv_norm[(size_t)bh * L + j];
        kb[t] = buckets[(size_t)seg * L + j];
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int KPL = 2 * C / 32;  // window keys per lane
    constexpr int EPL = D / 32;      // output elements per lane
    const int32_t *bs = bstart + seg * (nb + 1);
    for (int q = warp; q < C; q += kWarps) {
        const int s = chunk_id * C + q;
        const int ts = s - lo;
        const int bq = kb[ts];
        const int klo = max(lo, bs[bq]);
        const int khi = causal ? s : min(hi, bs[bq + 1]);
        float sc[KPL];
        float mx = -INFINITY;
#pragma unroll
        for (int m = 0; m < KPL; ++m) {
            const int t = lane + 32 * m;
            const int sidx = lo + t;
            float val = -INFINITY;
            if (t < nwin && sidx >= klo && sidx < khi && sidx != s) {
                float dot = 0.f;
#pragma unroll 8
                for (int e = 0; e < D; ++e) dot = fmaf(tof(Ks[ts * KS + e]), tof(Ks[t * KS + e]), dot);
                val = scale * dot * kin[t];
            }
            sc[m] = val;
            mx = fmaxf(mx, val);
        }
        mx = warp_max(mx);
        float o[EPL];
        float lse;
        if (mx == -INFINITY) {
#pragma unroll
            for (int i = 0; i < EPL; ++i) o[i] = tof(Vs[ts * D + lane + 32 * i]);
            lse = kSelfLogit;
        } else {
            float sum = 0.f;
#pragma unroll
            for (int m = 0; m < KPL; ++m) {
                sc[m] = (sc[m] == -INFINITY) ? 0.f : expf(sc[m] - mx);
                sum += sc[m];
            }
            sum = warp_sum(sum);
#pragma unroll
            for (int i = 0; i < EPL; ++i) o[i] = 0.f;
#pragma unroll
            for (int m = 0; m < KPL; ++m) {
                for (int src = 0; src < 32; ++src) {
                    const float pw = __shfl_sync(0xffffffffu, sc[m], src);
                    const int t = 32 * m + src;
                    if (pw != 0.f) {
#pragma unroll
                        for (int i = 0; i < EPL; ++i) o[i] = fmaf(pw, tof(Vs[t * D + lane + 32 * i]), o[i]);
                    }
                }
            }
            const float rs = 1.0f / sum;
#pragma unroll
            for (int i = 0; i < EPL; ++i) o[i] *= rs;
            lse = mx + logf(sum);
        }
        const size_t row = (size_t)seg * L + (token_order ? P[s] : s);
#pragma unroll
        for (int i = 0; i < EPL; ++i) st_elem(o_r, row * D + lane + 32 * i, o[i]);
        if (lane == 0) lse_r[row] = lse;
    }
}

template <typename T, typename TO, int D, int C>
cudaError_t launch(const Problem &p, const void *qk, const void *v, const int32_t *buckets,
                   const int32_t *perm, const int32_t *bstart, const float *inv_norm, void *o_r,
                   float *lse_r, cudaStream_t st)
{
    using E = Stage<T, D, C>;
    constexpr int KS = D + (sizeof(E) == 4 ? 1 : 2);
    const size_t smem = sizeof(E) * (2 * C * KS + 2 * C * D) + (sizeof(float) + sizeof(int)) * 2 * C;
    auto k = attn_simt_kernel<T, TO, D, C>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(p.L / C), (unsigned)p.n_seg());
    k<<<grid, kWarps * 32, smem, st>>>((const T *)qk, (const T *)v, buckets, perm, bstart,
                                       inv_norm, p.L, p.n_rounds, p.nb, p.causal, p.scale,
                                       p.token_order, (TO *)o_r, lse_r);
    return cudaGetLastError();
}

template <typename T, typename TO>
cudaError_t dispatch(const Problem &p, const void *qk, const void *v, const int32_t *buckets,
                     const int32_t *perm, const int32_t *bstart, const float *inv_norm, void *o_r,
                     float *lse_r, cudaStream_t st)
{
    if (p.d == 64)
        return p.chunk == 32 ? launch<T, TO, 64, 32>(p, qk, v, buckets, perm, bstart, inv_norm, o_r, lse_r, st)
             : p.chunk == 64 ? launch<T, TO, 64, 64>(p, qk, v, buckets, perm, bstart, inv_norm, o_r, lse_r, st)
                             : launch<T, TO, 64, 128>(p, qk, v, buckets, perm, bstart, inv_norm, o_r, lse_r, st);
    if (p.chunk == 128) {
        if constexpr (sizeof(T) == 2)
            return launch<T, TO, 128, 128>(p, qk, v, buckets, perm, bstart, inv_norm, o_r, lse_r, st);
        return cudaErrorInvalidValue;      // fp32 at d = 128: the window does not fit
    }
    return p.chunk == 32 ? launch<T, TO, 128, 32>(p, qk, v, buckets, perm, bstart, inv_norm, o_r, lse_r, st)
                         : launch<T, TO, 128, 64>(p, qk, v, buckets, perm, bstart, inv_norm, o_r, lse_r, st);
}

}  // namespace

cudaError_t attn_simt(const Problem &p, const void *qk, const void *v, const int32_t *buckets,
                      const int32_t *perm, const int32_t *bstart, const float *inv_norm,
                      void *o_r, float *lse_r, cudaStream_t st)
{
    if (p.dtype == LSH_F32)
        return dispatch<float, float>(p, qk, v, buckets, perm, bstart, inv_norm, o_r, lse_r, st);
    if (p.dtype == LSH_F16)
        return dispatch<__half, __nv_bfloat16>(p, qk, v, buckets, perm, bstart, inv_norm, o_r, lse_r, st);
    return dispatch<__nv_bfloat16, __nv_bfloat16>(p, qk, v, buckets, perm, bstart, inv_norm, o_r, lse_r, st);
}

}  // namespace lsh
