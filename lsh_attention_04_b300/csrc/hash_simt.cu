// hash_simt.cu -- angular LSH on CUDA cores (fp32 inputs, and bf16 shapes the tensor-core
// kernel does not take).
//
// "Reformer" glossary (ultralytics.com), section "Atencion LSH": multiply by a random
// matrix R and take the position of the largest entry of [xR, -xR] as the bucket.
// modulabs-hub Reformer notes, "Locality sensitive hashing": R has n_buckets/2 columns.
//
// One CTA = 128 tokens x one round; one thread per token.  The token tile is staged
// transposed in shared memory (conflict-free column reads), R_r is streamed through
// shared memory 32 columns at a time and read as broadcasts.  Each thread keeps the
// first index of the largest projection and of the smallest one; the bucket is the
// first argmax of the concatenation [p, -p]: the positive half wins ties.
#include <math.h>

#include "internal.cuh"

namespace lsh {
namespace {

constexpr int kTok = 128;   // tokens per CTA
constexpr int kCols = 32;   // columns of R_r per pass

template <typename T, int D>
__global__ void __launch_bounds__(kTok)
hash_simt_kernel(const T *__restrict__ qk, const T *__restrict__ R, long n_tok, int half,
                 int n_rounds, int L, int32_t *__restrict__ buckets, float *__restrict__ inv_norm)
{
    extern __shared__ float smem[];
    float *xs = smem;             // [D][kTok]
    float *rs = smem + D * kTok;  // [D][kCols]
    const int tid = threadIdx.x;
    const long tok0 = (long)blockIdx.x * kTok;
    const int r = blockIdx.y;

    for (int idx = tid; idx < kTok * D; idx += kTok) {
        const int row = idx / D, k = idx % D;
        const long t = tok0 + row;
        xs[k * kTok + row] = (t < n_tok) ? ld_f32(qk, (size_t)t * D + k) : 0.f;
    }
    __syncthreads();

    const long t = tok0 + tid;
    if (r == 0 && t < n_tok) {
        float s = 0.f;
        for (int k = 0; k < D; ++k) s = fmaf(xs[k * kTok + tid], xs[k * kTok + tid], s);
        inv_norm[t] = s > 0.f ? 1.0f / sqrtf(s) : 0.f;
    }

    float pmax = -INFINITY, nmin = INFINITY;
    int pidx = 0, nidx = 0;
    const T *Rr = R + (size_t)r * D * half;
    for (int j0 = 0; j0 < half; j0 += kCols) {
        __syncthreads();
        for (int idx = tid; idx < D * kCols; idx += kTok) {
            const int k = idx / kCols, jj = idx % kCols;
            rs[idx] = (j0 + jj < half) ? ld_f32(Rr, (size_t)k * half + j0 + jj) : 0.f;
        }
        __syncthreads();
        float acc[kCols];
#pragma unroll
        for (int jj = 0; jj < kCols; ++jj) acc[jj] = 0.f;
        for (int k = 0; k < D; ++k) {
            const float xv = xs[k * kTok + tid];
#pragma unroll
            for (int jj = 0; jj < kCols; ++jj) acc[jj] = fmaf(xv, rs[k * kCols + jj], acc[jj]);
        }
#pragma unroll
        for (int jj = 0; jj < kCols; ++jj) {
            const int j = j0 + jj;
            if (j < half) {
                if (acc[jj] > pmax) { pmax = acc[jj]; pidx = j; }
                if (acc[jj] < nmin) { nmin = acc[jj]; nidx = j; }
            }
        }
    }
    if (t < n_tok) {
        const int bucket = (pmax >= -nmin) ? pidx : half + nidx;
        const long bh = t / L, l = t % L;
        buckets[((size_t)bh * n_rounds + r) * L + l] = bucket;
    }
}

template <typename T, int D>
cudaError_t launch(const Problem &p, const void *qk, const void *R, int32_t *buckets,
                   float *inv_norm, cudaStream_t st)
{
    const size_t smem = sizeof(float) * (D * kTok + D * kCols);
    auto k = hash_simt_kernel<T, D>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const long n = p.n_tok();
    dim3 grid((unsigned)((n + kTok - 1) / kTok), (unsigned)p.n_rounds);
    k<<<grid, kTok, smem, st>>>((const T *)qk, (const T *)R, n, p.nb / 2, p.n_rounds, p.L,
                                buckets, inv_norm);
    return cudaGetLastError();
}

}  // namespace

cudaError_t hash_simt(const Problem &p, const void *qk, const void *R, int32_t *buckets,
                      float *inv_norm, cudaStream_t st)
{
    if (p.dtype == LSH_F32)
        return p.d == 64 ? launch<float, 64>(p, qk, R, buckets, inv_norm, st)
                         : launch<float, 128>(p, qk, R, buckets, inv_norm, st);
    if (p.dtype == LSH_F16)
        return p.d == 64 ? launch<__half, 64>(p, qk, R, buckets, inv_norm, st)
                         : launch<__half, 128>(p, qk, R, buckets, inv_norm, st);
    return p.d == 64 ? launch<__nv_bfloat16, 64>(p, qk, R, buckets, inv_norm, st)
                     : launch<__nv_bfloat16, 128>(p, qk, R, buckets, inv_norm, st);
}

}  // namespace lsh
