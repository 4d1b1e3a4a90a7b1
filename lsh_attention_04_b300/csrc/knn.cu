// knn.cu -- LSH bucketing as approximate k-nearest-neighbour search.
//
// "Reformer" glossary (ultralytics.com), section "Atencion LSH", the paragraph after the
// algorithm: locality-sensitive hashing is the classic approximate nearest-neighbour
// method; it finds most of a query's nearest neighbours at a small fraction of the cost of
// an exhaustive search.  Here the search reuses the attention's buckets and sort: the
// candidates of token i are the union over the rounds of the tokens that share its
// bucket in its chunk window (own chunk in both directions and the previous chunk, i left
// out), ranked by cosine similarity x_i.x_j / (|x_i| |x_j|) (0 for a zero vector), ties
// to the smaller j.  The k best are returned, a shorter list padded with (-1, -2).
//
// Two launches after the hash and the sort:
//   1. knn_round_kernel, one CTA per (segment, chunk): the window's rows are gathered
//      through the permutation into shared memory; the chunk x window similarity tile is
//      computed on the tensor cores with warp-level bf16 MMA (fp32 accumulation; fp32
//      inputs use an fp32 FMA loop), then each warp takes rows and keeps the k best
//      same-bucket candidates by k rounds of a warp-wide argmax.  Lists go to a per-round
//      buffer at the token's position.
//   2. knn_merge_kernel, one warp per token: the rounds' lists merged by the same k-round
//      argmax; a token found in several rounds has the same similarity in each (same
//      arithmetic), and every copy of a winner is retired at once, so it is listed once.
#include <limits.h>
#include <math.h>
#include <mma.h>

#include "internal.cuh"

namespace lsh {
namespace {

using namespace nvcuda;

constexpr int kKnnWarps = 8;
constexpr int kRowsInFlight = 4;       // rows a warp selects for at once (independent chains)
constexpr int kWinMax = 128;           // window rows: two chunks of at most 64
constexpr int kSPitch = kWinMax + 4;   // fp32 similarity tile row pitch

template <typename T> struct XRow;
template <> struct XRow<__nv_bfloat16> { static constexpr int pad = 8; };   // 16-byte rows for wmma
template <> struct XRow<float> { static constexpr int pad = 1; };           // odd pitch: no bank conflicts

// k best (largest similarity, then smallest index) of Q independent lists held across a
// warp, lane-major: list q has entries sim[q][m], idx[q][m], live[q][m] on every lane.
// k rounds of a warp-wide argmax; the Q lists' shuffle chains are independent, so they
// overlap.  Lane a < k ends with entry a of each list in out_idx[q], out_sim[q] (-1, -2
// when the list has fewer than k live entries).  Every copy of a winner's index retires.
template <int Q, int NE>
__device__ __forceinline__ void warp_top_k(const float (&sim)[Q][NE], const int (&idx)[Q][NE],
                                           bool (&live)[Q][NE], int k, int lane,
                                           int (&out_idx)[Q], float (&out_sim)[Q]) {
#pragma unroll
    for (int q = 0; q < Q; ++q) { out_idx[q] = -1; out_sim[q] = -2.f; }
    for (int a = 0; a < k; ++a) {
        float bs[Q];
        int bj[Q];
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            bs[q] = -INFINITY;
            bj[q] = INT_MAX;
#pragma unroll
            for (int m = 0; m < NE; ++m)
                if (live[q][m] && (sim[q][m] > bs[q] || (sim[q][m] == bs[q] && idx[q][m] < bj[q]))) {
                    bs[q] = sim[q][m];
                    bj[q] = idx[q][m];
                }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
            for (int q = 0; q < Q; ++q) {
                const float os = __shfl_xor_sync(0xffffffffu, bs[q], off);
                const int oj = __shfl_xor_sync(0xffffffffu, bj[q], off);
                if (os > bs[q] || (os == bs[q] && oj < bj[q])) { bs[q] = os; bj[q] = oj; }
            }
        }
        bool any = false;
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            if (bj[q] == INT_MAX) continue;          // this list has run out
            any = true;
            if (lane == a) { out_idx[q] = bj[q]; out_sim[q] = bs[q]; }
#pragma unroll
            for (int m = 0; m < NE; ++m) live[q][m] = live[q][m] && idx[q][m] != bj[q];
        }
        if (!any) break;                             // warp-uniform: every list ran out
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(kKnnWarps * 32)
knn_round_kernel(const T *__restrict__ qk, const int32_t *__restrict__ buckets,
                 const int32_t *__restrict__ perm, const float *__restrict__ inv_norm, int L,
                 int chunk, int n_rounds, int k, int32_t *__restrict__ cand_idx,
                 float *__restrict__ cand_sim)
{
    constexpr int XP = D + XRow<T>::pad;
    extern __shared__ __align__(128) uint8_t smem[];
    T *X = reinterpret_cast<T *>(smem);                                  // [kWinMax][XP]
    float *S = reinterpret_cast<float *>(smem + sizeof(T) * kWinMax * XP);  // [64][kSPitch]
    int *sb = reinterpret_cast<int *>(S + 64 * kSPitch);                 // window buckets
    int *sj = sb + kWinMax;                                              // window tokens
    float *sn = reinterpret_cast<float *>(sj + kWinMax);                 // window 1/|x|

    const long seg = blockIdx.x;
    const int cq = blockIdx.y;
    const long bh = seg / n_rounds;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int s0 = cq * chunk;                          // first sorted row of the chunk
    const int w0 = max(0, s0 - chunk);                  // first sorted row of the window
    const int n_win = min(L, s0 + chunk) - w0;          // window rows (own + previous)
    const int n_pad = (n_win + 15) & ~15;
    const int r0 = s0 - w0;                             // window row of the chunk's first row
    const int32_t *pseg = perm + seg * L;

    // ---- gather the window: tokens, buckets, norms, rows (zero rows pad to 16)
    for (int w = threadIdx.x; w < n_pad; w += blockDim.x) {
        int j = 0, b = -1;
        float nrm = 0.f;
        if (w < n_win) {
            j = pseg[w0 + w];
            j = (unsigned)j < (unsigned)L ? j : 0;      // a corrupt permutation stays in bounds
            b = buckets[seg * L + j];
            nrm = inv_norm[bh * L + j];
        }
        sj[w] = j;
        sb[w] = b;
        sn[w] = nrm;
    }
    __syncthreads();
    constexpr int kVec = 16 / sizeof(T);                 // elements per 16-byte piece
    constexpr int kPieces = D / kVec;
    for (int e = threadIdx.x; e < n_pad * kPieces; e += blockDim.x) {
        const int w = e / kPieces, pc = e % kPieces;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (w < n_win)
            v = *reinterpret_cast<const uint4 *>(qk + (bh * L + sj[w]) * (long)D + pc * kVec);
        T *dst = X + w * XP + pc * kVec;
        if constexpr (sizeof(T) == 2) {
            *reinterpret_cast<uint4 *>(dst) = v;        // 16-byte aligned: pitch D + 8
        } else {
            const float *f = reinterpret_cast<const float *>(&v);
#pragma unroll
            for (int q = 0; q < 4; ++q) dst[q] = f[q];
        }
    }
    __syncthreads();

    // ---- similarity tile: S[r][w] = x_(s0 + r) . x_(w0 + w), r < chunk, w < n_pad
    if constexpr (sizeof(T) == 2) {
        const int tr = chunk / 16, tc = n_pad / 16;
        for (int t = warp; t < tr * tc; t += kKnnWarps) {
            const int ti = t / tc, tj = t % tc;
            wmma::fragment<wmma::accumulator, 16, 16, 16, float> acc;
            wmma::fill_fragment(acc, 0.f);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                wmma::fragment<wmma::matrix_a, 16, 16, 16, __nv_bfloat16, wmma::row_major> a;
                wmma::fragment<wmma::matrix_b, 16, 16, 16, __nv_bfloat16, wmma::col_major> b;
                wmma::load_matrix_sync(a, X + (r0 + 16 * ti) * XP + 16 * kk, XP);
                wmma::load_matrix_sync(b, X + (16 * tj) * XP + 16 * kk, XP);
                wmma::mma_sync(acc, a, b, acc);
            }
            wmma::store_matrix_sync(S + (16 * ti) * kSPitch + 16 * tj, acc, kSPitch, wmma::mem_row_major);
        }
    } else {
        for (int e = threadIdx.x; e < chunk * n_pad; e += blockDim.x) {
            const int r = e / n_pad, w = e % n_pad;
            const T *a = X + (r0 + r) * XP, *b = X + w * XP;
            float acc = 0.f;
#pragma unroll 8
            for (int c = 0; c < D; ++c) acc = fmaf((float)a[c], (float)b[c], acc);
            S[r * kSPitch + w] = acc;
        }
    }
    __syncthreads();

    // ---- per row: the k best same-bucket candidates of the window (self left out),
    // kRowsInFlight rows of a warp at once
    constexpr int NE = kWinMax / 32;
    for (int rb = warp * kRowsInFlight; rb < chunk; rb += kKnnWarps * kRowsInFlight) {
        float sim[kRowsInFlight][NE];
        int idx[kRowsInFlight][NE];
        bool live[kRowsInFlight][NE];
#pragma unroll
        for (int q = 0; q < kRowsInFlight; ++q) {
            const int r = rb + q;
            const bool row_ok = r < chunk;
            const int ws = r0 + (row_ok ? r : 0);
            const int bs_ = sb[ws];
            const float ns = sn[ws];
#pragma unroll
            for (int m = 0; m < NE; ++m) {
                const int w = lane + 32 * m;
                live[q][m] = row_ok && w < n_win && w != ws && sb[w] == bs_;
                sim[q][m] = live[q][m] ? S[r * kSPitch + w] * ns * sn[w] : -INFINITY;
                idx[q][m] = live[q][m] ? sj[w] : INT_MAX;
            }
        }
        int out_idx[kRowsInFlight];
        float out_sim[kRowsInFlight];
        warp_top_k(sim, idx, live, k, lane, out_idx, out_sim);
        if (lane < k) {
#pragma unroll
            for (int q = 0; q < kRowsInFlight; ++q) {
                const int r = rb + q;
                if (r >= chunk) break;
                const size_t o = ((size_t)seg * L + sj[r0 + r]) * k + lane;
                cand_idx[o] = out_idx[q];
                cand_sim[o] = out_sim[q];
            }
        }
    }
}

// NE entries per lane; a warp merges Q tokens at once
template <int NE, int Q>
__global__ void __launch_bounds__(256)
knn_merge_kernel(const int32_t *__restrict__ cand_idx, const float *__restrict__ cand_sim,
                 long n_tok, int L, int n_rounds, int k, int32_t *__restrict__ nn_idx,
                 float *__restrict__ nn_sim)
{
    const long tok0 = ((long)blockIdx.x * 8 + (threadIdx.x >> 5)) * Q;
    const int lane = threadIdx.x & 31;
    if (tok0 >= n_tok) return;
    const int n_e = n_rounds * k;
    float sim[Q][NE];
    int idx[Q][NE];
    bool live[Q][NE];
#pragma unroll
    for (int q = 0; q < Q; ++q) {
        const long tok = tok0 + q;
        const long bh = tok / L, l = tok % L;
#pragma unroll
        for (int m = 0; m < NE; ++m) {
            const int e = lane + 32 * m;
            live[q][m] = false;
            sim[q][m] = -INFINITY;
            idx[q][m] = INT_MAX;
            if (tok < n_tok && e < n_e) {
                const int r = e / k, a = e % k;
                const size_t o = (((size_t)bh * n_rounds + r) * L + l) * k + a;
                const int j = cand_idx[o];
                if (j >= 0) { live[q][m] = true; idx[q][m] = j; sim[q][m] = cand_sim[o]; }
            }
        }
    }
    int out_idx[Q];
    float out_sim[Q];
    warp_top_k(sim, idx, live, k, lane, out_idx, out_sim);
    if (lane < k) {
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            const long tok = tok0 + q;
            if (tok >= n_tok) break;
            nn_idx[(size_t)tok * k + lane] = out_idx[q];
            nn_sim[(size_t)tok * k + lane] = out_sim[q];
        }
    }
}

template <typename T, int D>
cudaError_t launch_round(const Problem &p, int k, const void *qk, const int32_t *buckets,
                         const int32_t *perm, const float *inv_norm, int32_t *cand_idx,
                         float *cand_sim, cudaStream_t st)
{
    const size_t smem = sizeof(T) * kWinMax * (D + XRow<T>::pad) + sizeof(float) * 64 * kSPitch +
                        (sizeof(int) * 2 + sizeof(float)) * kWinMax;
    cudaError_t e = cudaFuncSetAttribute(knn_round_kernel<T, D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)p.n_seg(), p.L / p.chunk);
    knn_round_kernel<T, D><<<grid, kKnnWarps * 32, smem, st>>>(
        (const T *)qk, buckets, perm, inv_norm, p.L, p.chunk, p.n_rounds, k, cand_idx, cand_sim);
    return cudaGetLastError();
}

}  // namespace

cudaError_t knn_launch(const Problem &p, int k, const void *qk, const int32_t *buckets,
                       const int32_t *perm, const float *inv_norm, int32_t *cand_idx,
                       float *cand_sim, int32_t *nn_idx, float *nn_sim, cudaStream_t st)
{
    cudaError_t e;
    if (p.dtype == LSH_BF16)
        e = p.d == 64 ? launch_round<__nv_bfloat16, 64>(p, k, qk, buckets, perm, inv_norm, cand_idx, cand_sim, st)
                      : launch_round<__nv_bfloat16, 128>(p, k, qk, buckets, perm, inv_norm, cand_idx, cand_sim, st);
    else
        e = p.d == 64 ? launch_round<float, 64>(p, k, qk, buckets, perm, inv_norm, cand_idx, cand_sim, st)
                      : launch_round<float, 128>(p, k, qk, buckets, perm, inv_norm, cand_idx, cand_sim, st);
    if (e != cudaSuccess) return e;
    const long n = p.n_tok();
    const unsigned g4 = (unsigned)((n + 31) / 32), g2 = (unsigned)((n + 15) / 16);
    const int ne = (p.n_rounds * k + 31) / 32;
    if (ne <= 1)
        knn_merge_kernel<1, 4><<<g4, 256, 0, st>>>(cand_idx, cand_sim, n, p.L, p.n_rounds, k, nn_idx, nn_sim);
    else if (ne <= 2)
        knn_merge_kernel<2, 4><<<g4, 256, 0, st>>>(cand_idx, cand_sim, n, p.L, p.n_rounds, k, nn_idx, nn_sim);
    else if (ne <= 4)
        knn_merge_kernel<4, 4><<<g4, 256, 0, st>>>(cand_idx, cand_sim, n, p.L, p.n_rounds, k, nn_idx, nn_sim);
    else
        knn_merge_kernel<8, 2><<<g2, 256, 0, st>>>(cand_idx, cand_sim, n, p.L, p.n_rounds, k, nn_idx, nn_sim);
    return cudaGetLastError();
}

}  // namespace lsh
