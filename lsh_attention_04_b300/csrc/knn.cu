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
//      same-bucket candidates: 64-bit keys (similarity, then smaller index) sorted in
//      32-entry blocks by a bitonic network across the lanes and the blocks' top 32
//      merged.  Lists go to a per-round buffer at the token's position.
//   2. knn_merge_kernel, two tokens per warp: the rounds' sorted lists folded in one at a
//      time by the bitonic top-32 merge; a token found in several rounds has the same key
//      in each (the same similarity by the same arithmetic), so before each fold the list
//      drops the keys the running result already holds.
#include <limits.h>
#include <math.h>
#include <mma.h>

#include "internal.cuh"

namespace lsh {
namespace {

using namespace nvcuda;

constexpr int kKnnWarps = 16;
constexpr int kRowsInFlight = 2;       // rows a warp selects for at once (independent chains)
constexpr int kWinMax = 128;           // window rows: two chunks of at most 64
constexpr int kSPitch = kWinMax + 4;   // fp32 similarity tile row pitch

template <typename T> struct XRow;
template <> struct XRow<__nv_bfloat16> { static constexpr int pad = 8; };   // 16-byte rows for wmma
template <> struct XRow<float> { static constexpr int pad = 1; };           // odd pitch: no bank conflicts

// Candidate keys: (similarity, then smaller token index) as one 64-bit integer, so a
// larger key is a better candidate: the float's bits in an order-preserving form in the
// high word, the complement of the index in the low word; 0 for a dead entry (every live
// key is larger, the smallest finite float mapping to 0x00800000 in the high word).
__device__ __forceinline__ unsigned long long cand_key(float sim, int idx, bool live)
{
    unsigned u = sim == 0.f ? 0u : __float_as_uint(sim);       // -0 ranks as +0
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return live ? ((unsigned long long)u << 32) | (unsigned)(~idx) : 0ull;
}

__device__ __forceinline__ float key_sim(unsigned long long key)
{
    unsigned u = (unsigned)(key >> 32);
    u = (u & 0x80000000u) ? (u & 0x7fffffffu) : ~u;
    return __uint_as_float(u);
}

__device__ __forceinline__ unsigned long long kmax(unsigned long long a, unsigned long long b) { return a > b ? a : b; }
__device__ __forceinline__ unsigned long long kmin(unsigned long long a, unsigned long long b) { return a < b ? a : b; }

// One key per lane sorted descending across the warp (lane 0 the largest): a bitonic
// network of 15 compare-exchange stages over lane pairs.
__device__ __forceinline__ unsigned long long warp_sort_desc(unsigned long long x, int lane)
{
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const unsigned long long y = __shfl_xor_sync(0xffffffffu, x, stride);
            const bool keep_max = ((lane & stride) == 0) == ((lane & size) == 0);
            x = keep_max ? kmax(x, y) : kmin(x, y);
        }
    }
    return x;
}

// The 32 largest of two descending lane-sorted sequences, sorted descending: the
// elementwise maximum of one and the other reversed is bitonic and holds them; five
// merge stages sort it.
__device__ __forceinline__ unsigned long long warp_top32_of_two(unsigned long long a,
                                                                unsigned long long b, int lane)
{
    unsigned long long x = kmax(a, __shfl_sync(0xffffffffu, b, 31 - lane));
#pragma unroll
    for (int stride = 16; stride > 0; stride >>= 1) {
        const unsigned long long y = __shfl_xor_sync(0xffffffffu, x, stride);
        x = (lane & stride) == 0 ? kmax(x, y) : kmin(x, y);
    }
    return x;
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
    // kRowsInFlight rows of a warp at once.  The row's candidates are its bucket's run in
    // the window, cut into 32-entry blocks across the lanes: each block is sorted by key
    // and the blocks' top 32 are merged; lane a ends with the row's a-th best.
    constexpr int NE = kWinMax / 32;
    static_assert(NE == 4, "four 32-entry blocks per window");
    for (int rb = warp * kRowsInFlight; rb < chunk; rb += kKnnWarps * kRowsInFlight) {
        unsigned long long key[kRowsInFlight][NE], top[kRowsInFlight];
        int nblk = 0;                                      // warp-uniform, over the rows
#pragma unroll
        for (int q = 0; q < kRowsInFlight; ++q) {
            const int r = rb + q;
            const bool row_ok = r < chunk;
            const int ws = r0 + (row_ok ? r : 0);
            const int bs_ = sb[ws];
            const float ns = sn[ws];
            // the window is in sorted order, so the row's bucket is one run [a, b) of it:
            // only the blocks that run covers are sorted
            int a = kWinMax, b = 0;
#pragma unroll
            for (int m = 0; m < NE; ++m) {
                const unsigned bal = __ballot_sync(0xffffffffu, lane + 32 * m < n_win && sb[lane + 32 * m] == bs_);
                if (bal) {
                    a = min(a, 32 * m + __ffs(bal) - 1);
                    b = max(b, 32 * m + 32 - __clz(bal));
                }
            }
            if (row_ok && b > a) nblk = max(nblk, (b - a + 31) / 32);
#pragma unroll
            for (int m = 0; m < NE; ++m) {
                const int w = a + lane + 32 * m;
                const bool live = row_ok && w < b && w != ws;
                key[q][m] = cand_key(live ? S[r * kSPitch + w] * ns * sn[w] : 0.f,
                                     live ? sj[w] : 0, live);
            }
            top[q] = 0ull;
        }
        // the rows' sorting networks interleave (independent shuffle chains)
        if (nblk >= 1) {
#pragma unroll
            for (int q = 0; q < kRowsInFlight; ++q) top[q] = warp_sort_desc(key[q][0], lane);
        }
        if (nblk >= 2) {
#pragma unroll
            for (int q = 0; q < kRowsInFlight; ++q)
                top[q] = warp_top32_of_two(top[q], warp_sort_desc(key[q][1], lane), lane);
        }
        if (nblk == 3) {
#pragma unroll
            for (int q = 0; q < kRowsInFlight; ++q)
                top[q] = warp_top32_of_two(top[q], warp_sort_desc(key[q][2], lane), lane);
        }
        if (nblk == 4) {
#pragma unroll
            for (int q = 0; q < kRowsInFlight; ++q)
                top[q] = warp_top32_of_two(top[q], warp_top32_of_two(warp_sort_desc(key[q][2], lane),
                                                                     warp_sort_desc(key[q][3], lane), lane), lane);
        }
        if (lane < k) {
#pragma unroll
            for (int q = 0; q < kRowsInFlight; ++q) {
                const int r = rb + q;
                if (r >= chunk) break;
                const size_t o = ((size_t)seg * L + sj[r0 + r]) * k + lane;
                cand_idx[o] = top[q] ? (int)~(unsigned)top[q] : -1;
                cand_sim[o] = top[q] ? key_sim(top[q]) : -2.f;
            }
        }
    }
}

// Closes the gaps of a descending lane-sorted sequence whose dropped entries are 0:
// lane l takes the l-th kept entry, the freed lanes at the end become 0.
__device__ __forceinline__ unsigned long long warp_compact_desc(unsigned long long x, int lane)
{
    const unsigned mask = __ballot_sync(0xffffffffu, x != 0ull);
    const int n = __popc(mask);
    const int src = lane < n ? (int)__fns(mask, 0, lane + 1) : 0;
    const unsigned long long y = __shfl_sync(0xffffffffu, x, src);
    return lane < n ? y : 0ull;
}

// x (descending lane-sorted, distinct keys) without the keys that also occur in acc
// (descending lane-sorted, distinct): each lane finds its key in acc by a five-step binary
// search over the lanes, then the sequence is compacted.
__device__ __forceinline__ unsigned long long warp_remove_present(unsigned long long x,
                                                                  unsigned long long acc, int lane)
{
    int lo = 0;                                   // entries of acc greater than x
#pragma unroll
    for (int step = 16; step > 0; step >>= 1) {
        const unsigned long long v = __shfl_sync(0xffffffffu, acc, lo + step - 1);
        if (v > x) lo += step;
    }
    const unsigned long long at = __shfl_sync(0xffffffffu, acc, lo & 31);
    const bool present = x != 0ull && lo < 32 && at == x;
    return warp_compact_desc(present ? 0ull : x, lane);
}

// One warp merges the rounds' lists of Q tokens: each list is sorted (the round kernel
// writes entry a at lane a), so the lists are folded in one at a time by the bitonic
// top-32 merge; before each fold the list loses the tokens the running result already
// holds (the same key: the same similarity by the same arithmetic, and the same index),
// so the merged 32 are distinct.
template <int Q>
__global__ void __launch_bounds__(256)
knn_merge_kernel(const int32_t *__restrict__ cand_idx, const float *__restrict__ cand_sim,
                 long n_tok, int L, int n_rounds, int k, int32_t *__restrict__ nn_idx,
                 float *__restrict__ nn_sim)
{
    const long tok0 = ((long)blockIdx.x * 8 + (threadIdx.x >> 5)) * Q;
    const int lane = threadIdx.x & 31;
    if (tok0 >= n_tok) return;                          // warp-uniform
    auto list = [&](int q, int r) -> unsigned long long {
        const long tok = tok0 + q;
        if (tok >= n_tok || lane >= k) return 0ull;
        const long bh = tok / L, l = tok % L;
        const size_t o = (((size_t)bh * n_rounds + r) * L + l) * k + lane;
        const int j = cand_idx[o];
        return j >= 0 ? cand_key(cand_sim[o], j, true) : 0ull;
    };
    unsigned long long acc[Q];
#pragma unroll
    for (int q = 0; q < Q; ++q) acc[q] = list(q, 0);
    for (int r = 1; r < n_rounds; ++r) {
        unsigned long long nx[Q];
#pragma unroll
        for (int q = 0; q < Q; ++q) nx[q] = list(q, r);
#pragma unroll
        for (int q = 0; q < Q; ++q)
            acc[q] = warp_top32_of_two(acc[q], warp_remove_present(nx[q], acc[q], lane), lane);
    }
    if (lane < k) {
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            const long tok = tok0 + q;
            if (tok >= n_tok) break;
            nn_idx[(size_t)tok * k + lane] = acc[q] ? (int)~(unsigned)acc[q] : -1;
            nn_sim[(size_t)tok * k + lane] = acc[q] ? key_sim(acc[q]) : -2.f;
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
    const unsigned g2 = (unsigned)((n + 15) / 16);          // 8 warps x 2 tokens per CTA
    knn_merge_kernel<2><<<g2, 256, 0, st>>>(cand_idx, cand_sim, n, p.L, p.n_rounds, k, nn_idx, nn_sim);
    return cudaGetLastError();
}

}  // namespace lsh
