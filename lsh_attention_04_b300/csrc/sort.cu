// sort.cu -- segmented stable counting sort of bucket ids, one segment per
// (batch, head, round).
//
// ai-scholar.tech Reformer article, "LSH attention": after hashing, sort by LSH bucket;
// modulabs-hub notes, "LSH attention": the bucketed keys are put in order so that a
// chunked batch computation becomes possible.  Ties keep position order, so the result
// is the unique permutation that orders tokens by (bucket, position).
//
// Three launches, no inter-CTA waiting:
//   1. count   per 4096-key tile: a shared-memory histogram, written bucket-major as
//              counts[seg][bucket][tile];
//   2. scan    per segment: exclusive scan of counts in (bucket, tile) order gives every
//              tile's first output slot for each bucket, and bstart;
//   3. scatter per tile: 16 warps each own 256 consecutive keys; warp-level ranking
//              (__match_any_sync + popc) against per-warp shared histograms gives each
//              key its stable slot; writes perm[slot] = pos and inv[pos] = slot.
#include "internal.cuh"

namespace lsh {
namespace {

constexpr int kScatterWarps = 16;
constexpr int kKeysPerWarp = kSortTile / kScatterWarps;  // 256

__global__ void __launch_bounds__(512)
sort_count_kernel(const int32_t *__restrict__ buckets, int L, int nb, int tiles,
                  int32_t *__restrict__ counts)
{
    extern __shared__ int hist[];
    const int tile = blockIdx.x;
    const long seg = blockIdx.y;
    for (int b = threadIdx.x; b < nb; b += blockDim.x) hist[b] = 0;
    __syncthreads();
    const int32_t *keys = buckets + seg * L;
    const int lo = tile * kSortTile;
    const int hi = min(L, lo + kSortTile);
    for (int i = lo + threadIdx.x; i < hi; i += blockDim.x) {
        const int k = keys[i];
        if ((unsigned)k < (unsigned)nb) atomicAdd(&hist[k], 1);   // ids outside [0, nb) skipped
    }
    __syncthreads();
    int32_t *c = counts + (size_t)seg * nb * tiles;
    for (int b = threadIdx.x; b < nb; b += blockDim.x) c[(size_t)b * tiles + tile] = hist[b];
}

// Exclusive scan of counts[seg][0 .. nb*tiles) in place; bstart[seg][b] = start of bucket b.
__global__ void __launch_bounds__(1024)
sort_scan_kernel(int32_t *__restrict__ counts, int nb, int tiles, int L,
                 int32_t *__restrict__ bstart)
{
    __shared__ int warp_tot[32];
    const long seg = blockIdx.x;
    const int n = nb * tiles;
    int32_t *c = counts + (size_t)seg * n;
    const int per = (n + blockDim.x - 1) / blockDim.x;
    const int beg = min(n, (int)threadIdx.x * per);
    const int end = min(n, beg + per);
    int local = 0;
    for (int i = beg; i < end; ++i) local += c[i];
    // block-wide exclusive scan of `local`
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        const int nw = blockDim.x >> 5;
        int w = lane < nw ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < nw) warp_tot[lane] = w;
    }
    __syncthreads();
    int run = x - local + (warp > 0 ? warp_tot[warp - 1] : 0);
    int32_t *bs = bstart + seg * (nb + 1);
    for (int i = beg; i < end; ++i) {
        const int v = c[i];
        c[i] = run;
        if (i % tiles == 0) bs[i / tiles] = run;
        run += v;
    }
    if (threadIdx.x == 0) bs[nb] = L;
}

__global__ void __launch_bounds__(kScatterWarps * 32)
sort_scatter_kernel(const int32_t *__restrict__ buckets, const int32_t *__restrict__ offsets,
                    int L, int nb, int tiles, int32_t *__restrict__ perm,
                    int32_t *__restrict__ inv)
{
    extern __shared__ int whist[];  // [kScatterWarps][nb]
    const int tile = blockIdx.x;
    const long seg = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < kScatterWarps * nb; i += blockDim.x) whist[i] = 0;
    __syncthreads();

    const int32_t *keys = buckets + seg * L;
    const int wlo = tile * kSortTile + warp * kKeysPerWarp;
    int *hist = whist + warp * nb;
    const unsigned lt = (1u << lane) - 1u;

    // pass 1: per-warp counts
    for (int it = 0; it < kKeysPerWarp / 32; ++it) {
        const int pos = wlo + it * 32 + lane;
        int key = pos < L ? keys[pos] : -1;
        if (key >= nb) key = -1;
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        if (key >= 0 && (peers & lt) == 0) hist[key] += __popc(peers);
    }
    __syncthreads();

    // pass 2: turn per-warp counts into first slots (tile offset + earlier warps)
    const int32_t *off = offsets + (size_t)seg * nb * tiles;
    for (int b = threadIdx.x; b < nb; b += blockDim.x) {
        int run = off[(size_t)b * tiles + tile];
        for (int w = 0; w < kScatterWarps; ++w) {
            const int c = whist[w * nb + b];
            whist[w * nb + b] = run;
            run += c;
        }
    }
    __syncthreads();

    // pass 3: stable ranks in position order
    int32_t *P = perm + seg * L;
    int32_t *I = inv + seg * L;
    for (int it = 0; it < kKeysPerWarp / 32; ++it) {
        const int pos = wlo + it * 32 + lane;
        int key = pos < L ? keys[pos] : -1;
        if (key >= nb) key = -1;
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        int base = 0;
        if (key >= 0) base = hist[key];
        __syncwarp();
        if (key >= 0) {
            const int slot = base + __popc(peers & lt);
            P[slot] = pos;
            I[pos] = slot;
            if ((peers & lt) == 0) hist[key] = base + __popc(peers);
        }
        __syncwarp();
    }
}

}  // namespace

cudaError_t sort_launch(const Problem &p, const int32_t *buckets, int32_t *perm, int32_t *inv,
                        int32_t *bstart, int32_t *counts, cudaStream_t st)
{
    const int tiles = sort_tiles(p.L);
    const unsigned segs = (unsigned)p.n_seg();
    cudaError_t e;
    const size_t smem1 = sizeof(int) * p.nb;
    e = cudaFuncSetAttribute(sort_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem1);
    if (e != cudaSuccess) return e;
    sort_count_kernel<<<dim3(tiles, segs), 512, smem1, st>>>(buckets, p.L, p.nb, tiles, counts);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    sort_scan_kernel<<<segs, 1024, 0, st>>>(counts, p.nb, tiles, p.L, bstart);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const size_t smem3 = sizeof(int) * kScatterWarps * p.nb;
    e = cudaFuncSetAttribute(sort_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem3);
    if (e != cudaSuccess) return e;
    sort_scatter_kernel<<<dim3(tiles, segs), kScatterWarps * 32, smem3, st>>>(
        buckets, counts, p.L, p.nb, tiles, perm, inv);
    return cudaGetLastError();
}

}  // namespace lsh
