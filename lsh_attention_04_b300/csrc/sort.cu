// sort.cu -- segmented stable counting sort of bucket ids, one segment per
// (batch, head, round).
//
// ai-scholar.tech Reformer article, "LSH attention": after hashing, sort by LSH bucket;
// modulabs-hub notes, "LSH attention": the bucketed keys are put in order so that a
// chunked batch computation becomes possible.  Ties keep position order, so the result
// is the unique permutation that orders tokens by (bucket, position).
//
// Segments of up to 65536 keys: one launch (sort_cluster_kernel), one cluster of C CTAs
// per segment, C = ceil(L / 16384).  CTA r ranks the positions [16384 r, 16384 (r+1)) and
// owns the output slots of the same range.
//   1. per-warp histograms of the CTA's positions (16-bit counters, shared atomics);
//   2. after a cluster barrier every CTA reads the others' per-bucket totals through
//      distributed shared memory: a block-wide exclusive scan over buckets gives bstart,
//      and each (warp, bucket) its first slot (after the bucket's keys in lower-ranked
//      CTAs and lower warps);
//   3. ranking in position order, 32 keys per warp step: equal keys are found with a
//      per-warp table (each lane writes its lane index at its key and reads back the last
//      writer) and five ballots on that 5-bit value; slot = the warp's running slot for
//      the bucket + the number of equal keys in lower lanes.  inv[pos] = slot goes
//      straight out (coalesced) and pos goes into the shared-memory copy of the sorted
//      order held by the CTA that owns the slot;
//   4. after a second cluster barrier each CTA writes its slot range of perm, coalesced.
// Keys are loaded eight steps ahead so the L2 latency overlaps.  Positions and slots fit
// 16 bits.
//
// Larger segments: three launches, no inter-CTA waiting:
//   1. count   per 4096-key tile: a shared-memory histogram, written bucket-major as
//              counts[seg][bucket][tile];
//   2. scan    per segment: exclusive scan of counts in (bucket, tile) order gives every
//              tile's first output slot for each bucket, and bstart;
//   3. scatter per tile: 16 warps each own 256 consecutive keys; warp-level ranking
//              (__match_any_sync + popc) against per-warp shared histograms gives each
//              key its stable slot; writes perm[slot] = pos and inv[pos] = slot.
#include <cooperative_groups.h>

#include "internal.cuh"

namespace cg = cooperative_groups;

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

constexpr int kSegAhead = 8;          // iterations of keys loaded ahead
constexpr int kSegMaxL = 65536;       // positions and slots fit 16 bits

__host__ __device__ constexpr size_t a16(size_t x) { return (x + 15) & ~(size_t)15; }
constexpr int kClusterShift = 14;
constexpr int kClusterKeys = 1 << kClusterShift;   // positions per CTA of a cluster

// Lanes of the warp whose 5-bit values v are equal: the AND over the bits of the ballot
// of that bit or of its complement.
__device__ __forceinline__ unsigned equal_lanes(int v)
{
    unsigned m = 0xffffffffu;
#pragma unroll
    for (int i = 0; i < 5; ++i) {
        const unsigned bit = (v >> i) & 1u;
        m &= __ballot_sync(0xffffffffu, bit) ^ (bit - 1u);
    }
    return m;
}

// Block-wide exclusive scan of one int per thread; returns the exclusive prefix.
template <int W>
__device__ __forceinline__ int block_exclusive_scan(int v, int *tmp)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) tmp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < W ? tmp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < W) tmp[lane] = w;
    }
    __syncthreads();
    return x - v + (warp > 0 ? tmp[warp - 1] : 0);
}

// One segment per cluster of C CTAs (C = 1 for short segments).  CTA r of the cluster
// ranks the positions [r*Lc, (r+1)*Lc) and owns the output slots of the same range: it
// receives perm's entries for those slots from every CTA of the cluster (distributed
// shared memory) and writes them out.  W warps per CTA.
//   counts: per-warp 16-bit counters, two to a 32-bit word, bumped with shared atomics;
//   ranks:  each lane writes its lane index into a per-warp table at its key and reads
//           back the last writer, one lane per distinct key; equal keys are then equal
//           5-bit table values, found with five ballots.
template <int W>
__global__ void __launch_bounds__(W * 32)
sort_cluster_kernel(const int32_t *__restrict__ buckets, int L, int nb, int Lc, int lc_shift,
                    int32_t *__restrict__ perm, int32_t *__restrict__ inv,
                    int32_t *__restrict__ bstart, int vec_out)
{
    constexpr int T = W * 32;
    cg::cluster_group cluster = cg::this_cluster();
    const int C = (int)cluster.num_blocks();
    const int r = (int)cluster.block_rank();
    const int nbp = (nb + 1) & ~1;                    // per-warp stride, even
    extern __shared__ __align__(16) uint8_t seg_smem[];
    __shared__ int scan_tmp[32];
    uint16_t *lperm = reinterpret_cast<uint16_t *>(seg_smem);                  // [Lc]
    uint8_t *p8 = seg_smem + a16((size_t)2 * Lc);
    uint16_t *whist = reinterpret_cast<uint16_t *>(p8);                        // [W][nbp]
    p8 += a16((size_t)2 * W * nbp);
    int *ctot = reinterpret_cast<int *>(p8);                                   // [nb]
    p8 += a16((size_t)4 * nb);
    uint8_t *tab = p8 + (size_t)(threadIdx.x >> 5) * nbp;                      // [W][nbp]
    const long seg = blockIdx.x / C;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const unsigned lt = (1u << lane) - 1u;
    const int32_t *keys = buckets + seg * L;
    const int plo = r * Lc, phi = min(L, plo + Lc);
    const int per = (((phi - plo + W - 1) / W) + 31) & ~31;
    const int wlo = plo + warp * per, whi = min(phi, wlo + per);
    uint16_t *h = whist + warp * nbp;
    unsigned *h32 = reinterpret_cast<unsigned *>(h);

    for (int i = threadIdx.x; i < W * nbp / 2; i += T) reinterpret_cast<unsigned *>(whist)[i] = 0u;
    __syncthreads();

    // 1. per-warp counts (ids outside [0, nb) are skipped)
    for (int base = wlo; base < whi; base += 32 * kSegAhead) {
        int k[kSegAhead];
#pragma unroll
        for (int j = 0; j < kSegAhead; ++j) {
            const int pos = base + j * 32 + lane;
            k[j] = pos < whi ? __ldg(keys + pos) : -1;
        }
#pragma unroll
        for (int j = 0; j < kSegAhead; ++j)
            if ((unsigned)k[j] < (unsigned)nb) atomicAdd(h32 + (k[j] >> 1), 1u << ((k[j] & 1) << 4));
    }
    __syncthreads();
    for (int b = threadIdx.x; b < nb; b += T) {
        int c = 0;
        for (int w = 0; w < W; ++w) c += whist[w * nbp + b];
        ctot[b] = c;
    }
    cluster.sync();                      // every CTA's per-bucket totals are visible

    // 2. bucket starts over the whole segment, and each warp's first slot per bucket
    // (after the bucket's keys in lower-ranked CTAs and in lower warps)
    const int bpt = (nb + T - 1) / T;
    const int b0 = min(nb, (int)threadIdx.x * bpt), b1 = min(nb, b0 + bpt);
    int local = 0;
    for (int b = b0; b < b1; ++b)
        for (int q = 0; q < C; ++q) local += cluster.map_shared_rank(ctot, q)[b];
    int run = block_exclusive_scan<W>(local, scan_tmp);
    int32_t *bs = bstart + seg * (nb + 1);
    for (int b = b0; b < b1; ++b) {
        int tot = 0, pre = 0;
        for (int q = 0; q < C; ++q) {
            const int v = cluster.map_shared_rank(ctot, q)[b];
            tot += v;
            pre += q < r ? v : 0;
        }
        if (r == 0) bs[b] = run;
        int first = run + pre;
        for (int w = 0; w < W; ++w) {
            const int c = whist[w * nbp + b];
            whist[w * nbp + b] = (uint16_t)first;  // a slot below L whenever c > 0
            first += c;
        }
        run += tot;
    }
    if (r == 0 && threadIdx.x == 0) bs[nb] = L;
    __syncthreads();

    // 3. stable ranks in position order; perm's entry goes to the CTA owning the slot
    int32_t *I = inv + seg * L;
    for (int base = wlo; base < whi; base += 32 * kSegAhead) {
        int k[kSegAhead];
#pragma unroll
        for (int j = 0; j < kSegAhead; ++j) {
            const int pos = base + j * 32 + lane;
            k[j] = pos < whi ? __ldg(keys + pos) : -1;
        }
#pragma unroll
        for (int j = 0; j < kSegAhead; ++j) {
            const int pos = base + j * 32 + lane;
            const bool valid = (unsigned)k[j] < (unsigned)nb;
            if (valid) tab[k[j]] = (uint8_t)lane;
            __syncwarp();
            const int rep = valid ? tab[k[j]] : lane;    // no valid lane has an invalid one's index
            const unsigned peers = equal_lanes(rep);
            const int first = valid ? h[k[j]] : 0;
            __syncwarp();
            if (valid) {
                const int slot = first + __popc(peers & lt);
                const int owner = slot >> lc_shift;
                cluster.map_shared_rank(lperm, owner)[slot - (owner << lc_shift)] = (uint16_t)pos;
                I[pos] = slot;
                if ((peers & lt) == 0) h[k[j]] = (uint16_t)(first + __popc(peers));
            }
            __syncwarp();
        }
    }
    cluster.sync();                      // every entry of this CTA's slots has arrived

    // 4. perm for this CTA's slots, in slot order (16-byte stores when aligned)
    int32_t *P = perm + seg * L + plo;
    const int n = phi - plo;
    if (vec_out) {
        const uint2 *src = reinterpret_cast<const uint2 *>(lperm);
        int4 *dst = reinterpret_cast<int4 *>(P);
        for (int i = threadIdx.x; i < n / 4; i += T) {
            const uint2 v = src[i];
            dst[i] = make_int4((int)(v.x & 0xffffu), (int)(v.x >> 16), (int)(v.y & 0xffffu),
                               (int)(v.y >> 16));
        }
    } else {
        for (int i = threadIdx.x; i < n; i += T) P[i] = lperm[i];
    }
}

size_t cluster_smem_bytes(int Lc, int nb, int W)
{
    const size_t nbp = (size_t)((nb + 1) & ~1);
    return a16((size_t)2 * Lc) + a16(2 * W * nbp) + a16((size_t)4 * nb) + a16(W * nbp);
}

// Lc: positions per CTA, a power of two (1 << lc_shift) when C > 1.
template <int W>
cudaError_t launch_cluster_sort(const Problem &p, int C, int Lc, int lc_shift,
                                const int32_t *buckets, int32_t *perm, int32_t *inv,
                                int32_t *bstart, cudaStream_t st)
{
    const size_t smem = cluster_smem_bytes(Lc, p.nb, W);
    cudaError_t e = cudaFuncSetAttribute(sort_cluster_kernel<W>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int vec = (p.L % 4 == 0) && ((uintptr_t)perm % 16 == 0);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.n_seg() * C));
    cfg.blockDim = dim3(W * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, sort_cluster_kernel<W>, buckets, p.L, p.nb, Lc, lc_shift,
                              perm, inv, bstart, vec);
}

}  // namespace

// The one-launch path takes every segment of up to 65536 keys: its shared memory stays
// below the limit for every bucket count the library accepts (<= 2048).
int sort_launches(const Problem &p)
{
    return p.L <= kSegMaxL ? 1 : 3;
}

cudaError_t sort_launch(const Problem &p, const int32_t *buckets, int32_t *perm, int32_t *inv,
                        int32_t *bstart, int32_t *counts, cudaStream_t st)
{
    const int tiles = sort_tiles(p.L);
    const unsigned segs = (unsigned)p.n_seg();
    cudaError_t e;
    if (p.L <= kSegMaxL) {
        // segments longer than one CTA's share split over a cluster of power-of-two slices
        // (slot -> owner is a shift); shorter ones take one CTA
        const int C = (p.L + kClusterKeys - 1) / kClusterKeys;     // 1 .. 4
        const int Lc = C > 1 ? kClusterKeys : ((p.L + 3) & ~3);
        const int shift = C > 1 ? kClusterShift : 30;
        if (Lc >= 4096 && cluster_smem_bytes(Lc, p.nb, 16) <= kSortSegSmemMax)
            return launch_cluster_sort<16>(p, C, Lc, shift, buckets, perm, inv, bstart, st);
        if (cluster_smem_bytes(Lc, p.nb, 4) <= kSortSegSmemMax)
            return launch_cluster_sort<4>(p, C, Lc, shift, buckets, perm, inv, bstart, st);
    }
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
