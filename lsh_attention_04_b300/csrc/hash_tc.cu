// hash_tc.cu -- angular LSH on the tcgen05 tensor cores (bf16 or fp16 inputs, fp32
// accumulation).
//
// "Reformer" glossary (ultralytics.com), section "Atencion LSH": project every token
// with a random matrix R and take the position of the largest entry of [xR, -xR] as the
// bucket.  modulabs-hub Reformer notes, "Locality sensitive hashing": R_r has
// n_buckets/2 columns; the + and - halves are concatenated.  Several rounds use
// independent R_r ("Multi-round LSH attention").
//
// The projection x.R_r is a dense contraction, so it runs on the tensor cores:
//  * The columns of all rounds are laid out one round after another (each round padded
//    to a multiple of 32 columns with zero columns that never win) and cut into MMA
//    chunks of at most 128 columns: several whole rounds per chunk when a round has at
//    most 128 columns, otherwise 128-column parts of one round.
//  * Consecutive rounds form a "group" whose packed R image (<= 128 KB) stays resident in
//    shared memory for the whole kernel.  A pre-pass (lsh_rpack_kernel) writes that image
//    in the canonical K-major 128-byte-swizzled layout, so one bulk TMA copy stages it.
//  * Persistent CTAs: ctas_per_group CTAs per group walk the 128-token tiles in the same
//    order, so the CTAs of all groups read a tile of qk within a short time window and
//    only the first one fetches it from HBM (the others hit L2).
//  * Warp roles (12 warps): warp 8 issues TMA loads of the qk tile (2-D tensor map,
//    128-byte swizzle, 2-4 stages) and owns TMEM; warps 10-11 issue tcgen05.mma
//    M=128 x N=chunk x K=16 (each a whole warp, one lane elected per instruction); warps
//    0-7 are two epilogue warpgroups that read the projections with tcgen05.ld and keep,
//    per token and round, the entry of largest magnitude (first index on ties); warp 9
//    computes 1/|x| of each token from the staged tile (first group only).
//  * Four 128-column TMEM accumulators, two per epilogue warpgroup: warpgroup e and its
//    MMA warp 10 + e take the tiles it % 2 == e and alternate the tile's chunks between
//    accumulators 2e and 2e + 1, so the warpgroup scans one chunk while the next one is
//    being computed (a single accumulator per warpgroup left it waiting for every
//    refill), and it sees each round whole.
//  * Bucket rule: the largest entry of [p, -p] is the entry of p with the largest |p_j|,
//    taken with its sign: bucket = j if p_j >= 0, n_buckets/2 + j otherwise.  Scanning j
//    in order with a strict comparison keeps the first index.  Two entries of equal
//    magnitude and opposite sign have a zero top-1/top-2 margin, i.e. they are a near-tie.
// Every wait is bounded (see sm100::wait); on a timeout the kernel records the place in
// the workspace status block and winds down.
#include <math.h>

#include "sm100.cuh"

namespace lsh {
namespace {

using namespace sm100;

constexpr int kTileM = 128;          // tokens per tile = MMA M = TMEM lanes
constexpr int kChunkMax = 128;       // MMA N per chunk (TMEM columns per accumulator)
constexpr int kTmemBufs = 4;         // accumulators: 4 x 128 TMEM columns
constexpr int kRCapBytes = 128 * 1024;
constexpr int kMaxXStages = 4;         // qk tile stages (as many as shared memory holds)
constexpr size_t kSmemCap = 227 * 1024;
constexpr int kEpiGroups = 2;         // epilogue warpgroups, two accumulators each
constexpr int kMmaWarps = kEpiGroups; // one MMA-issuing warp per epilogue warpgroup
constexpr int kEpiWarps = 4 * kEpiGroups;
constexpr int kProdWarp = kEpiWarps;      // producer (also the TMEM owner)
constexpr int kNormWarp = kEpiWarps + 1;  // 1 / |x|
constexpr int kMma0 = kEpiWarps + 2;      // MMA issuers kMma0 .. kMma0 + 1
// 12 warps: a multiple of 4, so every scheduler holds the same number of warps
constexpr int kThreads = 12 * 32;

struct HashPlan {
    long long n_tok;
    int L, d, half, hp, n_rounds;
    int split;            // 0: chunk = rpc whole rounds; 1: round = cpr chunks
    int rpc, cpr, rpg;    // rounds per chunk, chunks per round, rounds per group
    int n_groups, ctas_per_group, n_tiles;
    int group_bytes;      // bytes of one group's packed R image (stride in rpack)
    int x_stages;         // qk tile stages in shared memory
    int f16;              // inputs are fp16 (else bf16)
};

// ---- geometry of chunk k of a group with nr rounds (host and device) ----
__host__ __device__ __forceinline__ int n_chunks(const HashPlan &P, int nr) {
    return P.split ? nr * P.cpr : (nr + P.rpc - 1) / P.rpc;
}
__host__ __device__ __forceinline__ int chunk_col0(const HashPlan &P, int k) {
    return P.split ? (k / P.cpr) * P.hp + kChunkMax * (k % P.cpr) : k * P.rpc * P.hp;
}
__host__ __device__ __forceinline__ int chunk_width(const HashPlan &P, int nr, int k) {
    if (P.split) return min(kChunkMax, P.hp - kChunkMax * (k % P.cpr));
    return min(P.rpc, nr - k * P.rpc) * P.hp;
}

// ---- R pre-pack: R [n_rounds][d][half] -> per-group K-major SW128 images ----
__global__ void __launch_bounds__(256)
lsh_rpack_kernel(const uint16_t *__restrict__ R, HashPlan P, uint8_t *__restrict__ rpack)
{
    const int kch = P.d / 8;  // 16-byte pieces per packed row
    const long long total = (long long)P.n_rounds * P.hp * kch;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int c = (int)(i % kch);
        const int jp = (int)((i / kch) % P.hp);
        const int r = (int)(i / ((long long)kch * P.hp));
        const int g = r / P.rpg, r_in = r % P.rpg;
        const int nr = min(P.rpg, P.n_rounds - g * P.rpg);
        int k, n;
        if (P.split) { k = r_in * P.cpr + jp / kChunkMax; n = jp % kChunkMax; }
        else { k = r_in / P.rpc; n = (r_in % P.rpc) * P.hp + jp; }
        const int width = chunk_width(P, nr, k);
        const size_t dst = (size_t)g * P.group_bytes + (size_t)chunk_col0(P, k) * P.d * 2 +
                           kmajor_sw128_off(n, c * 8, width);
        __align__(16) uint16_t v[8];       // 16-bit values moved as bits (zero is 0 in both types)
#pragma unroll
        for (int e = 0; e < 8; ++e)
            v[e] = jp < P.half ? R[((size_t)r * P.d + c * 8 + e) * P.half + jp] : (uint16_t)0;
        *reinterpret_cast<uint4 *>(rpack + dst) = *reinterpret_cast<const uint4 *>(v);
    }
}

// ---- the hash kernel ----
struct __align__(8) HashBarriers {
    uint64_t x_full[kMaxXStages], x_empty[kMaxXStages];
    uint64_t tm_full[kTmemBufs], tm_empty[kTmemBufs];
    uint64_t r_full, mma_done;
    uint32_t tmem_base;
    int abort_flag;
};

__device__ __forceinline__ void write_bucket(int32_t *buckets, const HashPlan &P, long long tok,
                                             int r, float best, int bidx) {
    const long long bh = tok / P.L, l = tok - bh * P.L;
    buckets[((size_t)bh * P.n_rounds + r) * P.L + l] = best >= 0.f ? bidx : P.half + bidx;
}

// Entry of largest magnitude among 32 projections (columns j0 .. j0+31 of a round), first
// index on ties, merged into the running (best, bidx).  A pairwise tree (depth 5) keeps the
// dependency chains short; at every merge the left (earlier) operand wins ties, so the
// result is the first index of the largest |p|.  Zero-padding columns project to exactly 0
// and can never win against an earlier column.
__device__ __forceinline__ void scan32(const uint32_t (&v)[32], int j0, float &best, int &bidx) {
    float b[16];
    int ix[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const float x0 = __uint_as_float(v[2 * k]), x1 = __uint_as_float(v[2 * k + 1]);
        const bool t = fabsf(x1) > fabsf(x0);
        b[k] = t ? x1 : x0;
        ix[k] = 2 * k + (t ? 1 : 0);
    }
#pragma unroll
    for (int w = 8; w >= 1; w >>= 1) {
#pragma unroll
        for (int k = 0; k < w; ++k) {
            const bool t = fabsf(b[2 * k + 1]) > fabsf(b[2 * k]);
            b[k] = t ? b[2 * k + 1] : b[2 * k];
            ix[k] = t ? ix[2 * k + 1] : ix[2 * k];
        }
    }
    if (fabsf(b[0]) > fabsf(best)) { best = b[0]; bidx = j0 + ix[0]; }
}

// One 32-column batch of the epilogue: (r, j) is the round and the column within it of
// the batch's first column; the bucket is written when the round's last batch is done.
__device__ __forceinline__ void scan_batch(const uint32_t (&v)[32], const HashPlan &P, int &r, int &j,
                                           int &cur, float &best, int &bidx, bool live,
                                           int32_t *buckets, long long tok, int r0) {
    if (r != cur) {
        cur = r;
        best = 0.f;
        bidx = 0;
    }
    scan32(v, j, best, bidx);
    j += 32;
    if (j >= P.hp) {
        if (live) write_bucket(buckets, P, tok, r0 + r, best, bidx);
        j = 0;
        ++r;
    }
}

__global__ void __launch_bounds__(kThreads, 1)
lsh_hash_tc_kernel(const __grid_constant__ CUtensorMap xmap, const uint8_t *__restrict__ rpack,
                   const HashPlan P, int32_t *__restrict__ buckets, float *__restrict__ inv_norm,
                   StatusBlock *status)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ HashBarriers sb;
    // 1024-byte aligned base, derived from the shared array by pointer arithmetic so the
    // compiler keeps the shared state space (shared loads, not generic ones)
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int x_bytes = kTileM * P.d * 2;
    uint8_t *Rs = smem;
    uint8_t *Xs = smem + P.group_bytes;  // group_bytes is a multiple of 1024

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = blockIdx.x / P.ctas_per_group;
    const int cj = blockIdx.x % P.ctas_per_group;
    const int r0 = g * P.rpg;
    const int nr = min(P.rpg, P.n_rounds - r0);
    const int nch = n_chunks(P, nr);
    volatile int *abort_flag = &sb.abort_flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < P.x_stages; ++s) {
            mbar_init(&sb.x_full[s], 1);
            mbar_init(&sb.x_empty[s], kMmaWarps + (g == 0 ? 1 : 0));
        }
        for (int b = 0; b < kTmemBufs; ++b) {
            mbar_init(&sb.tm_full[b], 1);
            mbar_init(&sb.tm_empty[b], 128);
        }
        mbar_init(&sb.r_full, 1);
        mbar_init(&sb.mma_done, kMmaWarps);
        sb.abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == kProdWarp) tmem_alloc(&sb.tmem_base, 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = sb.tmem_base;

    if (warp == kProdWarp) {
        // ---------------- producer: R group once, then qk tiles ----------------
        if (lane == 0) {
            prefetch_tmap(&xmap);
            const int rbytes = nr * P.hp * P.d * 2;
            mbar_expect_tx(&sb.r_full, (uint32_t)rbytes);
            const uint8_t *src = rpack + (size_t)g * P.group_bytes;
            for (int off = 0; off < rbytes; off += 32768)
                bulk_g2s(Rs + off, src + off, (uint32_t)min(32768, rbytes - off), &sb.r_full);
            uint32_t pending = 0;  // stages with a fill in flight (for the wind-down)
            int it = 0;
            for (int t = cj; t < P.n_tiles; t += P.ctas_per_group, ++it) {
                const int s = it % P.x_stages;
                const uint32_t ph = (it / P.x_stages) & 1;
                if (!wait(&sb.x_empty[s], ph ^ 1, abort_flag, status, 0x101)) break;
                mbar_expect_tx(&sb.x_full[s], (uint32_t)x_bytes);
                for (int kb = 0; kb < P.d / 64; ++kb)
                    tma_load_2d(Xs + s * x_bytes + kb * kTileM * 128, &xmap, kb * 64, t * kTileM,
                                &sb.x_full[s]);
                pending |= 1u << s;
            }
            // wind-down: every issued copy has landed before the CTA exits
            int last = it - 1;
            for (int k = 0; k < P.x_stages && last - k >= 0; ++k) {
                const int i2 = last - k, s = i2 % P.x_stages;
                if (pending & (1u << s)) {
                    const uint32_t ph = (i2 / P.x_stages) & 1;
                    int dummy = 0;
                    wait(&sb.x_full[s], ph, &dummy, status, 0x102);
                }
            }
            int dummy = 0;
            wait(&sb.r_full, 0, &dummy, status, 0x103);
        }
    } else if (warp >= kMma0 && warp < kMma0 + kMmaWarps) {
        // ---------------- MMA issuers: warp kMma0 + e feeds epilogue warpgroup e ----------
        // Each issuer is a whole converged warp (the MMA wrappers elect one lane).  Tile
        // `it` belongs to warpgroup it % 2; its chunks alternate between the warpgroup's
        // accumulators 2e and 2e + 1 (use u of the warpgroup goes to 2e + u % 2).
        {
            const int mi = warp - kMma0;
            bool ok = wait_w(&sb.r_full, 0, abort_flag, status, 0x201);
            fence_after_sync();
            int it = 0;
            const uint32_t rs = smem_u32(Rs), xs = smem_u32(Xs);
            for (int t = cj; ok && t < P.n_tiles; t += P.ctas_per_group, ++it) {
                const int s = it % P.x_stages;
                if (!(ok = wait_w(&sb.x_full[s], (it / P.x_stages) & 1, abort_flag, status, 0x202))) break;
                fence_after_sync();
                bool touched = false;
                if (it % kEpiGroups == mi) {
                    for (int k = 0; k < nch; ++k) {
                        const int use = (it / kEpiGroups) * nch + k;
                        const int b = 2 * mi + (use & 1);
                        if (!(ok = wait_w(&sb.tm_empty[b], ((use >> 1) & 1) ^ 1, abort_flag, status, 0x203))) break;
                        fence_after_sync();
                        const int width = chunk_width(P, nr, k);
                        const uint32_t idesc = idesc_16(kTileM, width, 0, 0, P.f16);
                        const uint32_t rbase = rs + chunk_col0(P, k) * P.d * 2;
                        for (int ks = 0; ks < P.d / 16; ++ks) {
                            const int kb = ks >> 2, ko = (ks & 3) * 32;
                            const uint64_t a = smem_desc(xs + s * x_bytes + kb * kTileM * 128 + ko, 16, 1024);
                            const uint64_t bd = smem_desc(rbase + kb * width * 128 + ko, 16, 1024);
                            mma_ss(tmem + b * kChunkMax, a, bd, idesc, ks > 0);
                        }
                        mma_commit(smem_u32(&sb.tm_full[b]));
                        touched = true;
                    }
                }
                if (!ok) break;
                // this warp is done with the staged tile once its MMAs (if any) complete
                if (touched) mma_commit(smem_u32(&sb.x_empty[s]));
                else if (lane == 0) mbar_arrive(&sb.x_empty[s]);
                __syncwarp();
            }
            // wind-down: all issued MMAs complete before TMEM is released
            mma_commit(smem_u32(&sb.mma_done));
            int dummy = 0;
            wait_w(&sb.mma_done, 0, &dummy, status, 0x204);
        }
    } else if (warp == kNormWarp) {
        // ---------------- 1/|x| of each token (first group only) ----------------
        if (g == 0) {
            int it = 0;
            for (int t = cj; t < P.n_tiles; t += P.ctas_per_group, ++it) {
                const int s = it % P.x_stages;
                bool ok = wait(&sb.x_full[s], (it / P.x_stages) & 1, abort_flag, status, 0x301);
                if (!__all_sync(0xffffffffu, ok)) break;
                const uint8_t *xt = Xs + s * x_bytes;
                for (int rr = 0; rr < 4; ++rr) {
                    const int row = lane + 32 * rr;
                    float acc = 0.f;
                    for (int kb = 0; kb < P.d / 64; ++kb) {
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            const uint4 q = *reinterpret_cast<const uint4 *>(
                                xt + kb * kTileM * 128 + row * 128 + ((c ^ (row & 7)) << 4));
                            const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&q);
                            const __half2 *hh = reinterpret_cast<const __half2 *>(&q);
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 f = P.f16 ? __half22float2(hh[e]) : __bfloat1622float2(h[e]);
                                acc = fmaf(f.x, f.x, acc);
                                acc = fmaf(f.y, f.y, acc);
                            }
                        }
                    }
                    const long long tok = (long long)t * kTileM + row;
                    if (tok < P.n_tok) inv_norm[tok] = acc > 0.f ? 1.0f / sqrtf(acc) : 0.f;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sb.x_empty[s]);
            }
        }
    } else if (warp < kEpiWarps) {
        // ---------------- epilogue warpgroups: warpgroup e takes the tiles it % 2 == e ------
        // It sees every chunk of its tile (alternately in its accumulators 2e, 2e + 1),
        // hence every round whole: no merging between warpgroups.
        const int e = warp >> 2, q = warp & 3;
        const int row = q * 32 + lane;
        const uint32_t tlane0 = tmem + ((uint32_t)(q * 32) << 16);
        int it = 0;
        bool ok = true;
        for (int t = cj; ok && t < P.n_tiles; t += P.ctas_per_group, ++it) {
            if (it % kEpiGroups != e) continue;
            const long long tok = (long long)t * kTileM + row;
            const bool live = tok < P.n_tok;
            int cur = -1;
            float best = 0.f;
            int bidx = 0;
            for (int k = 0; k < nch; ++k) {
                const int use = (it / kEpiGroups) * nch + k;
                const int buf = 2 * e + (use & 1);
                const uint32_t tlane = tlane0 + buf * kChunkMax;
                bool w = wait(&sb.tm_full[buf], (use >> 1) & 1, abort_flag, status, 0x401);
                if (!(ok = __all_sync(0xffffffffu, w))) break;
                fence_after_sync();
                const int width = chunk_width(P, nr, k);
                // round and in-round column of the chunk's first column
                int rr, jj;
                if (P.split) { rr = k / P.cpr; jj = kChunkMax * (k % P.cpr); }
                else { const int col = chunk_col0(P, k); rr = col / P.hp; jj = col - rr * P.hp; }
                // 32-column batches, one at a time; the accumulator goes back to its MMA
                // warp as soon as its last batch is in registers.
                const int nbat = width / 32;
                for (int q2 = 0; q2 < nbat; ++q2) {
                    uint32_t va[32];
                    tmem_ld32(tlane + 32 * q2, va);
                    tmem_wait_ld(va);
                    if (q2 == nbat - 1) {
                        fence_before_sync();
                        mbar_arrive(&sb.tm_empty[buf]);
                    }
                    scan_batch(va, P, rr, jj, cur, best, bidx, live, buckets, tok, r0);
                }
            }
        }
    }

    fence_before_sync();
    __syncthreads();
    if (warp == kProdWarp) {
        __syncwarp();
        fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

bool make_plan(const Problem &p, HashPlan &P, int num_sms)
{
    P.n_tok = p.n_tok();
    P.f16 = p.dtype == LSH_F16;
    P.L = p.L;
    P.d = p.d;
    P.half = p.nb / 2;
    P.hp = (P.half + 31) / 32 * 32;
    P.n_rounds = p.n_rounds;
    const int cap = kRCapBytes / (p.d * 2);
    if (P.hp > cap) return false;
    P.split = P.hp > kChunkMax;
    P.rpc = P.split ? 1 : kChunkMax / P.hp;
    P.cpr = P.split ? (P.hp + kChunkMax - 1) / kChunkMax : 1;
    const int rpg_max = cap / P.hp;
    P.n_groups = (p.n_rounds + rpg_max - 1) / rpg_max;
    P.rpg = (p.n_rounds + P.n_groups - 1) / P.n_groups;
    P.n_tiles = (int)((P.n_tok + kTileM - 1) / kTileM);
    P.ctas_per_group = num_sms / P.n_groups;
    if (P.ctas_per_group < 1) P.ctas_per_group = 1;
    if (P.ctas_per_group > P.n_tiles) P.ctas_per_group = P.n_tiles;
    P.group_bytes = P.rpg * P.hp * p.d * 2;  // multiple of 32*64*2 = 4096
    const size_t x_bytes = (size_t)kTileM * p.d * 2;
    const size_t room = kSmemCap - 1024 - (size_t)P.group_bytes;
    P.x_stages = (int)(room / x_bytes);
    if (P.x_stages > kMaxXStages) P.x_stages = kMaxXStages;
    if (P.x_stages < 2) return false;
    return true;
}

size_t smem_bytes(const HashPlan &P)
{
    return 1024 + (size_t)P.group_bytes + (size_t)P.x_stages * kTileM * P.d * 2;
}

int num_sms_current()
{
    int dev = 0, n = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n;
}

}  // namespace

bool hash_tc_supported(const Problem &p)
{
    if (p.dtype != LSH_BF16 && p.dtype != LSH_F16) return false;
    HashPlan P;
    return make_plan(p, P, 148);
}

size_t hash_tc_pack_bytes(const Problem &p)
{
    HashPlan P;
    if (!make_plan(p, P, 148)) return 0;
    return (size_t)P.n_groups * P.group_bytes;
}

int hash_tc_launches(const Problem &) { return 2; }

cudaError_t hash_tc(const Problem &p, const void *qk, const void *R, void *rpack, int32_t *buckets,
                    float *inv_norm, StatusBlock *status, cudaStream_t st)
{
    HashPlan P;
    if (!make_plan(p, P, num_sms_current())) return cudaErrorNotSupported;
    CUtensorMap xmap;       // the copy moves 16-bit values; the map's element type is only their size
    if (!make_tmap_2d_bf16(&xmap, qk, (uint64_t)P.n_tok, (uint64_t)p.d, 64, kTileM))
        return cudaErrorNotSupported;
    const long long pack_items = (long long)P.n_rounds * P.hp * (p.d / 8);
    const long long want = (pack_items + 255) / 256;
    const int pack_blocks = (int)(want < 4096 ? want : 4096);
    lsh_rpack_kernel<<<pack_blocks, 256, 0, st>>>((const uint16_t *)R, P, (uint8_t *)rpack);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t smem = smem_bytes(P);
    e = cudaFuncSetAttribute(lsh_hash_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    lsh_hash_tc_kernel<<<P.n_groups * P.ctas_per_group, kThreads, smem, st>>>(
        xmap, (const uint8_t *)rpack, P, buckets, inv_norm, status);
    return cudaGetLastError();
}

}  // namespace lsh
