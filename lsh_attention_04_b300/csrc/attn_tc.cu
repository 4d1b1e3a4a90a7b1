// attn_tc.cu -- chunked look-one-back LSH attention on the tcgen05 tensor cores (bf16
// inputs, fp32 accumulation, chunk 64, d = 64 or 128).
//
// "Reformer" glossary (ultralytics.com), section "Atencion LSH": the bucket-sorted
// sequence is cut into equal chunks; each token attends to its own chunk and the
// previous one.  modulabs-hub Reformer notes, section "LSH attention": keys outside the
// query's bucket get -infinity, the token itself is removed (under shared QK it would
// always score highest; it stays only when nothing else is left), and in the causal
// case only earlier positions remain.  Keys are L2-normalised, queries are not.
//
// Tile = 128 consecutive sorted rows (chunks 2t and 2t+1 of one (batch, head, round)
// segment).  Their keys live in the 192-row window of chunks 2t-1, 2t, 2t+1: rows of
// chunk 2t use window columns 0-127, rows of chunk 2t+1 use columns 64-191.
//   S = Q K^T     one chain of tcgen05.mma M=128, N=192, K=16 steps over d; A (window
//                 rows 64-191) and B (all 192 rows) come from the tile's own Q/K window
//                 buffer in shared memory; fp32 into TMEM (2 x 192 columns).
//   P             packed bf16 pairs written into TMEM over S: the 32 keys of S columns
//                 32j..32j+31 go to columns 32j..32j+15, so every warp overwrites only
//                 S columns it has already read.
//   O = P V       tcgen05.mma M=128, N=d, K=16 steps with A read from TMEM and V as an
//                 MN-major shared-memory operand (the same 128-byte-swizzled row layout
//                 as Q/K).
// One thread issues a tcgen05.mma only every few hundred cycles whatever N is, so the S
// chain and the P V chain are issued from two different warps and overlap.
// Masks: sorted order keeps each bucket in one run, so the keys of sorted row s form one
// interval of window columns: [max(window start, bucket start), causal ? s : min(window
// end, bucket end)), minus s itself when not causal.  The loaders fetch the bucket's run
// bounds; the softmax needs no per-key bucket test.  A row with no key but itself gives
// its own column weight 1, so P V returns v_i exactly; its lse is the self logit -1e5.
// Softmax without a running maximum: with unit keys every score of query i is bounded
// by m_i = |scale| * |q_i| (Cauchy-Schwarz), so p = exp(s - m_i) cannot overflow.  If
// m_i is so large that every p could underflow (|scale| |q_i| log2 e > 64), the warp
// first takes the exact row maximum instead.  lse = m_i + log(sum p).
// Rows are gathered through the sort permutation by TMA tile::gather4 (4 rows per
// instruction, 128-byte swizzle): each tile's 192 Q/K rows into one of two window
// buffers (the look-back chunk is gathered again for the next tile, which keeps the
// window contiguous for the single N=192 MMA), and V rows with the row metadata into a
// ring of 6 chunk slots (chunk c in slot c mod 6), released after the last P V that
// reads them.
// Warp roles: 0-7 softmax + output epilogue (warps w and w+4 share TMEM lane quarter w
// and split the row's columns and O's columns), 8 V loader (one owner for all slots, so
// each slot's fills, and the parity waits on its barrier, happen in order), 9 Q/K window
// loader, 10 S issuer and TMEM owner, 11 P V issuer.
// Persistent CTAs take contiguous ranges of tiles of a group of heads small enough for
// L2, so all rounds of those heads share cached rows.  Every wait is bounded
// (sm100::wait); on a timeout the kernel records where in the workspace status block and
// winds down.
#include <math.h>

#include "sm100.cuh"

namespace lsh {
namespace {

using namespace sm100;

constexpr int kC = 64;            // chunk length
constexpr int kRows = 128;        // rows per tile
constexpr int kWin = 192;         // S columns per tile (window rows)
constexpr int kSlots = 6;         // V ring
constexpr int kSmWarps = 8;       // softmax / epilogue warps
constexpr int kVLoaders = 1;      // V loader warps (12 warps in all: 3 per scheduler keeps 168 registers per thread)
constexpr int kQkWarp = kSmWarps + kVLoaders;
constexpr int kSWarp = kQkWarp + 1;
constexpr int kPvWarp = kSWarp + 1;
constexpr int kThreads = (kPvWarp + 1) * 32;
constexpr int kTmemO = 2 * kWin;  // O accumulator column (384)
constexpr int kLBufs = 4;         // tiles of partial row sums kept in shared memory
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kExactMaxLog2 = 64.f;
constexpr size_t kL2Budget = 48ull << 20;

struct AttnPlan {
    int L, d, nb, n_rounds, causal;
    float scale;
    int nchunks, tps;            // chunks and 128-row tiles per segment
    int n_heads, heads_per_group, n_groups;
};

struct SlotMeta {
    float cs[kC];    // key column scale: scale * log2(e) / |k_j|
    float m2[kC];    // query bound in log2 units: |scale| * log2(e) * |q_i|
    int blo[kC];     // sorted index where the row's bucket starts
    int bhi[kC];     // sorted index where the row's bucket ends
};

struct __align__(8) AttnBarriers {
    uint64_t qk_full[2], qk_empty[2];             // Q/K window buffers (free after S)
    uint64_t v_full[kSlots], v_empty[kSlots];     // V rows + metadata (free after P V)
    uint64_t s_full[2], p_full[2], pv_done[2];
    uint64_t o_full, o_empty, mma_done;
    uint32_t tmem_base;
    int abort_flag;
};

// The tiles of head group `grp` are split into gridDim.x contiguous ranges of global
// units u = seg * tps + tile (seg = bh * n_rounds + r).
__device__ __forceinline__ void group_range(const AttnPlan &P, int grp, long long &lo,
                                            long long &hi) {
    const int h0 = grp * P.heads_per_group;
    const int h1 = min(P.n_heads, h0 + P.heads_per_group);
    const long long per_head = (long long)P.n_rounds * P.tps;
    const long long units = (long long)(h1 - h0) * per_head;
    const long long base = (long long)h0 * per_head;
    lo = base + units * blockIdx.x / gridDim.x;
    hi = base + units * (blockIdx.x + 1) / gridDim.x;
}

// Walk the CTA's items (seg, tiles [tb, te)) in order; f(seg, tb, te).
template <typename F>
__device__ __forceinline__ bool for_items(const AttnPlan &P, F &&f) {
    for (int grp = 0; grp < P.n_groups; ++grp) {
        long long u, hi;
        group_range(P, grp, u, hi);
        while (u < hi) {
            const long long seg = u / P.tps;
            const int tb = (int)(u - seg * P.tps);
            const long long te_ll = tb + (hi - u);
            const int te = te_ll < P.tps ? (int)te_ll : P.tps;
            if (!f(seg, tb, te)) return false;
            u += te - tb;
        }
    }
    return true;
}

__device__ __forceinline__ void gather4(uint32_t dst, const CUtensorMap *map, int x, int r0, int r1,
                                        int r2, int r3, uint32_t bar) {
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];"
                 :: "r"(dst), "l"((uint64_t)map), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(bar)
                 : "memory");
}

// Range checks of a self-checking build (-DLSH_CHECKED): a failed check records `code`
// in the status block and the access is skipped (the index is replaced by 0).
#ifdef LSH_CHECKED
#define LSH_IDX(idx, bound, code)                                                        \
    (((unsigned long long)(idx) < (unsigned long long)(bound))                           \
         ? (idx) : (sm100::report(status, abort_flag, (code)), decltype(idx)(0)))
#else
#define LSH_IDX(idx, bound, code) ((void)(bound), (idx))
#endif

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ void st_global_v8(void *p, const uint32_t *r) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                 :: "l"(p), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
                    "r"(r[6]), "r"(r[7]) : "memory");
}

// TMEM column of the packed P values of keys 16m .. 16m+15 (relative to the S buffer).
__host__ __device__ __forceinline__ int p_col(int m) { return 32 * (m >> 1) + 8 * (m & 1); }

// Softmax of one 32-key batch: key jj is a candidate iff jj + off lies in [0, len) (and,
// not causal, jj != skip); candidates get p = 2^(s cs - m2), the rest 0 -- except column
// one_at, which gets weight 1 (the self fallback).  Returns the sum of the p.
template <bool kSelfCol>
__device__ __forceinline__ float softmax_batch(const uint32_t (&s32)[32], const float *cs, int off,
                                               unsigned len, int skip, int one_at, float m2,
                                               uint32_t (&pk)[16]) {
    float l = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        float p2[2];
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
            const int jj = 2 * k + e2;
            bool ok = (unsigned)(jj + off) < len;
            if (kSelfCol) ok = ok && jj != skip;
            const float x = fmaf(__uint_as_float(s32[jj]), cs[jj], -m2);
            float p = ok ? ex2(x) : 0.f;
            if (kSelfCol) p = jj == one_at ? 1.f : p;
            p2[e2] = p;
        }
        pk[k] = pack_bf16(p2[0], p2[1]);
        l += p2[0] + p2[1];
    }
    return l;
}

__global__ void __launch_bounds__(kThreads, 1)
lsh_attn_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap vmap,
                   const AttnPlan P, const int32_t *__restrict__ buckets,
                   const int32_t *__restrict__ perm, const int32_t *__restrict__ bstart,
                   const float *__restrict__ inv_norm, __nv_bfloat16 *__restrict__ o_r,
                   float *__restrict__ lse_r, StatusBlock *status)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ AttnBarriers sb;
    __shared__ float l_part[kLBufs][2][kRows];   // partial row sums of the two column halves
    // 1024-byte aligned base, derived from the shared array by pointer arithmetic so the
    // compiler keeps the shared state space (shared loads, not generic ones)
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int nkb = P.d / 64;                      // 64-column blocks of a row
    const int wkb = kWin * 128;                    // Q/K window: [w][kb][192 rows][128 B]
    const int wstride = nkb * wkb;
    const int vslot = nkb * kC * 128;              // V ring: [slot][kb][64 rows][128 B]
    uint8_t *QKW = smem;
    uint8_t *V = QKW + 2 * wstride;
    SlotMeta *meta = (SlotMeta *)(V + kSlots * vslot);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int *abort_flag = &sb.abort_flag;
    const uint32_t FULL = 0xffffffffu;
    uint32_t armed = 0, armed_par = 0;   // loaders: last fill per slot / window (wind-down)

    if (threadIdx.x == 0) {
        for (int w = 0; w < 2; ++w) {
            mbar_init(&sb.qk_full[w], 1);           // expect_tx arrive
            mbar_init(&sb.qk_empty[w], 1);
        }
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(&sb.v_full[s], 1 + 32);       // expect_tx arrive + 32 metadata lanes
            mbar_init(&sb.v_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sb.s_full[b], 1);
            mbar_init(&sb.p_full[b], 32 * kSmWarps);
            mbar_init(&sb.pv_done[b], 1);
        }
        mbar_init(&sb.o_full, 1);
        mbar_init(&sb.o_empty, 32 * kSmWarps);
        mbar_init(&sb.mma_done, 2);
        sb.abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == kSWarp) tmem_alloc(&sb.tmem_base, 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = sb.tmem_base;
    const size_t n_rows = (size_t)P.n_heads * P.n_rounds * P.L;
    const long long n_tok = (long long)P.n_heads * P.L;

    if (warp >= kSmWarps && warp < kSmWarps + kVLoaders) {
        // ------------------------------------------------------------- V loaders
        const int lw = warp - kSmWarps;
        if (lane == 0) prefetch_tmap(&vmap);
        uint32_t v_bits = (1u << kSlots) - 1;        // parity to wait per slot
        const float ascale = fabsf(P.scale) * kLog2e, cscale = P.scale * kLog2e;
        for_items(P, [&](long long seg, int tb, int te) -> bool {
            const long long bh = seg / P.n_rounds;
            const int c_begin = tb > 0 ? 2 * tb - 1 : 0;
            const int c_end = min(2 * te, P.nchunks);
            for (int c = c_begin; c < c_end; ++c) {
                const int s = c % kSlots;
                if (s % kVLoaders != lw) continue;
                const uint32_t pv = (v_bits >> s) & 1u;
                v_bits ^= 1u << s;
                // metadata first (it does not need the slot): rows lane and lane + 32
                const size_t row0 = (size_t)seg * P.L + (size_t)c * kC;
                const int j0 = perm[LSH_IDX(row0 + lane, n_rows, 0x511)];
                const int j1 = perm[LSH_IDX(row0 + 32 + lane, n_rows, 0x512)];
                int g[4];   // rows 4*lane .. 4*lane+3 of the chunk (lanes 0-15 gather)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int row = (4 * lane + k) & 63;
                    const int a = __shfl_sync(FULL, j0, row & 31);
                    const int b = __shfl_sync(FULL, j1, row & 31);
                    g[k] = (int)(bh * P.L) + (row < 32 ? a : b);
                }
                const int b0 = buckets[LSH_IDX((size_t)seg * P.L + j0, n_rows, 0x513)];
                const int b1 = buckets[LSH_IDX((size_t)seg * P.L + j1, n_rows, 0x514)];
                const float n0 = inv_norm[LSH_IDX(bh * P.L + j0, n_tok, 0x515)];
                const float n1 = inv_norm[LSH_IDX(bh * P.L + j1, n_tok, 0x516)];
                const size_t bs0 = (size_t)seg * (P.nb + 1);
                const size_t n_bs = (size_t)P.n_heads * P.n_rounds * (P.nb + 1);
                const int lo0 = bstart[LSH_IDX(bs0 + b0, n_bs, 0x517)];
                const int hi0 = bstart[LSH_IDX(bs0 + b0 + 1, n_bs, 0x518)];
                const int lo1 = bstart[LSH_IDX(bs0 + b1, n_bs, 0x519)];
                const int hi1 = bstart[LSH_IDX(bs0 + b1 + 1, n_bs, 0x51a)];
                bool ok = wait(&sb.v_empty[s], pv, abort_flag, status, 0x503);
                if (!__all_sync(FULL, ok)) return false;
                if (lane == 0) mbar_expect_tx(&sb.v_full[s], (uint32_t)(kC * P.d * 2));
                __syncwarp();
                if (lane < 16)
                    for (int kb = 0; kb < nkb; ++kb)
                        gather4(smem_u32(V + s * vslot + kb * kC * 128 + 4 * lane * 128), &vmap,
                                kb * 64, g[0], g[1], g[2], g[3], smem_u32(&sb.v_full[s]));
                SlotMeta &m = meta[s];
                m.cs[lane] = cscale * n0;
                m.cs[lane + 32] = cscale * n1;
                m.m2[lane] = n0 > 0.f ? ascale / n0 : 0.f;
                m.m2[lane + 32] = n1 > 0.f ? ascale / n1 : 0.f;
                m.blo[lane] = lo0;
                m.blo[lane + 32] = lo1;
                m.bhi[lane] = hi0;
                m.bhi[lane + 32] = hi1;
                mbar_arrive(&sb.v_full[s]);
                armed |= 1u << s;
                armed_par = (armed_par & ~(1u << s)) | (pv << s);
            }
            return true;
        });
    } else if (warp == kQkWarp) {
        // ------------------------------------------------------------- Q/K window loader
        if (lane == 0) prefetch_tmap(&qmap);
        int ctr = 0;
        for_items(P, [&](long long seg, int tb, int te) -> bool {
            const long long bh = seg / P.n_rounds;
            for (int t = tb; t < te; ++t, ++ctr) {
                const int w = ctr & 1;
                const bool has_lb = t > 0, has_hi = 2 * t + 1 < P.nchunks;
                int j[3][2];
#pragma unroll
                for (int ci = 0; ci < 3; ++ci) {
                    const int c = 2 * t - 1 + ci;
                    const bool present = ci == 1 || (ci == 0 ? has_lb : has_hi);
                    const size_t row0 = (size_t)seg * P.L + (size_t)(present ? c : 0) * kC;
                    j[ci][0] = present ? perm[LSH_IDX(row0 + lane, n_rows, 0x521)] : 0;
                    j[ci][1] = present ? perm[LSH_IDX(row0 + 32 + lane, n_rows, 0x522)] : 0;
                }
                const uint32_t par = ((ctr >> 1) & 1) ^ 1;
                bool ok = wait(&sb.qk_empty[w], par, abort_flag, status, 0x501);
                if (!__all_sync(FULL, ok)) return false;
                const int n_present = 1 + (has_lb ? 1 : 0) + (has_hi ? 1 : 0);
                if (lane == 0) mbar_expect_tx(&sb.qk_full[w], (uint32_t)(n_present * kC * P.d * 2));
                __syncwarp();
#pragma unroll
                for (int ci = 0; ci < 3; ++ci) {
                    const bool present = ci == 1 || (ci == 0 ? has_lb : has_hi);
                    if (!present) continue;
                    int g[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int row = (4 * lane + k) & 63;
                        const int a = __shfl_sync(FULL, j[ci][0], row & 31);
                        const int b = __shfl_sync(FULL, j[ci][1], row & 31);
                        g[k] = (int)(bh * P.L) + (row < 32 ? a : b);
                    }
                    if (lane < 16)
                        for (int kb = 0; kb < nkb; ++kb)
                            gather4(smem_u32(QKW + w * wstride + kb * wkb + (ci * kC + 4 * lane) * 128),
                                    &qmap, kb * 64, g[0], g[1], g[2], g[3], smem_u32(&sb.qk_full[w]));
                }
                armed |= 1u << w;
                armed_par = (armed_par & ~(1u << w)) | (par << w);
            }
            return true;
        });
    } else if (warp == kSWarp) {
        // ------------------------------------------------------------- S issuer
        {
            const uint32_t qk_base = smem_u32(QKW);
            const uint32_t idesc = idesc_bf16(kRows, kWin, 0, 0);
            int ctr = 0;
            for_items(P, [&](long long, int tb, int te) -> bool {
                for (int t = tb; t < te; ++t, ++ctr) {
                    const int w = ctr & 1, b = ctr & 1;
                    if (!wait_w(&sb.qk_full[w], (ctr >> 1) & 1, abort_flag, status, 0x601)) return false;
                    if (ctr >= 2 && !wait_w(&sb.pv_done[b], ((ctr - 2) >> 1) & 1, abort_flag, status, 0x604))
                        return false;
                    fence_after_sync();
                    for (int ks = 0; ks < P.d / 16; ++ks) {
                        const int kb = ks >> 2, ko = (ks & 3) * 32;
                        const uint32_t wb = qk_base + w * wstride + kb * wkb + ko;
                        mma_ss(tmem + b * kWin, smem_desc(wb + kC * 128, 16, 1024),
                               smem_desc(wb, 16, 1024), idesc, ks > 0);
                    }
                    mma_commit(smem_u32(&sb.s_full[b]));
                    mma_commit(smem_u32(&sb.qk_empty[w]));
                }
                return true;
            });
            mma_commit(smem_u32(&sb.mma_done));
            int dummy = 0;
            wait_w(&sb.mma_done, 0, &dummy, status, 0x605);
        }
    } else if (warp == kPvWarp) {
        // ------------------------------------------------------------- P V issuer
        {
            const uint32_t v_base = smem_u32(V);
            const uint32_t idesc = idesc_bf16(kRows, P.d, 0, 1);
            uint32_t v_bits = 0;
            int ctr = 0;
            auto needv = [&](int c) -> bool {
                const int s = c % kSlots;
                const bool ok = wait_w(&sb.v_full[s], (v_bits >> s) & 1u, abort_flag, status, 0x606);
                v_bits ^= 1u << s;
                return ok;
            };
            for_items(P, [&](long long, int tb, int te) -> bool {
                for (int t = tb; t < te; ++t, ++ctr) {
                    const int q = ctr, b = q & 1;
                    if (t == tb && tb > 0 && !needv(2 * t - 1)) return false;
                    if (!needv(2 * t)) return false;
                    if (2 * t + 1 < P.nchunks && !needv(2 * t + 1)) return false;
                    if (!wait_w(&sb.p_full[b], (q >> 1) & 1, abort_flag, status, 0x602)) return false;
                    if (!wait_w(&sb.o_empty, (q & 1) ^ 1, abort_flag, status, 0x603)) return false;
                    fence_after_sync();
                    uint32_t acc = 0;
                    for (int wc = 0; wc < 3; ++wc) {
                        const int kc = 2 * t - 1 + wc;
                        if (kc < 0 || kc >= P.nchunks) continue;
                        const int s = kc % kSlots;
                        for (int m4 = 0; m4 < 4; ++m4) {
                            const uint64_t bd = smem_desc(v_base + s * vslot + m4 * 2048, kC * 128, 1024);
                            mma_ts(tmem + kTmemO, tmem + b * kWin + p_col(4 * wc + m4), bd, idesc, acc);
                            acc = 1;
                        }
                    }
                    mma_commit(smem_u32(&sb.o_full));
                    mma_commit(smem_u32(&sb.pv_done[b]));
                    // release the V rows whose last use was this tile
                    if (t > 0) mma_commit(smem_u32(&sb.v_empty[(2 * t - 1) % kSlots]));
                    mma_commit(smem_u32(&sb.v_empty[(2 * t) % kSlots]));
                    if (t == te - 1 && 2 * t + 1 < P.nchunks)
                        mma_commit(smem_u32(&sb.v_empty[(2 * t + 1) % kSlots]));
                }
                return true;
            });
            mma_commit(smem_u32(&sb.mma_done));
            int dummy = 0;
            wait_w(&sb.mma_done, 0, &dummy, status, 0x607);
        }
    } else if (warp < kSmWarps) {
        // ------------------------------------------------------------- softmax + epilogue
        const int q4 = warp & 3;                   // TMEM lane quarter
        const int half = warp >> 2;                // which half of the row's columns
        const int i = q4 * 32 + lane;              // tile row = TMEM lane
        const int hi_half = i >= kC;               // row of chunk 2t+1
        const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);
        const int colA = (hi_half ? kC : 0) + 64 * half;   // this warp's 64 S columns
        // the third of the window outside the row's reach, zeroed by one of the halves
        const int colZ = (hi_half ? 0 : 2 * kC) + 32 * half;
        const int self_c0 = kC + 32 * q4;          // batch holding the rows' own columns
        const int dh = P.d / 2;                    // O columns of this warp
        uint32_t full_bits = 0;
        int ctr = 0;
        // epilogue state of the previous tile
        long long e_row = -1;
        float e_m2 = 0.f;
        bool e_live = false, e_self = false;
        bool ok = true;
        const uint32_t zero16[16] = {0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0};

        auto epilogue = [&](int q) -> bool {
            bool w = wait(&sb.o_full, q & 1, abort_flag, status, 0x702);
            // p_full of tile q (complete by now) orders the partner warp's partial sum
            w = w && wait(&sb.p_full[q & 1], (q >> 1) & 1, abort_flag, status, 0x704);
            if (!__all_sync(FULL, w)) return false;
            fence_after_sync();
            LSH_SPAN_BEGIN(t_ep);
            const float l = l_part[q % kLBufs][0][i] + l_part[q % kLBufs][1][i];
            const float inv_l = l > 0.f ? 1.f / l : 0.f;
            __nv_bfloat16 *dst = o_r + LSH_IDX(e_row, (long long)n_rows, 0x712) * P.d + half * dh;
            for (int c = 0; c < dh; c += 32) {
                uint32_t o[32];
                tmem_ld32(tl + kTmemO + half * dh + c, o);
                tmem_wait_ld(o);
                if (e_live) {
                    uint32_t pk[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        pk[k] = pack_bf16(__uint_as_float(o[2 * k]) * inv_l,
                                          __uint_as_float(o[2 * k + 1]) * inv_l);
                    st_global_v8(dst + c, pk);
                    st_global_v8(dst + c + 16, pk + 8);
                }
            }
            if (e_live && half == 0)
                lse_r[LSH_IDX(e_row, (long long)n_rows, 0x713)] =
                    e_self ? kSelfLogit : (e_m2 + __log2f(l)) * kLn2;
            LSH_SPAN_END(t_ep, 0x783);
            fence_before_sync();
            mbar_arrive(&sb.o_empty);
            return true;
        };

        ok = for_items(P, [&](long long seg, int tb, int te) -> bool {
            for (int t = tb; t < te; ++t) {
                auto need = [&](int c) -> bool {
                    const int s = c % kSlots;
                    bool w = wait(&sb.v_full[s], (full_bits >> s) & 1u, abort_flag, status, 0x701);
                    full_bits ^= 1u << s;
                    return __all_sync(FULL, w);
                };
                if (t == tb && tb > 0 && !need(2 * t - 1)) return false;
                if (!need(2 * t)) return false;
                if (2 * t + 1 < P.nchunks && !need(2 * t + 1)) return false;
                const int b = ctr & 1;
                bool w = wait(&sb.s_full[b], (ctr >> 1) & 1, abort_flag, status, 0x703);
                if (!__all_sync(FULL, w)) return false;
                fence_after_sync();

                // this row: its keys are the sorted indices [klo, khi) (minus itself when
                // not causal); the window of a row of chunk cq is chunks cq-1 and cq
                const int cq = 2 * t + hi_half;
                const int srow = t * kRows + i;
                const bool live = cq < P.nchunks;
                const SlotMeta &mq = meta[cq % kSlots];
                const int r = i & (kC - 1);
                int klo = 0, khi = 0;
                float m2 = 0.f;
                if (live) {
                    const int wlo = cq > 0 ? (cq - 1) * kC : 0;
                    klo = max(wlo, mq.blo[r]);
                    khi = P.causal ? srow : min((cq + 1) * kC, mq.bhi[r]);
                    m2 = mq.m2[r];
                }
                // keys other than the row itself?
                const bool self_only = live && (P.causal ? klo >= khi : khi - klo <= 1);
                const int tk0 = (2 * t - 1) * kC;          // sorted index of S column 0
                const uint32_t sbase = tl + b * kWin;

                auto batch_needed = [&](int c0) -> bool {
                    const int t0 = tk0 + c0;
                    const bool nb = (live && klo < t0 + 32 && khi > t0 && klo < khi) ||
                                    (self_only && c0 == self_c0);
                    return __any_sync(FULL, nb);
                };

                // optional exact maximum (huge |scale| |q|): both halves must agree on m2,
                // so the warp pair computes it over the row's whole range
                if (__any_sync(FULL, live && m2 > kExactMaxLog2)) {
                    float mx = -INFINITY;
                    const int cfull = hi_half ? kC : 0;
                    for (int c0 = cfull; c0 < cfull + 2 * kC; c0 += 32) {
                        if (!batch_needed(c0)) continue;
                        uint32_t s32[32];
                        tmem_ld32(sbase + c0, s32);
                        tmem_wait_ld(s32);
                        const SlotMeta &mk = meta[(2 * t - 1 + c0 / kC + kSlots) % kSlots];
                        const int rk = c0 & (kC - 1);
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj) {
                            const int tj = tk0 + c0 + jj;
                            const bool okj = tj >= klo && tj < khi && (P.causal || tj != srow);
                            if (okj) mx = fmaxf(mx, __uint_as_float(s32[jj]) * mk.cs[rk + jj]);
                        }
                    }
                    m2 = mx == -INFINITY ? 0.f : mx;
                    // The pass read the partner warp's S columns: both warps of the lane
                    // quarter (which take this branch together: same rows, same bound)
                    // finish reading before either overwrites S with P.
                    named_bar_sync(1 + q4, 64);
                }

                LSH_SPAN_BEGIN(t_sm);
                float l = 0.f;
                const unsigned len = live ? (unsigned)(khi - klo) : 0u;
                // both 32-column batches in flight before one wait
                const bool nb0 = batch_needed(colA), nb1 = batch_needed(colA + 32);
                uint32_t s32[2][32];
                if (nb0) tmem_ld32(sbase + colA, s32[0]);
                if (nb1) tmem_ld32(sbase + colA + 32, s32[1]);
                if (nb0 || nb1) tmem_wait_ld(s32[0], s32[1]);
                LSH_SPAN_END(t_sm, 0x784);
                LSH_SPAN_BEGIN(t_c);
                uint32_t pkk[2][16];
                bool wr[2] = {false, false};
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int cc = colA + 32 * h;
                    if (!(h ? nb1 : nb0)) continue;
                    const SlotMeta &mk = meta[(2 * t - 1 + cc / kC + kSlots) % kSlots];
                    const float *cs = mk.cs + (cc & (kC - 1));
                    const int off = tk0 + cc - klo;        // key jj is valid iff jj + off in [0, len)
                    if (cc == self_c0)   // the rows' own columns are in this batch: self rules
                        l += softmax_batch<true>(s32[h], cs, off, len, P.causal ? -1 : lane,
                                                 self_only ? lane : -1, m2, pkk[h]);
                    else
                        l += softmax_batch<false>(s32[h], cs, off, len, -1, -1, m2, pkk[h]);
                    wr[h] = true;
                }
                LSH_SPAN_END(t_c, 0x785);
                LSH_SPAN_BEGIN(t_st2);
                if (wr[0]) tmem_st16(sbase + colA, pkk[0]); else tmem_st16(sbase + colA, zero16);
                if (wr[1]) tmem_st16(sbase + colA + 32, pkk[1]); else tmem_st16(sbase + colA + 32, zero16);
                LSH_SPAN_END(t_st2, 0x786);
                LSH_SPAN_END(t_sm, 0x781);
                tmem_st16(sbase + colZ, zero16);
                l_part[ctr % kLBufs][half][i] = l;
                tmem_wait_st();
                fence_before_sync();
                mbar_arrive(&sb.p_full[b]);

                if (ctr >= 1 && !epilogue(ctr - 1)) return false;
                e_live = live;
                e_row = seg * P.L + srow;
                e_m2 = m2;
                e_self = self_only;
                ++ctr;
            }
            return true;
        });
        if (ok && ctr >= 1) epilogue(ctr - 1);
    }

    fence_before_sync();
    __syncthreads();
    if (warp == kSWarp) {
        __syncwarp();
        fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
    if (*abort_flag && warp >= kSmWarps && warp <= kQkWarp) {
        // Wind-down after a timeout: the gathers a loader issued last into each of its
        // slots (or windows) may still be in flight (no consumer waited for them); let
        // them land before the CTA exits.  A fill that was consumed and refilled has
        // landed already; its stale phase is skipped by the bounded wait.
        const bool qk = warp == kQkWarp;
        for (int s = 0; s < (qk ? 2 : kSlots); ++s) {
            if (!(armed & (1u << s))) continue;
            int dummy = 0;
            // a fill waited on parity p of the empty barrier; its full phase has parity p ^ 1
            const uint32_t fp = ((armed_par >> s) & 1u) ^ 1u;
            wait(qk ? &sb.qk_full[s] : &sb.v_full[s], fp, &dummy, nullptr, 0x502);
        }
    }
}

bool make_plan(const Problem &p, AttnPlan &P)
{
    P.L = p.L; P.d = p.d; P.nb = p.nb; P.n_rounds = p.n_rounds; P.causal = p.causal;
    P.scale = p.scale;
    P.nchunks = p.L / kC;
    P.tps = (P.nchunks + 1) / 2;
    P.n_heads = p.B * p.H;
    const size_t head_bytes = (size_t)p.L * p.d * 2 * 2;
    size_t hpg = kL2Budget / head_bytes;
    if (hpg < 1) hpg = 1;
    if (hpg > (size_t)P.n_heads) hpg = P.n_heads;
    P.heads_per_group = (int)hpg;
    P.n_groups = (P.n_heads + P.heads_per_group - 1) / P.heads_per_group;
    return true;
}

size_t smem_bytes(const AttnPlan &P)
{
    const int nkb = P.d / 64;
    return 1024 + (size_t)2 * nkb * kWin * 128 + (size_t)kSlots * nkb * kC * 128 +
           (size_t)kSlots * sizeof(SlotMeta);
}

}  // namespace

bool attn_tc_supported(const Problem &p)
{
    return p.dtype == LSH_BF16 && p.chunk == kC && (p.d == 64 || p.d == 128);
}

cudaError_t attn_tc(const Problem &p, const void *qk, const void *v, const int32_t *buckets,
                    const int32_t *perm, const int32_t *bstart, const float *inv_norm, void *o_r,
                    float *lse_r, StatusBlock *status, cudaStream_t st)
{
    AttnPlan P;
    make_plan(p, P);
    CUtensorMap qmap, vmap;
    if (!make_tmap_2d_bf16(&qmap, qk, (uint64_t)p.n_tok(), (uint64_t)p.d, 64, 1) ||
        !make_tmap_2d_bf16(&vmap, v, (uint64_t)p.n_tok(), (uint64_t)p.d, 64, 1))
        return cudaErrorNotSupported;
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const size_t smem = smem_bytes(P);
    cudaError_t e = cudaFuncSetAttribute(lsh_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    lsh_attn_tc_kernel<<<sms, kThreads, smem, st>>>(qmap, vmap, P, buckets, perm, bstart, inv_norm,
                                                    (__nv_bfloat16 *)o_r, lse_r, status);
    return cudaGetLastError();
}

}  // namespace lsh
