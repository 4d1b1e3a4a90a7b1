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
//   S = Q K^T     tcgen05.mma M=128, N=64 (chunk 2t-1) + N=128 (chunks 2t, 2t+1), K=d,
//                 A and B K-major from shared memory, fp32 into TMEM (2 x 192 columns).
//   P             written back over S in TMEM as packed bf16 pairs.
//   O = P V       tcgen05.mma M=128, N=d, K=192 with A read from TMEM and V as an MN-major
//                 shared-memory operand (the same 128-byte-swizzled row layout as Q/K).
// Softmax without a running maximum: with unit keys every score of query i is bounded
// by m_i = |scale| * |q_i| (Cauchy-Schwarz), so p = exp(s - m_i) cannot overflow.  If
// m_i is so large that every p could underflow (|scale| |q_i| log2 e > 64), the warp
// first takes the exact row maximum instead.  lse = m_i + log(sum p).
// Rows are gathered through the sort permutation by TMA tile::gather4 (4 rows per
// instruction, 128-byte swizzle) into a ring of 6 chunk slots; chunk c sits in slot
// c mod 6, which keeps the two query chunks of a tile in adjacent slots.
// Warp roles: 0-3 softmax + output epilogue (one TMEM lane quarter each), 4-9 loaders
// (warp 4+s fills slot s: permutation, buckets and 1/|k| of the rows, then the
// gathers), 10 MMA issuer and TMEM owner.  Persistent CTAs take contiguous ranges of tiles of a
// group of heads small enough for L2, so all rounds of those heads share cached rows.
// Every wait is bounded (sm100::wait); on a timeout the kernel records where in the
// workspace status block and winds down.
#include <math.h>

#include "sm100.cuh"

namespace lsh {
namespace {

using namespace sm100;

constexpr int kC = 64;            // chunk length
constexpr int kRows = 128;        // rows per tile
constexpr int kWin = 192;         // S columns per tile
constexpr int kSlots = 6;         // chunk ring
constexpr int kLoaders = kSlots;  // loader warps: warp 4+s owns slot s
constexpr int kThreads = (4 + kLoaders + 1) * 32;
constexpr int kMmaWarp = 4 + kLoaders;
constexpr int kTmemO = 2 * kWin;  // O accumulator column (384)
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
    int sb[kC];      // bucket of the sorted row
    int j[kC];       // original position of the sorted row
};

struct __align__(8) AttnBarriers {
    uint64_t chunk_full[kSlots], slot_empty[kSlots];
    uint64_t s_full[2], p_full[2], pv_done[2];
    uint64_t o_full, o_empty, mma_done;
    uint32_t tmem_base;
    int abort_flag;
};

// The tiles of head group `grp` are split into ncta contiguous ranges of global units
// u = seg * tps + tile (seg = bh * n_rounds + r).
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
#define LSH_IDX(idx, bound, code) (idx)
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

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

__global__ void __launch_bounds__(kThreads, 1)
lsh_attn_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap vmap,
                   const AttnPlan P, const int32_t *__restrict__ buckets,
                   const int32_t *__restrict__ perm, const float *__restrict__ inv_norm,
                   const __nv_bfloat16 *__restrict__ v, __nv_bfloat16 *__restrict__ o_r,
                   float *__restrict__ lse_r, StatusBlock *status)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ AttnBarriers sb;
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int nkb = P.d / 64;                      // 64-column blocks of a row
    const int kb_stride = kSlots * kC * 128;       // Q/K: [kb][slot][64 rows][128 B]
    const int vslot = nkb * kC * 128;              // V:   [slot][kb][64 rows][128 B]
    uint8_t *QK = smem;
    uint8_t *V = QK + nkb * kb_stride;
    SlotMeta *meta = (SlotMeta *)(V + kSlots * vslot);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int *abort_flag = &sb.abort_flag;
    const uint32_t FULL = 0xffffffffu;
    uint32_t loader_armed = 0, loader_armed_par = 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(&sb.chunk_full[s], 1 + 32);   // expect_tx arrive + 32 metadata lanes
            mbar_init(&sb.slot_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sb.s_full[b], 1);
            mbar_init(&sb.p_full[b], 128);
            mbar_init(&sb.pv_done[b], 1);
        }
        mbar_init(&sb.o_full, 1);
        mbar_init(&sb.o_empty, 128);
        mbar_init(&sb.mma_done, 1);
        sb.abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == kMmaWarp) tmem_alloc(&sb.tmem_base, 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = sb.tmem_base;

    if (warp >= 4 && warp < 4 + kLoaders) {
        // ------------------------------------------------------------- loaders
        const int lw = warp - 4;
        if (lane == 0) { prefetch_tmap(&qmap); prefetch_tmap(&vmap); }
        uint32_t empty_bits = (1u << kSlots) - 1;   // parity to wait per slot
        uint32_t armed = 0;                          // slots this warp filled (wind-down)
        uint32_t armed_par = 0;
        const float ascale = fabsf(P.scale) * kLog2e, cscale = P.scale * kLog2e;
        for_items(P, [&](long long seg, int tb, int te) -> bool {
            const long long bh = seg / P.n_rounds;
            const int c_begin = tb > 0 ? 2 * tb - 1 : 0;
            const int c_end = min(2 * te, P.nchunks);
            for (int c = c_begin; c < c_end; ++c) {
                const int s = c % kSlots;
                // Each slot has one owning warp, so its fills (and the parity waits on its
                // slot_empty barrier) happen strictly in order: a parity wait cannot tell a
                // phase from the one two fills later.
                if (s != lw) continue;
                const uint32_t par = (empty_bits >> s) & 1u;
                empty_bits ^= 1u << s;
                const size_t row0 = (size_t)seg * P.L + (size_t)c * kC;
                const size_t n_rows = (size_t)P.n_heads * P.n_rounds * P.L;
                const int j0 = perm[LSH_IDX(row0 + lane, n_rows, 0x511)];
                const int j1 = perm[LSH_IDX(row0 + 32 + lane, n_rows, 0x512)];
                const int b0 = buckets[LSH_IDX((size_t)seg * P.L + j0, n_rows, 0x513)];
                const int b1 = buckets[LSH_IDX((size_t)seg * P.L + j1, n_rows, 0x514)];
                const long long n_tok = (long long)P.n_heads * P.L;
                const float n0 = inv_norm[LSH_IDX(bh * P.L + j0, n_tok, 0x515)];
                const float n1 = inv_norm[LSH_IDX(bh * P.L + j1, n_tok, 0x516)];
#ifdef LSH_CHECKED
                if ((unsigned)j0 >= (unsigned)P.L || (unsigned)j1 >= (unsigned)P.L) report(status, abort_flag, 0x517);
                if ((unsigned)b0 >= (unsigned)P.nb || (unsigned)b1 >= (unsigned)P.nb) report(status, abort_flag, 0x518);
#endif
                bool ok = wait(&sb.slot_empty[s], par, abort_flag, status, 0x501);
                if (!__all_sync(FULL, ok)) return false;
                if (lane == 0) mbar_expect_tx(&sb.chunk_full[s], (uint32_t)(kC * P.d * 2 * 2));
                __syncwarp();
                // rows 4*lane .. 4*lane+3 of the chunk (lanes 0-15 issue the gathers)
                int g[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int row = (4 * lane + k) & 63;
                    const int a = __shfl_sync(FULL, j0, row & 31);
                    const int b = __shfl_sync(FULL, j1, row & 31);
                    g[k] = (int)(bh * P.L) + (row < 32 ? a : b);
                }
#ifdef LSH_CHECKED
                for (int k = 0; k < 4; ++k)
                    if (lane < 16 && (unsigned)g[k] >= (unsigned)(P.n_heads * P.L)) {
                        report(status, abort_flag, 0x519);
                        g[k] = 0;
                    }
#endif
                if (lane < 16) {
                    const uint32_t bar = smem_u32(&sb.chunk_full[s]);
                    for (int kb = 0; kb < nkb; ++kb) {
                        gather4(smem_u32(QK + kb * kb_stride + s * kC * 128 + 4 * lane * 128), &qmap,
                                kb * 64, g[0], g[1], g[2], g[3], bar);
                        gather4(smem_u32(V + s * vslot + kb * kC * 128 + 4 * lane * 128), &vmap,
                                kb * 64, g[0], g[1], g[2], g[3], bar);
                    }
                }
                SlotMeta &m = meta[s];
                m.cs[lane] = cscale * n0;
                m.cs[lane + 32] = cscale * n1;
                m.m2[lane] = n0 > 0.f ? ascale / n0 : 0.f;
                m.m2[lane + 32] = n1 > 0.f ? ascale / n1 : 0.f;
                m.sb[lane] = b0;
                m.sb[lane + 32] = b1;
                m.j[lane] = j0;
                m.j[lane + 32] = j1;
                mbar_arrive(&sb.chunk_full[s]);
                armed |= 1u << s;
                armed_par = (armed_par & ~(1u << s)) | (par << s);
            }
            return true;
        });
        loader_armed = armed;
        loader_armed_par = armed_par;
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            uint32_t full_bits = 0;
            int ctr = 0;
            int pt = 0, ptb = 0, pte = 0;    // the tile whose P V is still to be issued
            const uint32_t qk_base = smem_u32(QK), v_base = smem_u32(V);
            const uint32_t idesc64 = idesc_bf16(kRows, 64, 0, 0);
            const uint32_t idesc128 = idesc_bf16(kRows, 128, 0, 0);
            const uint32_t idesc_pv = idesc_bf16(kRows, P.d, 0, 1);

            auto need = [&](int c) -> bool {
                const int s = c % kSlots;
                const bool ok = wait(&sb.chunk_full[s], (full_bits >> s) & 1u, abort_flag, status, 0x601);
                full_bits ^= 1u << s;
                return ok;
            };
            auto do_pv = [&](int t, int tb, int te, int q) -> bool {
                const int b = q & 1;
                if (!wait(&sb.p_full[b], (q >> 1) & 1, abort_flag, status, 0x602)) return false;
                if (!wait(&sb.o_empty, (q & 1) ^ 1, abort_flag, status, 0x603)) return false;
                fence_after_sync();
                uint32_t acc = 0;
                for (int w = 0; w < 3; ++w) {
                    const int kc = 2 * t - 1 + w;
                    if (kc < 0 || kc >= P.nchunks) continue;
                    const int s = kc % kSlots;
                    for (int m4 = 0; m4 < 4; ++m4) {
                        const int m = 4 * w + m4;
                        const uint64_t bd = smem_desc(v_base + s * vslot + m4 * 2048, kC * 128, 1024);
                        mma_ts(tmem + kTmemO, tmem + b * kWin + m * 8, bd, idesc_pv, acc);
                        acc = 1;
                    }
                }
                mma_commit(smem_u32(&sb.o_full));
                mma_commit(smem_u32(&sb.pv_done[b]));
                // release the chunks whose last use was this tile
                if (t > 0) mma_commit(smem_u32(&sb.slot_empty[(2 * t - 1) % kSlots]));
                mma_commit(smem_u32(&sb.slot_empty[(2 * t) % kSlots]));
                if (t == te - 1 && 2 * t + 1 < P.nchunks)
                    mma_commit(smem_u32(&sb.slot_empty[(2 * t + 1) % kSlots]));
                return true;
            };

            bool pending = false;             // P V of tile (pt, ptb, pte) not issued yet
            bool ok = for_items(P, [&](long long seg, int tb, int te) -> bool {
                for (int t = tb; t < te; ++t) {
                    // The first chunks of a new item may reuse slots that the previous item's
                    // last tile releases only after its P V: issue that P V first.
                    if (t == tb && pending) {
                        if (!do_pv(pt, ptb, pte, ctr - 1)) return false;
                        pending = false;
                    }
                    if (t == tb && tb > 0 && !need(2 * t - 1)) return false;
                    if (!need(2 * t)) return false;
                    const bool hi = 2 * t + 1 < P.nchunks;
                    if (hi && !need(2 * t + 1)) return false;
                    const int b = ctr & 1;
                    if (ctr >= 2 && !wait(&sb.pv_done[b], ((ctr - 2) >> 1) & 1, abort_flag, status, 0x604))
                        return false;
                    fence_after_sync();
                    const int sq = (2 * t) % kSlots;
                    const int sl = (2 * t + kSlots - 1) % kSlots;
                    for (int ks = 0; ks < P.d / 16; ++ks) {
                        const int kb = ks >> 2, ko = (ks & 3) * 32;
                        const uint32_t kbase = qk_base + kb * kb_stride + ko;
                        const uint64_t a = smem_desc(kbase + sq * kC * 128, 16, 1024);
                        if (t > 0)
                            mma_ss(tmem + b * kWin, a, smem_desc(kbase + sl * kC * 128, 16, 1024),
                                   idesc64, ks > 0);
                        mma_ss(tmem + b * kWin + 64, a, smem_desc(kbase + sq * kC * 128, 16, 1024),
                               hi ? idesc128 : idesc64, ks > 0);
                    }
                    mma_commit(smem_u32(&sb.s_full[b]));
                    if (pending && !do_pv(pt, ptb, pte, ctr - 1)) return false;
                    pt = t; ptb = tb; pte = te;
                    pending = true;
                    ++ctr;
                }
                return true;
            });
            if (ok && pending) do_pv(pt, ptb, pte, ctr - 1);
            mma_commit(smem_u32(&sb.mma_done));
            int dummy = 0;
            wait(&sb.mma_done, 0, &dummy, status, 0x605);
        }
    } else if (warp < 4) {
        // ------------------------------------------------------------- softmax + epilogue
        const int i = warp * 32 + lane;            // tile row = TMEM lane
        const int hi_half = i >= kC;               // row of chunk 2t+1
        const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
        const int col0 = hi_half ? kC : 0;         // first S column this row may use
        uint32_t full_bits = 0;
        int ctr = 0;
        // epilogue state of the previous tile
        long long e_row = -1, e_vrow = 0;
        float e_l = 0.f, e_lse = 0.f;
        bool e_live = false;
        bool ok = true;

        auto epilogue = [&](int q) -> bool {
            bool w = wait(&sb.o_full, q & 1, abort_flag, status, 0x702);
            if (!__all_sync(FULL, w)) return false;
            fence_after_sync();
            const float inv_l = e_l > 0.f ? 1.f / e_l : 0.f;
            for (int c = 0; c < P.d; c += 32) {
                uint32_t o[32];
                tmem_ld32(tl + kTmemO + c, o);
                tmem_wait_ld();
                if (e_live) {
                    uint32_t pk[16];
                    if (e_l > 0.f) {
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            pk[k] = pack_bf16(__uint_as_float(o[2 * k]) * inv_l,
                                              __uint_as_float(o[2 * k + 1]) * inv_l);
                    } else {
                        const uint4 *src = reinterpret_cast<const uint4 *>(
                            v + LSH_IDX(e_vrow, (long long)P.n_heads * P.L, 0x711) * P.d + c);
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint4 x = src[k];
                            pk[4 * k] = x.x; pk[4 * k + 1] = x.y; pk[4 * k + 2] = x.z; pk[4 * k + 3] = x.w;
                        }
                    }
                    uint4 *dst = reinterpret_cast<uint4 *>(
                        o_r + LSH_IDX(e_row, (long long)P.n_heads * P.n_rounds * P.L, 0x712) * P.d + c);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        dst[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
                }
            }
            if (e_live) lse_r[LSH_IDX(e_row, (long long)P.n_heads * P.n_rounds * P.L, 0x713)] = e_lse;
            fence_before_sync();
            mbar_arrive(&sb.o_empty);
            return true;
        };

        ok = for_items(P, [&](long long seg, int tb, int te) -> bool {
            const long long bh = seg / P.n_rounds;
            for (int t = tb; t < te; ++t) {
                auto need = [&](int c) -> bool {
                    const int s = c % kSlots;
                    bool w = wait(&sb.chunk_full[s], (full_bits >> s) & 1u, abort_flag, status, 0x701);
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

                // this row
                const int cq = 2 * t + hi_half;                 // its chunk
                const long long srow = (long long)t * kRows + i;  // sorted index
                const bool live = cq < P.nchunks;
                const SlotMeta &mq = meta[cq % kSlots];
                const int r = i & (kC - 1);
                const int bq = live ? mq.sb[r] : -1;
                const int jq = live ? mq.j[r] : 0;
                float m2 = live ? mq.m2[r] : 0.f;
                const long long tk0 = (long long)(2 * t - 1) * kC;  // sorted index of column 0
                const uint32_t sbase = tl + b * kWin;

                // per 32-column batch: does any row of the warp have a candidate in it?
                auto batch_needed = [&](int c0) -> bool {
                    const long long t0 = tk0 + c0;
                    const int kc = 2 * t - 1 + c0 / kC;
                    bool need_b = false;
                    if (live && kc >= 0 && kc < P.nchunks) {
                        const SlotMeta &mk = meta[kc % kSlots];
                        const int rk = c0 & (kC - 1);
                        need_b = mk.sb[rk] <= bq && bq <= mk.sb[rk + 31] &&
                                 (!P.causal || t0 < srow);
                    }
                    return __any_sync(FULL, need_b);
                };

                // optional exact maximum (huge |scale| |q|)
                if (__any_sync(FULL, live && m2 > kExactMaxLog2)) {
                    float mx = -INFINITY;
                    for (int c0 = col0; c0 < col0 + 2 * kC; c0 += 32) {
                        if (!batch_needed(c0)) continue;
                        uint32_t s32[32];
                        tmem_ld32(sbase + c0, s32);
                        tmem_wait_ld();
                        const SlotMeta &mk = meta[(2 * t - 1 + c0 / kC + kSlots) % kSlots];
                        const int rk = c0 & (kC - 1);
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj) {
                            const long long tj = tk0 + c0 + jj;
                            const bool ok_j = mk.sb[rk + jj] == bq &&
                                              (P.causal ? tj < srow : tj != srow);
                            if (ok_j) mx = fmaxf(mx, __uint_as_float(s32[jj]) * mk.cs[rk + jj]);
                        }
                    }
                    m2 = mx == -INFINITY ? 0.f : mx;
                }

                float l = 0.f;
                const uint32_t zero16[16] = {0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0};
                if (hi_half) tmem_st16(sbase + 0, zero16), tmem_st16(sbase + 16, zero16);
                for (int c0 = col0; c0 < col0 + 2 * kC; c0 += 32) {
                    if (!batch_needed(c0)) {
                        tmem_st16(sbase + c0 / 2, zero16);
                        continue;
                    }
                    uint32_t s32[32];
                    tmem_ld32(sbase + c0, s32);
                    tmem_wait_ld();
                    const SlotMeta &mk = meta[(2 * t - 1 + c0 / kC + kSlots) % kSlots];
                    const int rk = c0 & (kC - 1);
                    const long long tbase = tk0 + c0;
                    uint32_t pk[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        float p2[2];
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int jj = 2 * k + h;
                            const long long tj = tbase + jj;
                            const bool ok_j = live && mk.sb[rk + jj] == bq &&
                                              (P.causal ? tj < srow : tj != srow);
                            const float x = fmaf(__uint_as_float(s32[jj]), mk.cs[rk + jj], -m2);
                            p2[h] = ok_j ? ex2(x) : 0.f;
                        }
                        pk[k] = pack_bf16(p2[0], p2[1]);
                        l += bf16_lo(pk[k]) + bf16_hi(pk[k]);
                    }
                    tmem_st16(sbase + c0 / 2, pk);
                }
                if (!hi_half) tmem_st16(sbase + 64, zero16), tmem_st16(sbase + 80, zero16);
                tmem_wait_st();
                fence_before_sync();
                mbar_arrive(&sb.p_full[b]);

                if (ctr >= 1 && !epilogue(ctr - 1)) return false;
                e_live = live;
                e_row = (long long)seg * P.L + srow;
                e_vrow = bh * P.L + jq;
                e_l = l;
                e_lse = l > 0.f ? (m2 + __log2f(l)) * kLn2 : kSelfLogit;
                ++ctr;
            }
            return true;
        });
        if (ok && ctr >= 1) epilogue(ctr - 1);
    }

    fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
    if (*abort_flag && warp >= 4 && warp < 4 + kLoaders) {
        // Wind-down after a timeout: the gathers this warp issued last into each slot may
        // still be in flight (no consumer waited for them); let them land before the CTA
        // exits.  A fill that was consumed and refilled has landed already; its stale
        // phase is skipped by the bounded wait.
        for (int s = 0; s < kSlots; ++s) {
            if (!(loader_armed & (1u << s))) continue;
            int dummy = 0;
            const uint32_t fp = ((loader_armed_par >> s) & 1u) ^ 1u;  // chunk_full parity of that fill
            wait(&sb.chunk_full[s], fp, &dummy, nullptr, 0x502);
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
    return 1024 + (size_t)nkb * kSlots * kC * 128 * 2 + (size_t)kSlots * sizeof(SlotMeta);
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
    (void)bstart;
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
    lsh_attn_tc_kernel<<<sms, kThreads, smem, st>>>(qmap, vmap, P, buckets, perm, inv_norm,
                                                    (const __nv_bfloat16 *)v, (__nv_bfloat16 *)o_r,
                                                    lse_r, status);
    return cudaGetLastError();
}

}  // namespace lsh
