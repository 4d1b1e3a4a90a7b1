// attn_tc.cu -- chunked look-one-back LSH attention on the tcgen05 tensor cores (bf16 or
// fp16 inputs, fp32 accumulation, chunk 64 or 32, d = 64 or 128).  Chunk 32 runs on the
// same 64-row chunks with each row's keys clipped to its own 32-row chunk and the one
// before (a sub-window of its 64-row window), so L must then be a multiple of 64.
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
//   S = Q K^T     tcgen05.mma M=128, K=16 steps over d; A = the tile's 128 rows, B = the
//                 window's 192 rows, both from the chunk ring in shared memory, fp32 into
//                 TMEM (2 x 192 columns).  One N=192 chain when the three chunks sit in
//                 consecutive ring slots, else N=64 (look-back) + N=128.
//   P             packed bf16 pairs written into TMEM over S: the 32 keys of S columns
//                 32j..32j+31 go to columns 32j..32j+15, so every warp overwrites only
//                 S columns it has already read.
//   O = P V       tcgen05.mma M=128, N=d, K=16 steps with A read from TMEM and V as an
//                 MN-major shared-memory operand (the same 128-byte-swizzled row layout
//                 as Q/K).
// The S chain and the P V chain are issued from two different warps and overlap.
// Masks: sorted order keeps each bucket in one run, so the keys of sorted row s form one
// interval of window columns: [max(window start, bucket start), causal ? s : min(window
// end, bucket end)), minus s itself when not causal.  The metadata warp marks where runs
// start and end inside each chunk (warp ballots over neighbouring rows' buckets); a
// softmax lane turns the marks of its chunk and the previous one into its interval, so
// neither needs the bucket-start table or a per-key bucket test.  A row with no key but itself
// gives its own column weight 1, so P V returns v_i exactly; its lse is the self logit
// -1e5.
// Softmax without a running maximum: with unit keys every score of query i is bounded
// by m_i = |scale| * |q_i| (Cauchy-Schwarz), so p = exp(s - m_i) cannot overflow.  Every
// score is also at least -m_i, so in log2 units p >= 2^(-2 m2) with m2 = m_i log2 e.
// While m2 <= 32 that is >= 2^-64: far inside the normal range of fp32 and bf16 (ex2's
// flush-to-zero starts below 2^-126), so no row can end with a zero sum.  Above that the
// warp first takes the exact row maximum instead.  lse = m_i + log(sum p).  With fp16
// inputs P is packed to fp16 for P V, whose smallest normal number is 2^-14, so there
// the exact maximum takes over above m2 = 7.
// Data movement: a ring of 6 chunk slots (chunk c in slot c mod 6) holds each chunk's
// Q/K rows, V rows and row metadata, loaded once and released after the last P V that
// reads the chunk.  Rows are gathered through the sort permutation by 16-byte cp.async
// pieces written straight into the 128-byte-swizzled operand layout (row r's piece c at
// r * 128 + ((c ^ (r & 7)) * 16)).  (A tensor-map gather moves only 512 bytes per
// operation here, about 7 bytes per clock per SM, and its issue stalls the issuing warp;
// one warp's cp.async stream manages about 5-10.)  So every chunk is filled by several
// loader warps at once.  The MMA warps fence the async proxy after each wait, since the
// rows were written through the generic one.
// Warp roles (28 warps, 72 registers each): 0-15 softmax + output epilogue (warps w, w+4,
// w+8 and w+12 share TMEM lane quarter w and split the row's columns and O's columns four
// ways), 16 the metadata warp, 17-25 row copiers, 26 S issuer and TMEM owner, 27 P V issuer.
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
constexpr int kSlots = 6;         // chunk ring (even: chunk parity = slot parity)
constexpr int kSmWarps = 16;      // softmax / epilogue warps (4 per TMEM lane quarter)
constexpr int kLoaders = 10;      // loader warps: 1 metadata warp + kCopyWarps row copiers
constexpr int kCopyWarps = kLoaders - 1;
constexpr int kSWarp = kSmWarps + kLoaders;
constexpr int kPvWarp = kSWarp + 1;
constexpr int kThreads = (kPvWarp + 1) * 32;
constexpr int kTmemO = 2 * kWin;  // O accumulator column (384)
constexpr int kLBufs = 4;         // tiles of partial row sums kept in shared memory
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kExactMaxLog2 = 32.f;   // bound path keeps every p >= 2^-64
// fp16 P: the bound path keeps every p >= 2^-14, fp16's smallest normal number (its
// subnormals carry too few bits: a weight near 2^-20 would keep four)
constexpr float kExactMaxLog2F16 = 7.f;
constexpr size_t kL2Budget = 48ull << 20;

struct AttnPlan {
    int L, d, nb, n_rounds, causal, token_order;
    float scale;
    int nchunks, tps;            // 64-row chunks and 128-row tiles per segment
    int window;                  // the attention chunk: 64, or 32 (a sub-window, see below)
    int n_heads, heads_per_group, n_groups;
};

struct __align__(16) SlotMeta {
    float cs[kC];    // key column scale: scale * log2(e) / |k_j|
    float m2[kC];    // query bound in log2 units: |scale| * log2(e) * |q_i|
    unsigned long long starts;   // bit r: a bucket run starts at row r (bit 0 also when
                                 // the chunk opens its segment)
    unsigned long long ends;     // bit r: a run ends at row r (row 63 never marked)
    int jrow[kC];                // original position of each row
};

struct __align__(8) AttnBarriers {
    uint64_t full[kSlots], empty[kSlots];         // chunk slots (free after the last P V)
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

// Range checks of a self-checking build (-DLSH_CHECKED): a failed check records `code`
// in the status block and the access is skipped (the index is replaced by 0).
#ifdef LSH_CHECKED
#define LSH_IDX(idx, bound, code)                                                        \
    (((unsigned long long)(idx) < (unsigned long long)(bound))                           \
         ? (idx) : (sm100::report(status, abort_flag, (code)), decltype(idx)(0)))
#else
#define LSH_IDX(idx, bound, code) ((void)(bound), (idx))
#endif

// A permuted row index as a safe row: out of [0, L) (a corrupt permutation) it is
// reported in a self-checking build and replaced by 0 in every build, so no copy ever
// leaves the tensor.
#ifdef LSH_CHECKED
#define LSH_ROW(j, L, code) LSH_IDX(j, L, code)
#else
#define LSH_ROW(j, L, code) ((unsigned)(j) < (unsigned)(L) ? (j) : 0)
#endif

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ void st_global_v8(void *p, const uint32_t *r) {
    // streaming store (.cs): the per-round outputs are read back once by the round
    // combination much later, so they should not evict the gathered Q/K/V rows from L2
    asm volatile("st.global.cs.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                 :: "l"(p), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
                    "r"(r[6]), "r"(r[7]) : "memory");
}

// TMEM column of the packed P values of keys 16m .. 16m+15 (relative to the S buffer).
__host__ __device__ __forceinline__ int p_col(int m) { return 32 * (m >> 1) + 8 * (m & 1); }

// Bits lo..hi-1 of a 32-bit mask (the batch columns inside a row's key interval).
__device__ __forceinline__ uint32_t range_mask(int lo, int hi) {
    lo = max(lo, 0);
    hi = min(hi, 32);
    if (lo >= hi) return 0u;
    const uint32_t below_hi = hi == 32 ? 0xffffffffu : (1u << hi) - 1u;
    return below_hi & (0xffffffffu << lo);
}

// One 16-column quarter of a row: p_j = 2^(s_j * cs_j - m2) for the columns whose bit
// is set in the low 16 bits of `vm`, 0 elsewhere (ex2 of -inf), packed to bf16 pairs.
// Returns sum_j p_j.  `cs` is 16-byte aligned shared memory.
template <bool F16>
__device__ __forceinline__ float softmax_quarter(const uint32_t (&s16)[16], const float *cs,
                                                 uint32_t vm, float m2, uint32_t (&pk)[8]) {
    float la = 0.f, lb = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float4 c4 = reinterpret_cast<const float4 *>(cs)[q];
        const float c[4] = {c4.x, c4.y, c4.z, c4.w};
        float p[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int jj = 4 * q + e;
            const float x = fmaf(__uint_as_float(s16[jj]), c[e], -m2);
            p[e] = ex2((vm >> jj) & 1u ? x : -INFINITY);
        }
        pk[2 * q] = F16 ? pack_f16(p[0], p[1]) : pack_bf16(p[0], p[1]);
        pk[2 * q + 1] = F16 ? pack_f16(p[2], p[3]) : pack_bf16(p[2], p[3]);
        la += p[0] + p[1];
        lb += p[2] + p[3];
    }
    return la + lb;
}

template <bool F16>
__global__ void __launch_bounds__(kThreads, 1)
lsh_attn_tc_kernel(const __nv_bfloat16 *__restrict__ qk, const __nv_bfloat16 *__restrict__ vv,
                   const AttnPlan P, const int32_t *__restrict__ buckets,
                   const int32_t *__restrict__ perm,
                   const float *__restrict__ inv_norm, __nv_bfloat16 *__restrict__ o_r,
                   float *__restrict__ lse_r, StatusBlock *status)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ AttnBarriers sb;
#ifdef LSH_WAIT_PROF
    __shared__ volatile long long slot_clk[kSlots];   // when a slot's fill was released
#endif
    __shared__ float l_part[kLBufs][4][kRows];   // partial row sums of the four column parts
    // 1024-byte aligned base, derived from the shared array by pointer arithmetic so the
    // compiler keeps the shared state space (shared loads, not generic ones)
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int nkb = P.d / 64;                      // 64-column blocks of a row
    // Q/K rows: [kb][slot][64 rows][128 B] (for one kb the slots are consecutive, so the
    // rows of chunks in consecutive slots form one operand); V rows: [slot][kb][64][128 B]
    const int qk_plane = kSlots * kC * 128;
    const int vslot = nkb * kC * 128;
    uint8_t *QK = smem;
    uint8_t *V = QK + nkb * qk_plane;
    SlotMeta *meta = (SlotMeta *)(V + kSlots * vslot);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int *abort_flag = &sb.abort_flag;
    const uint32_t FULL = 0xffffffffu;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kSlots; ++s) {
            // metadata lanes + copy warps' cp.async lanes
            mbar_init(&sb.full[s], 32 + 32 * kCopyWarps);

            mbar_init(&sb.empty[s], 1);
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

    if (warp >= kSmWarps && warp < kSmWarps + kLoaders) {
        // ------------------------------------------------------------- loaders
        // Every chunk is filled by all loader warps together, so a chunk lands in about a
        // ninth of the time one warp's cp.async stream needs (the ring cannot hold more
        // chunks in flight).  Warp kSmWarps is the metadata warp (row metadata); the copy
        // warps copy the Q/K and V rows.  Every loader waits for the slot itself and
        // takes part in every fill of every slot, in order, so no warp can fall a phase
        // behind on a slot's barriers (a fill completes only with every warp's arrival).
        const int lw = warp - kSmWarps;
        uint32_t e_bits = (1u << kSlots) - 1;        // parity of the next empty wait, per slot
        const float ascale = fabsf(P.scale) * kLog2e, cscale = P.scale * kLog2e;
        for_items(P, [&](long long seg, int tb, int te) -> bool {
            const long long bh = seg / P.n_rounds;
            const int c_begin = tb > 0 ? 2 * tb - 1 : 0;
            const int c_end = min(2 * te, P.nchunks);
            const size_t seg_row0 = (size_t)seg * P.L;
            if (lw > 0) {
                // ---- copy warp k = lw - 1: row groups g = k, k + kCopyWarps, ... of
                // rpi = 32 / (d / 8) rows, from both Q/K and V.  Each lane loads the
                // permutation entry of its own row, one chunk ahead.
                const int k = lw - 1;
                const int lpr = P.d >> 3, rpi = 32 / lpr;
                const int cpiece = lane & (lpr - 1), c16 = cpiece & 7, kb = cpiece >> 3;
                const int rsub = lane / lpr;
                const int n_grp = kC / rpi;
                constexpr int kMine = (kC / 2 + kCopyWarps - 1) / kCopyWarps;  // groups per warp (d = 128)
                int jn[kMine];
                auto ld_j = [&](int cc) {
#pragma unroll
                    for (int q = 0; q < kMine; ++q) {
                        const int g = k + q * kCopyWarps;
                        jn[q] = g < n_grp ? LSH_ROW(perm[LSH_IDX(seg_row0 + (size_t)cc * kC + g * rpi + rsub,
                                                                   n_rows, 0x51c)], P.L, 0x51d)
                                          : 0;
                    }
                };
                if (c_begin < c_end) ld_j(c_begin);
                for (int c = c_begin; c < c_end; ++c) {
                    const int s = c % kSlots;
                    int jc[kMine];
#pragma unroll
                    for (int q = 0; q < kMine; ++q) jc[q] = jn[q];
                    if (c + 1 < c_end) ld_j(c + 1);
                    const bool ok = wait(&sb.empty[s], (e_bits >> s) & 1u, abort_flag, status, 0x504);
                    if (!__all_sync(FULL, ok)) return false;
                    e_bits ^= 1u << s;
                    const uint32_t qdst = smem_u32(QK + s * kC * 128) + kb * qk_plane;
                    const uint32_t vdst = smem_u32(V + s * vslot) + kb * kC * 128;
#pragma unroll
                    for (int q = 0; q < kMine; ++q) {
                        const int g = k + q * kCopyWarps;
                        if (g >= n_grp) break;
                        const int r = g * rpi + rsub;
                        const long long off = (bh * P.L + jc[q]) * P.d + cpiece * 8;
                        const uint32_t sw = r * 128 + ((c16 ^ (r & 7)) << 4);
                        cp_async16(qdst + sw, qk + off);
                        cp_async16(vdst + sw, vv + off);
                    }
                    cp_async_mbar_arrive(&sb.full[s]);
                }
                return true;
            }
            // ---- metadata warp.  Loads are software-pipelined over the chunks: the
            // permutation two chunks ahead, buckets and norms one chunk ahead.  Lane k holds
            // rows k and k + 32; every lane also holds the row before the chunk.
            int c = c_begin;
            if (c >= c_end) return true;
            int ja0 = 0, ja1 = 0, jap = 0, jb0 = 0, jb1 = 0, jbp = 0;
            auto ld_perm = [&](int cc, int &j0, int &j1, int &jp) {
                const size_t row0 = seg_row0 + (size_t)cc * kC;
                j0 = LSH_ROW(perm[LSH_IDX(row0 + lane, n_rows, 0x511)], P.L, 0x517);
                j1 = LSH_ROW(perm[LSH_IDX(row0 + 32 + lane, n_rows, 0x512)], P.L, 0x518);
                jp = cc > 0 ? LSH_ROW(perm[LSH_IDX(row0 - 1, n_rows, 0x519)], P.L, 0x51a) : 0;
            };
            int bk0, bk1, bkp;                           // buckets of the rows
            float nm0, nm1;                              // 1 / |k| of the rows
            auto ld_rows = [&](int j0, int j1, int jp) {
                bk0 = buckets[LSH_IDX(seg_row0 + j0, n_rows, 0x513)];
                bk1 = buckets[LSH_IDX(seg_row0 + j1, n_rows, 0x514)];
                bkp = buckets[LSH_IDX(seg_row0 + jp, n_rows, 0x51b)];
                nm0 = inv_norm[LSH_IDX(bh * P.L + j0, n_tok, 0x515)];
                nm1 = inv_norm[LSH_IDX(bh * P.L + j1, n_tok, 0x516)];
            };
            ld_perm(c, ja0, ja1, jap);
            if (c + 1 < c_end) ld_perm(c + 1, jb0, jb1, jbp);
            ld_rows(ja0, ja1, jap);
            for (; c < c_end; ++c) {
                LSH_SPAN_BEGIN(t_meta);
                const int s = c % kSlots;
                const uint32_t pe = (e_bits >> s) & 1u;
                const int j0 = ja0, j1 = ja1, b0 = bk0, b1 = bk1, bp = bkp;
                const float n0 = nm0, n1 = nm1;
                ja0 = jb0;
                ja1 = jb1;
                jap = jbp;
                if (c + 2 < c_end) ld_perm(c + 2, jb0, jb1, jbp);
                if (c + 1 < c_end) ld_rows(ja0, ja1, jap);
                // where bucket runs start and end inside the chunk
                const int up0 = __shfl_up_sync(FULL, b0, 1), up1 = __shfl_up_sync(FULL, b1, 1);
                const int last0 = __shfl_sync(FULL, b0, 31);
                const int dn0 = __shfl_down_sync(FULL, b0, 1), dn1 = __shfl_down_sync(FULL, b1, 1);
                const int first1 = __shfl_sync(FULL, b1, 0);
                const bool st0 = lane > 0 ? b0 != up0 : (c == 0 || b0 != bp);
                const bool st1 = b1 != (lane > 0 ? up1 : last0);
                const bool en0 = b0 != (lane < 31 ? dn0 : first1);
                const bool en1 = lane < 31 && b1 != dn1;
                const unsigned long long starts = (unsigned long long)__ballot_sync(FULL, st0) |
                                                  ((unsigned long long)__ballot_sync(FULL, st1) << 32);
                const unsigned long long ends = (unsigned long long)__ballot_sync(FULL, en0) |
                                                ((unsigned long long)__ballot_sync(FULL, en1) << 32);
                bool ok = wait(&sb.empty[s], pe, abort_flag, status, 0x503);
                if (!__all_sync(FULL, ok)) return false;
                e_bits ^= 1u << s;   // now the parity of this fill's full phase
                SlotMeta &m = meta[s];
                m.jrow[lane] = j0;
                m.jrow[lane + 32] = j1;
#ifdef LSH_WAIT_PROF
                if (lane == 0) slot_clk[s] = clock64();
#endif
                m.cs[lane] = cscale * n0;
                m.cs[lane + 32] = cscale * n1;
                m.m2[lane] = n0 > 0.f ? ascale / n0 : 0.f;
                m.m2[lane + 32] = n1 > 0.f ? ascale / n1 : 0.f;
                if (lane == 0) {
                    m.starts = starts;
                    m.ends = ends;
                }
                mbar_arrive(&sb.full[s]);
                LSH_SPAN_END(t_meta, 0x5b0);
            }
            return true;
        });
    } else if (warp == kSWarp) {
        // ------------------------------------------------------------- S issuer
        {
            const uint32_t qk_base = smem_u32(QK);
            uint32_t f_bits = 0;
            int ctr = 0;
            auto need = [&](int c) -> bool {
                const int s = c % kSlots;
                const bool ok = wait_w(&sb.full[s], (f_bits >> s) & 1u, abort_flag, status, 0x601);
                f_bits ^= 1u << s;
#ifdef LSH_WAIT_PROF
                if (lane == 0) {   // from the slot's release to the S issuer seeing it full
                    atomicAdd(&g_wait_cycles[0x5b1], (unsigned long long)(clock64() - slot_clk[s]));
                    atomicAdd(&g_wait_count[0x5b1], 1ull);
                }
#endif
                return ok;
            };
            for_items(P, [&](long long, int tb, int te) -> bool {
                for (int t = tb; t < te; ++t, ++ctr) {
                    const int b = ctr & 1;
                    if (t == tb && tb > 0 && !need(2 * t - 1)) return false;
                    if (!need(2 * t)) return false;
                    if (2 * t + 1 < P.nchunks && !need(2 * t + 1)) return false;
                    if (ctr >= 2 && !wait_w(&sb.pv_done[b], ((ctr - 2) >> 1) & 1, abort_flag, status, 0x604))
                        return false;
                    fence_after_sync();
                    // the rows were written by cp.async (generic proxy); the MMA reads them
                    // through the async proxy
                    fence_proxy_async();
                    const int s0 = (2 * t) % kSlots;      // even: chunks 2t, 2t+1 in s0, s0+1
                    // one N=192 chain when the look-back chunk sits in slot s0 - 1; else the
                    // look-back (if any) as an N=64 chain into columns 0-63
                    const bool joined = s0 > 0 && t > 0;
                    for (int ks = 0; ks < P.d / 16; ++ks) {
                        const int kb = ks >> 2, ko = (ks & 3) * 32;
                        const uint32_t pb = qk_base + kb * qk_plane + ko;
                        const uint64_t a = smem_desc(pb + s0 * kC * 128, 16, 1024);
                        if (joined) {
                            mma_ss(tmem + b * kWin, a, smem_desc(pb + (s0 - 1) * kC * 128, 16, 1024),
                                   idesc_16(kRows, kWin, 0, 0, F16), ks > 0);
                        } else {
                            if (t > 0)
                                mma_ss(tmem + b * kWin, a,
                                       smem_desc(pb + (kSlots - 1) * kC * 128, 16, 1024),
                                       idesc_16(kRows, kC, 0, 0, F16), ks > 0);
                            mma_ss(tmem + b * kWin + kC, a, smem_desc(pb + s0 * kC * 128, 16, 1024),
                                   idesc_16(kRows, 2 * kC, 0, 0, F16), ks > 0);
                        }
                    }
                    mma_commit(smem_u32(&sb.s_full[b]));
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
            const uint32_t idesc = idesc_16(kRows, P.d, 0, 1, F16);
            uint32_t v_bits = 0;
            int ctr = 0;
            auto needv = [&](int c) -> bool {
                const int s = c % kSlots;
                const bool ok = wait_w(&sb.full[s], (v_bits >> s) & 1u, abort_flag, status, 0x606);
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
                    fence_proxy_async();   // V rows were written by cp.async
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
                    // release the chunks whose last use was this tile (their S MMAs
                    // completed before this tile's P was written)
                    if (t > 0) mma_commit(smem_u32(&sb.empty[(2 * t - 1) % kSlots]));
                    mma_commit(smem_u32(&sb.empty[(2 * t) % kSlots]));
                    if (t == te - 1 && 2 * t + 1 < P.nchunks)
                        mma_commit(smem_u32(&sb.empty[(2 * t + 1) % kSlots]));
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
        const int part = warp >> 2;                // which quarter of the row's columns
        const int i = q4 * 32 + lane;              // tile row = TMEM lane
        const int hi_half = i >= kC;               // row of chunk 2t+1
        const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);
        const int colA = (hi_half ? kC : 0) + 32 * part;   // this warp's 32 S columns
        // the third of the window outside the row's reach (64 keys = packed P columns
        // [z, z + 16) and [z + 32, z + 48)), zeroed 8 packed columns per part
        const int colZ = (hi_half ? 0 : 2 * kC) + 32 * (part >> 1) + 8 * (part & 1);
        const int self_c0 = kC + 32 * q4;          // batch holding the rows' own columns
        const int dh = P.d / 4;                    // O columns of this warp
        uint32_t full_bits = 0;
        int ctr = 0;
        // epilogue state of the previous tile
        long long e_row = -1;
        float e_m2 = 0.f;
        bool e_live = false, e_self = false;
        bool ok = true;

        auto epilogue = [&](int q) -> bool {
            bool w = wait(&sb.o_full, q & 1, abort_flag, status, 0x702);
            // p_full of tile q (complete by now) orders the partner warp's partial sum
            w = w && wait(&sb.p_full[q & 1], (q >> 1) & 1, abort_flag, status, 0x704);
            if (!__all_sync(FULL, w)) return false;
            fence_after_sync();
            LSH_SPAN_BEGIN(t_ep);
            const float l = (l_part[q % kLBufs][0][i] + l_part[q % kLBufs][1][i]) +
                            (l_part[q % kLBufs][2][i] + l_part[q % kLBufs][3][i]);
            const float inv_l = l > 0.f ? 1.f / l : 0.f;
            __nv_bfloat16 *dst = o_r + LSH_IDX(e_row, (long long)n_rows, 0x712) * P.d + part * dh;
            if (dh == 32) {
                uint32_t o[32];
                tmem_ld32(tl + kTmemO + part * dh, o);
                tmem_wait_ld(o);
                if (e_live) {
                    uint32_t pk[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        pk[k] = pack_bf16(__uint_as_float(o[2 * k]) * inv_l,
                                          __uint_as_float(o[2 * k + 1]) * inv_l);
                    st_global_v8(dst, pk);
                    st_global_v8(dst + 16, pk + 8);
                }
            } else {
                uint32_t o[16];
                tmem_ld16(tl + kTmemO + part * dh, o);
                tmem_wait_ld16(o);
                if (e_live) {
                    uint32_t pk[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        pk[k] = pack_bf16(__uint_as_float(o[2 * k]) * inv_l,
                                          __uint_as_float(o[2 * k + 1]) * inv_l);
                    st_global_v8(dst, pk);
                }
            }
            if (e_live && part == 0)
                __stcs(&lse_r[LSH_IDX(e_row, (long long)n_rows, 0x713)],
                       e_self ? kSelfLogit : (e_m2 + __log2f(l)) * kLn2);
            LSH_SPAN_END(t_ep, 0x783);
            fence_before_sync();
            mbar_arrive(&sb.o_empty);
            return true;
        };

        ok = for_items(P, [&](long long seg, int tb, int te) -> bool {
            for (int t = tb; t < te; ++t) {
                LSH_SPAN_BEGIN(t_tile);
                auto need = [&](int c) -> bool {
                    const int s = c % kSlots;
                    bool w = wait(&sb.full[s], (full_bits >> s) & 1u, abort_flag, status, 0x701);
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
                LSH_SPAN_BEGIN(t_setup);

                // this row: its keys are the sorted indices [klo, khi) (minus itself when
                // not causal); the window of a row of chunk cq is chunks cq-1 and cq
                const int cq = 2 * t + hi_half;
                const int srow = t * kRows + i;
                const bool live = cq < P.nchunks;
                const SlotMeta &mq = meta[cq % kSlots];
                const int r = i & (kC - 1);
                int klo = 0, khi = 0;
                float m2 = 0.f;
                // where the row's outputs go: its sorted index, or its original position
                const int orow = P.token_order ? mq.jrow[r] : srow;
                if (live) {
                    // the row's bucket run clipped to its window, from the run marks of its
                    // chunk (and of the previous chunk when the run reaches back into it)
                    const unsigned long long sm = mq.starts & (~0ull >> (63 - r));
                    const unsigned long long sp = meta[(cq - 1 + kSlots) % kSlots].starts | 1ull;
                    klo = sm ? cq * kC + 63 - __clzll((long long)sm)
                             : (cq - 1) * kC + 63 - __clzll((long long)sp);
                    const unsigned long long em = mq.ends & (~0ull << r);
                    khi = P.causal ? srow : (em ? cq * kC + __ffsll((long long)em) : (cq + 1) * kC);
                    if (P.window == 32) {
                        // chunks of 32: the row's window is its 32-chunk and the one before,
                        // which lie inside its 64-row window; clip the run to it
                        const int w0 = (srow & ~31) - 32;
                        klo = max(klo, w0);
                        khi = min(khi, w0 + 64);
                    }
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
                if (__any_sync(FULL, live && m2 > (F16 ? kExactMaxLog2F16 : kExactMaxLog2))) {
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
                    named_bar_sync(1 + q4, 128);
                }

                LSH_SPAN_END(t_setup, 0x791);
                LSH_SPAN_BEGIN(t_sm);
                float l = 0.f;
                // This warp's 32 columns are one 32-key batch (a mask and key scales),
                // processed as two 16-column quarters; both loads are in flight before
                // the one wait.  P of quarter q (8 words at colA + 8 q) only covers S
                // columns already read.
                const bool nb0 = batch_needed(colA);
                const int t0 = tk0 + colA;                 // sorted index of batch column 0
                uint32_t vm0 = live ? range_mask(klo - t0, khi - t0) : 0u;
                if (colA == self_c0 && !P.causal) vm0 &= ~(1u << lane);
                const float *cs0 = meta[(2 * t - 1 + colA / kC + kSlots) % kSlots].cs + (colA & (kC - 1));
                const bool self_here = colA == self_c0;
                auto quarter = [&](const uint32_t (&sq)[16], int hq) {
                    uint32_t pk[8];
                    l += softmax_quarter<F16>(sq, cs0 + 16 * hq, vm0 >> (16 * hq), m2, pk);
                    if (self_here) {
                        // a row with no key but itself: weight 1 on its own column (all
                        // its other columns are masked).  Selects, not a conditional store
                        // into pk, which would move pk to local memory.
                        // 1.0 in the operand type: bf16 0x3F80, fp16 0x3C00
                        const uint32_t one16 = F16 ? 0x3C00u : 0x3F80u;
                        const uint32_t one = (lane & 1) ? one16 << 16 : one16;
                        const int kself = self_only && (lane >> 4) == hq ? (lane & 15) >> 1 : -1;
#pragma unroll
                        for (int k = 0; k < 8; ++k) pk[k] = k == kself ? one : pk[k];
                    }
                    tmem_st8(sbase + colA + 8 * hq, pk);
                };
                if (nb0) {
                    uint32_t qa[16], qb[16];
                    tmem_ld16(sbase + colA, qa);
                    tmem_ld16(sbase + colA + 16, qb);
                    tmem_wait_ld16(qa);
                    tmem_tie16(qb);
                    quarter(qa, 0);
                    quarter(qb, 1);
                } else {
                    tmem_st16_zero(sbase + colA);
                }
                if (self_here && self_only) l = 1.f;
                LSH_SPAN_END(t_sm, 0x781);
                LSH_SPAN_BEGIN(t_tail);
                {
                    const uint32_t z8[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
                    tmem_st8(sbase + colZ, z8);
                }
                l_part[ctr % kLBufs][part][i] = l;
                tmem_wait_st();
                fence_before_sync();
                mbar_arrive(&sb.p_full[b]);

                LSH_SPAN_END(t_tail, 0x792);
                if (ctr >= 1 && !epilogue(ctr - 1)) return false;
                e_live = live;
                e_row = seg * P.L + orow;
                e_m2 = m2;
                e_self = self_only;
                ++ctr;
                LSH_SPAN_END(t_tile, 0x790);
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
    // Loaders: every copy they issued lands before the CTA exits (after a timeout no
    // consumer may have waited for the last ones).
    if (warp >= kSmWarps && warp < kSmWarps + kLoaders) cp_async_wait_all();
}

bool make_plan(const Problem &p, AttnPlan &P)
{
    P.L = p.L; P.d = p.d; P.nb = p.nb; P.n_rounds = p.n_rounds; P.causal = p.causal;
    P.token_order = p.token_order;
    P.scale = p.scale;
    P.nchunks = p.L / kC;
    P.window = p.chunk;
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
    return 1024 + (size_t)2 * kSlots * nkb * kC * 128 + (size_t)kSlots * sizeof(SlotMeta);
}

}  // namespace

bool attn_tc_supported(const Problem &p)
{
    // chunk 32 runs as 64-row chunks with each row's keys clipped to its 32-row window
    return (p.dtype == LSH_BF16 || p.dtype == LSH_F16) && (p.d == 64 || p.d == 128) &&
           (p.chunk == kC || (p.chunk == 32 && p.L % kC == 0));
}

cudaError_t attn_tc(const Problem &p, const void *qk, const void *v, const int32_t *buckets,
                    const int32_t *perm, const int32_t *bstart, const float *inv_norm, void *o_r,
                    float *lse_r, StatusBlock *status, cudaStream_t st)
{
    (void)bstart;   // bucket runs come from the sorted rows' buckets (see the V loader)
    AttnPlan P;
    make_plan(p, P);
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const size_t smem = smem_bytes(P);
    // qk and v rows are copied as bytes; only the MMA operand type and P's packing differ
    auto kern = p.dtype == LSH_F16 ? lsh_attn_tc_kernel<true> : lsh_attn_tc_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<sms, kThreads, smem, st>>>((const __nv_bfloat16 *)qk, (const __nv_bfloat16 *)v, P, buckets, perm,
                                      inv_norm, (__nv_bfloat16 *)o_r, lse_r, status);
    return cudaGetLastError();
}

}  // namespace lsh
