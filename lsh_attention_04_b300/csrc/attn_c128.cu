// attn_c128.cu -- chunked look-one-back LSH attention at chunk 128 on the tcgen05 tensor
// cores (bf16 or fp16 inputs, d = 128, L a multiple of 128).
//
// "Reformer" glossary (ultralytics.com), section "Atencion LSH": the bucket-sorted
// sequence is cut into equal chunks; each token attends to its own chunk and the
// previous one.  modulabs-hub Reformer notes, section "LSH attention": keys outside the
// query's bucket get -infinity, the token itself is removed (it stays only when nothing
// else is left), and in the causal case only earlier positions remain.  Keys are
// L2-normalised, queries are not.
//
// One unit = chunk t of one (batch, head, round) segment: its 128 sorted rows are the
// queries and the window of chunks t-1 and t (256 sorted rows; the first 128 absent for
// t = 0) holds every key they may see.
//   S = Q K^T   tcgen05.mma M=128, N=256 (the whole window), K=16 steps over d, fp32 into
//               TMEM columns [0, 256); Q is the window's last 128 rows.
//   P           packed 16-bit pairs written over S: the 32 keys of S columns 32j..32j+31
//               go to columns 32j..32j+15, so a warp overwrites only columns it has read.
//   O = P V     M=128, N=d, K=16-key steps with A read from TMEM and V an MN-major
//               shared-memory operand, into TMEM columns [256, 384).
// A query's keys are one interval of the window: its bucket run (sorted order keeps a
// bucket together and position order inside it, so "causal" is "before the row"), less
// the row itself when not causal.  Run bounds come from a forward max-scan of run starts
// and a backward min-scan of run ends over the window's rows, once per unit.
// Softmax without a running maximum, as in the chunk-64 kernel: with unit keys every score
// of query i is at most m_i = |scale| |q_i| and at least -m_i, so p = 2^(s log2e - m_i
// log2e) lies in [2^(-2 m2), 1] (m2 = m_i log2 e); above m2 = 32 (7 for fp16 weights) the
// row takes its exact maximum instead.  A row with no key but itself gives its own column
// weight 1 (O = v_i) and lse the self logit.
// Persistent CTAs of 16 warps, one per SM, take the units in turn and run each one's
// gather, S, softmax, P V and epilogue in sequence: warps w, w+4, w+8 and w+12 share TMEM
// lane quarter w (32 query rows) and split the 256 key columns and the 128 output columns
// four ways; warp 0 also issues the MMAs and owns TMEM.  The next unit's permutation
// entries and row metadata are fetched (4-byte cp.async) while the current one computes.
// Every wait is bounded (sm100::wait).
#include <limits.h>
#include <math.h>

#include "sm100.cuh"

namespace lsh {
namespace {

using namespace sm100;

constexpr int kC = 128;           // chunk = query rows per unit
constexpr int kWin = 256;         // window rows (previous chunk + own chunk)
constexpr int kD = 128;
constexpr int kThreads = 512;     // 16 warps
constexpr int kPl = kWin * 128;   // one 64-column plane of a window tile (bytes)
constexpr int kTmemO = kWin;      // O accumulator column
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kExactMaxLog2 = 32.f;
constexpr float kExactMaxLog2F16 = 7.f;

struct __align__(16) C128Meta {
    int tok[kWin];         // original position of each window row (INT_MAX: absent)
    int bkt[kWin];         // bucket (-1: absent)
    float kcs[kWin];       // key column scale: scale * log2(e) / |k_j|
    int rs[kWin], re[kWin];// bucket run of each window row: [rs, re)
    float m2[kC];          // query bound in log2 units: |scale| * log2(e) * |q_i|
    float lpart[4][kC];    // partial row sums of the four column parts
};
constexpr size_t kOffK = 0, kOffV = 2 * (size_t)kPl, kOffMeta = 4 * (size_t)kPl;
constexpr size_t kSmem = 1024 + kOffMeta + sizeof(C128Meta);

// byte offset of element (row, col) of a window tile (64-column planes, 128-byte swizzle)
__device__ __forceinline__ uint32_t sw_off(int row, int col)
{
    return (uint32_t)((col >> 6) * kPl + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4) + (col & 7) * 2);
}
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ uint32_t pack16(float lo, float hi, bool f16) {
    if (f16) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
// Key columns [lo, hi) of a 32-column batch as a bit mask.
__device__ __forceinline__ uint32_t range_mask(int lo, int hi) {
    lo = max(lo, 0);
    hi = min(hi, 32);
    if (lo >= hi) return 0u;
    const uint32_t below_hi = hi == 32 ? 0xffffffffu : (1u << hi) - 1u;
    return below_hi & (0xffffffffu << lo);
}
// p TMEM column of the 16-key step m (keys 16m .. 16m+15 as 8 packed columns)
__host__ __device__ __forceinline__ int p_col(int m) { return 32 * (m >> 1) + 8 * (m & 1); }

// One 16-column quarter of a row: p_j = 2^(s_j * cs_j - m2) where bit j of vm is set, else
// 0, packed to 16-bit pairs; returns sum_j p_j.  cs is 16-byte aligned shared memory.
template <bool F16>
__device__ __forceinline__ float quarter(const uint32_t (&s16)[16], const float *cs, uint32_t vm,
                                         float m2, uint32_t (&pk)[8]) {
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
        pk[2 * q] = pack16(p[0], p[1], F16);
        pk[2 * q + 1] = pack16(p[2], p[3], F16);
        la += p[0] + p[1];
        lb += p[2] + p[3];
    }
    return la + lb;
}

template <bool F16>
__global__ void __launch_bounds__(kThreads, 1)
lsh_attn_c128_kernel(const __nv_bfloat16 *__restrict__ qk, const __nv_bfloat16 *__restrict__ vv,
                     const int32_t *__restrict__ buckets, const int32_t *__restrict__ perm,
                     const float *__restrict__ inv_norm, int L, int n_rounds, long n_units,
                     int causal, float scale, int token_order, __nv_bfloat16 *__restrict__ o_r,
                     float *__restrict__ lse_r, StatusBlock *status)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t bar_s, bar_o;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag_s;
    // the next unit's permutation entries and row metadata, fetched while this one computes
    __shared__ int nx_tok[kWin], nx_bkt[kWin];
    __shared__ float nx_kin[kWin];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    C128Meta &mt = *reinterpret_cast<C128Meta *>(sm + kOffMeta);
    volatile int *abort_flag = &abort_flag_s;
    const uint32_t FULL = 0xffffffffu;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q4 = warp & 3, part = warp >> 2;
    const int i = 32 * q4 + lane;                  // query row = TMEM lane
    const int qw = kC + i;                         // its window row
    const int self_c0 = kC + 32 * q4;              // batch holding the rows' own columns
    const int tpc = L / kC;                        // units per segment
    const float ascale = fabsf(scale) * kLog2e, cscale = scale * kLog2e;
    const uint32_t kb = smem_u32(sm + kOffK), vb = smem_u32(sm + kOffV);

    if (threadIdx.x == 0) {
        mbar_init(&bar_s, 1);
        mbar_init(&bar_o, 1);
        abort_flag_s = 0;
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(&tmem_slot, 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = tmem_slot;
    const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);

    int it = 0;
    bool failed = false;
    for (long u = blockIdx.x; u < n_units; u += gridDim.x, ++it) {
        const long seg = u / tpc;
        const int t = (int)(u - seg * tpc);
        const long bh = seg / n_rounds;
        const size_t head = (size_t)bh * L;
        const int32_t *Pm = perm + seg * L;
        const int w0 = kC * (t - 1);               // sorted index of window row 0
        const long un = u + gridDim.x;             // this CTA's next unit
        const long seg2 = un / tpc;
        const int t2 = (int)(un - seg2 * tpc);
        const bool pre = it > 0;                   // this unit's metadata was prefetched

        // ---- 1. the window's permutation entries, then its rows and row metadata
        for (int w = threadIdx.x; w < kWin; w += kThreads) {
            const int s = w0 + w;
            const int j = s >= 0 ? (pre ? nx_tok[w] : Pm[s]) : INT_MAX;
            mt.tok[w] = s >= 0 ? ((unsigned)j < (unsigned)L ? j : 0) : INT_MAX;
        }
        __syncthreads();
        for (int x = threadIdx.x; x < kWin * 16; x += kThreads) {
            const int w = x >> 4, pc = x & 15;
            const uint32_t o = sw_off(w, 8 * pc);
            const int j = mt.tok[w];
            if (j != INT_MAX) {
                cp_async16(kb + o, qk + (head + j) * kD + 8 * pc);
                cp_async16(vb + o, vv + (head + j) * kD + 8 * pc);
            } else {
                *reinterpret_cast<uint4 *>(sm + kOffK + o) = make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4 *>(sm + kOffV + o) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        for (int w = threadIdx.x; w < kWin; w += kThreads) {
            const int j = mt.tok[w];
            const bool present = j != INT_MAX;
            const int jj = present ? j : 0;
            const float kn = present ? (pre ? nx_kin[w] : inv_norm[head + jj]) : 0.f;
            mt.bkt[w] = present ? (pre ? nx_bkt[w] : buckets[seg * L + jj]) : -1;
            mt.kcs[w] = cscale * kn;
            if (w >= kC) mt.m2[w - kC] = kn > 0.f ? ascale / kn : 0.f;
        }
        __syncthreads();
        // bucket runs of the window: warp 0 scans the start flags forward and the end
        // flags backward, 32 rows at a time
        if (warp == 0) {
            int carry = 0;
            for (int b0 = 0; b0 < kWin; b0 += 32) {
                const int w = b0 + lane;
                int x = (w == 0 || mt.bkt[w] != mt.bkt[w - 1]) ? w : 0;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) x = max(x, __shfl_up_sync(FULL, x, o));
                x = max(x, carry);
                mt.rs[w] = x;
                carry = __shfl_sync(FULL, x, 31);
            }
            carry = kWin;
            for (int b0 = kWin - 32; b0 >= 0; b0 -= 32) {
                const int w = b0 + lane;
                int x = (w == kWin - 1 || mt.bkt[w] != mt.bkt[w + 1]) ? w + 1 : kWin;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) x = min(x, __shfl_down_sync(FULL, x, o));
                x = min(x, carry);
                mt.re[w] = x;
                carry = __shfl_sync(FULL, x, 0);
            }
        }
        cp_async_wait_all();
        fence_proxy_async();                       // rows written by cp.async, read by MMA
        fence_before_sync();
        __syncthreads();
        fence_after_sync();

        // ---- 2. S = Q K^T
        if (warp == 0) {
            const uint32_t idesc = idesc_16(kC, kWin, 0, 0, F16);
            for (int ks = 0; ks < kD / 16; ++ks) {
                const int pl = ks >> 2, ko = (ks & 3) * 32;
                mma_ss(tmem, smem_desc(kb + pl * kPl + kC * 128 + ko, 16, 1024),
                       smem_desc(kb + pl * kPl + ko, 16, 1024), idesc, ks > 0);
            }
            mma_commit(smem_u32(&bar_s));
        }

        // the row's keys: window rows [klo, khi), minus itself when not causal
        const int klo = mt.rs[qw];
        const int khi = causal ? qw : mt.re[qw];
        const bool self_only = causal ? klo >= khi : khi - klo <= 1;
        float m2 = mt.m2[i];
        auto batch_needed = [&](int c0) -> bool {
            const bool nb = (klo < c0 + 32 && khi > c0 && klo < khi) || (self_only && c0 == self_c0);
            return __any_sync(FULL, nb);
        };
        bool ok = __all_sync(FULL, wait(&bar_s, it & 1, abort_flag, status, 0xc01));
        fence_after_sync();
        // the next unit's permutation entries (this thread's window row), in flight until
        // the epilogue
        if (un < n_units && threadIdx.x < kWin) {
            const int s2 = kC * (t2 - 1) + (int)threadIdx.x;
            if (s2 >= 0) cp_async4(smem_u32(&nx_tok[threadIdx.x]), perm + seg2 * L + s2);
        }

        // ---- 3. softmax over this warp's 64 columns; P over S
        if (ok) {
            if (__any_sync(FULL, m2 > (F16 ? kExactMaxLog2F16 : kExactMaxLog2))) {
                // exact maximum over the row's keys; the lane quarter's four warps take the
                // same branch (same rows) and all read S before any of them writes P
                float mx = -INFINITY;
                for (int c0 = 0; c0 < kWin; c0 += 32) {
                    if (!batch_needed(c0)) continue;
                    uint32_t s32[32];
                    tmem_ld32(tl + c0, s32);
                    tmem_wait_ld(s32);
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) {
                        const int w = c0 + jj;
                        if (w >= klo && w < khi && (causal || w != qw))
                            mx = fmaxf(mx, __uint_as_float(s32[jj]) * mt.kcs[w]);
                    }
                }
                m2 = mx == -INFINITY ? 0.f : mx;
                named_bar_sync(1 + q4, 128);
            }
            float l = 0.f;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int c0 = 64 * part + 32 * h;
                if (!batch_needed(c0)) {
                    tmem_st16_zero(tl + c0);
                    continue;
                }
                uint32_t vm = range_mask(klo - c0, khi - c0);
                if (c0 == self_c0 && !causal) vm &= ~(1u << lane);
                uint32_t sa[16], sb[16];
                tmem_ld16(tl + c0, sa);
                tmem_ld16(tl + c0 + 16, sb);
                tmem_wait_ld16(sa);
                tmem_tie16(sb);
#pragma unroll
                for (int hq = 0; hq < 2; ++hq) {
                    uint32_t pk[8];
                    l += quarter<F16>(hq ? sb : sa, &mt.kcs[c0 + 16 * hq], vm >> (16 * hq), m2, pk);
                    if (c0 == self_c0) {
                        // a row with no key but itself: weight 1 on its own column (all its
                        // other columns are masked); selects keep pk in registers
                        const uint32_t one16 = F16 ? 0x3C00u : 0x3F80u;
                        const uint32_t one = (lane & 1) ? one16 << 16 : one16;
                        const int kself = self_only && (lane >> 4) == hq ? (lane & 15) >> 1 : -1;
#pragma unroll
                        for (int k = 0; k < 8; ++k) pk[k] = k == kself ? one : pk[k];
                    }
                    tmem_st8(tl + c0 + 8 * hq, pk);
                }
                if (c0 == self_c0 && self_only) l = 1.f;
            }
            mt.lpart[part][i] = l;
        }
        tmem_wait_st();
        fence_before_sync();
        __syncthreads();
        fence_after_sync();

        // ---- 4. O = P V
        if (warp == 0 && __all_sync(FULL, ok)) {
            const uint32_t idesc = idesc_16(kC, kD, 0, 1, F16);
            for (int m = 0; m < kWin / 16; ++m)
                mma_ts(tmem + kTmemO, tmem + p_col(m), smem_desc(vb + m * 2048, kPl, 1024), idesc, m > 0);
            mma_commit(smem_u32(&bar_o));
        }

        // the next unit's row metadata, from its permutation entries (landed by now)
        if (un < n_units && threadIdx.x < kWin) {
            const int w = threadIdx.x, s2 = kC * (t2 - 1) + w;
            cp_async_wait_all();
            if (s2 >= 0) {
                int j = nx_tok[w];
                j = (unsigned)j < (unsigned)L ? j : 0;
                cp_async4(smem_u32(&nx_bkt[w]), buckets + seg2 * L + j);
                cp_async4(smem_u32(&nx_kin[w]), inv_norm + (size_t)(seg2 / n_rounds) * L + j);
            }
        }

        // ---- 5. epilogue: O / l in 16 bits, lse
        if (ok) {
            ok = __all_sync(FULL, wait(&bar_o, it & 1, abort_flag, status, 0xc02));
            fence_after_sync();
        }
        if (ok) {
            const float lt = (mt.lpart[0][i] + mt.lpart[1][i]) + (mt.lpart[2][i] + mt.lpart[3][i]);
            const float inv_l = lt > 0.f ? 1.f / lt : 0.f;
            const long long orow = seg * (long long)L + (token_order ? mt.tok[qw] : kC * t + i);
            uint32_t o[32];
            tmem_ld32(tl + kTmemO + 32 * part, o);
            tmem_wait_ld(o);
            uint32_t pk[16];
#pragma unroll
            for (int k = 0; k < 16; ++k)
                pk[k] = pack16(__uint_as_float(o[2 * k]) * inv_l, __uint_as_float(o[2 * k + 1]) * inv_l, false);
            __nv_bfloat16 *dst = o_r + orow * kD + 32 * part;
            *reinterpret_cast<uint4 *>(dst) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            *reinterpret_cast<uint4 *>(dst + 8) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            *reinterpret_cast<uint4 *>(dst + 16) = make_uint4(pk[8], pk[9], pk[10], pk[11]);
            *reinterpret_cast<uint4 *>(dst + 24) = make_uint4(pk[12], pk[13], pk[14], pk[15]);
            if (part == 0) lse_r[orow] = self_only ? kSelfLogit : (m2 + __log2f(lt)) * kLn2;
        }
        // the next unit overwrites the tiles, the metadata and TMEM: every thread is done
        // with them, and its prefetched metadata has landed (a failed wait anywhere ends
        // the loop for the whole CTA)
        cp_async_wait_all();
        fence_before_sync();
        failed = __syncthreads_or(!ok) != 0;
        fence_after_sync();
        if (failed) break;
    }

    // ---- teardown.  Normally every MMA has completed (each unit waited for its P V);
    // after a failed wait, give the unit's MMAs a bounded wait first.
    if (warp == 0 && failed) {
        int dummy = 0;
        wait_w(&bar_s, it & 1, &dummy, status, 0xc03);
        wait_w(&bar_o, it & 1, &dummy, status, 0xc04);
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

bool attn_c128_supported(const Problem &p)
{
    return (p.dtype == LSH_BF16 || p.dtype == LSH_F16) && p.d == kD && p.chunk == kC &&
           p.L % kC == 0;
}

cudaError_t attn_c128(const Problem &p, const void *qk, const void *v, const int32_t *buckets,
                      const int32_t *perm, const float *inv_norm, void *o_r, float *lse_r,
                      StatusBlock *status, cudaStream_t st)
{
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long units = p.n_seg() * (p.L / kC);
    const long grid = units < sms ? units : sms;
    auto kern = p.dtype == LSH_F16 ? lsh_attn_c128_kernel<true> : lsh_attn_c128_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    if (e != cudaSuccess) return e;
    if (grid == 0) return cudaSuccess;
    kern<<<(unsigned)grid, kThreads, kSmem, st>>>((const __nv_bfloat16 *)qk, (const __nv_bfloat16 *)v,
                                                 buckets, perm, inv_norm, p.L, p.n_rounds, units,
                                                 p.causal, p.scale, p.token_order,
                                                 (__nv_bfloat16 *)o_r, lse_r, status);
    return cudaGetLastError();
}

}  // namespace lsh
