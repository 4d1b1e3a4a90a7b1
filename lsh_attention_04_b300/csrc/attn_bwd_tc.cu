// attn_bwd_tc.cu -- backward pass of multi-round LSH attention for bf16 inputs, its five
// contractions on the tensor cores (warp-level bf16 MMA, fp32 accumulation).
//
// The derivative is the one attn_bwd.cu states (the Reformer pages train by
// back-propagation, modulabs-hub notes, "Introduction", but print no gradient): for the
// loss sum_i g_out_i . out_i + sum_i g_lse_i lse_i with the buckets held fixed,
//     pi_ij = exp(s_ij - LSE_i),   s_ij = scale * (qk_i . qk_j) / |qk_j|,
//     ds_ij = pi_ij (g_out_i . v_j - D_i + g_lse_i),      D_i = g_out_i . out_i,
//     dv_j  += pi_ij g_out_i,
//     dqk_i += scale sum_j ds_ij khat_j                       (query role)
//     dqk_j += (g - khat_j (khat_j . g)) / |qk_j|,  g = scale sum_i ds_ij qk_i   (key role).
//
// A prepass writes g_out in bf16 and D_i once per token.  Then one CTA per (head, round,
// chunk): the window is the previous chunk (rows 0..C-1; absent for chunk 0) and the own
// chunk (rows C..2C-1, which are also the query rows), its qk and v rows gathered through
// the permutation into shared memory in bf16 by 16-byte cp.async pieces.  Per 16 x 16 tile of the [C x 2C] score
// block a warp computes S = Q K^T and dP = G V^T (G = g_out in bf16), and from them, with
// the masks, pi and ds in fp32; it keeps pi, ds*scale/|k_j| and ds*scale in bf16 for the
// three products that follow:
//     dV^T-rows  = P^T G          [2C x d] over the C queries
//     g          = (ds scale)^T Q  [2C x d] over the C queries
//     dQ         = (ds scale/|k|) K  [C x d] over the 2C keys
// and adds them into dqk and dv (fp32, 16-byte atomics; the entry point clears both).
// Rows with no candidate in any round take 1/n_rounds of g_out in dv from each round, as
// in attn_bwd.cu.  No waits but __syncthreads / __syncwarp.
#include <limits.h>
#include <mma.h>

#include "internal.cuh"
#include "sm100.cuh"

namespace lsh {
namespace {

using namespace nvcuda;
using namespace sm100;

// g16 = bf16(g_out); dsum = g_out . out, one warp per token, 4 columns per lane.
__global__ void __launch_bounds__(256)
bwd_prep_kernel(const float *__restrict__ g_out, const float *__restrict__ out,
                __nv_bfloat16 *__restrict__ g16, float *__restrict__ dsum, long n_tok, int d)
{
    const int lane = threadIdx.x & 31;
    const long nwarps = ((long)gridDim.x * blockDim.x) >> 5;
    for (long t = (blockIdx.x * (long)blockDim.x + threadIdx.x) >> 5; t < n_tok; t += nwarps) {
        float s = 0.f;
        for (int c = lane * 4; c < d; c += 128) {
            const float4 g = *reinterpret_cast<const float4 *>(g_out + t * d + c);
            const float4 o = *reinterpret_cast<const float4 *>(out + t * d + c);
            s = fmaf(g.x, o.x, s);
            s = fmaf(g.y, o.y, s);
            s = fmaf(g.z, o.z, s);
            s = fmaf(g.w, o.w, s);
            __nv_bfloat162 a = __floats2bfloat162_rn(g.x, g.y), b = __floats2bfloat162_rn(g.z, g.w);
            uint2 u;
            u.x = *reinterpret_cast<uint32_t *>(&a);
            u.y = *reinterpret_cast<uint32_t *>(&b);
            *reinterpret_cast<uint2 *>(g16 + t * d + c) = u;
        }
        s = warp_sum(s);
        if (lane == 0) dsum[t] = s;
    }
}

template <int D, int C>
struct TcBwd {
    static constexpr int W = C / 4;          // warps: 16 at chunk 64, 8 at chunk 32
    static constexpr int T = W * 32;
    static constexpr int NW = 2 * C;         // window rows
    static constexpr int PB = D + 8;         // bf16 pitch of the qk, v and g rows
    static constexpr int PW = NW + 8;        // bf16 pitch of the [C][2C] score-shaped tiles
    static constexpr int PS = D + 4;         // fp32 pitch of the key-role staging
    static constexpr size_t r128(size_t x) { return (x + 127) & ~(size_t)127; }
    static constexpr size_t kK = 0;
    static constexpr size_t kG = kK + r128((size_t)NW * PB * 2);
    static constexpr size_t kE1 = kG + r128((size_t)C * PB * 2);
    static constexpr size_t kE2 = kE1 + r128((size_t)C * PW * 2);
    static constexpr size_t kU = kE2 + r128((size_t)C * PW * 2);
    // region U: V rows, P, and two 16 x 16 fp32 tiles per warp; later the key-role staging
    static constexpr size_t kV = kU;
    static constexpr size_t kP = kV + r128((size_t)NW * PB * 2);
    static constexpr size_t kStg = kP + r128((size_t)C * PW * 2);
    static constexpr size_t kUEnd = kStg + (size_t)W * 2 * 256 * 4;
    static constexpr size_t kGks = kU;       // fp32 [2C][PS], after V and P are done
    static_assert(kU + (size_t)NW * PS * 4 <= kUEnd, "key-role staging fits region U");
    static constexpr size_t kMeta = r128(kUEnd);
    // meta: tok[NW] bkt[NW] kin[NW] used[NW] lse[C] has[C] qmeta[C][2] qf[C][2]
    static constexpr size_t kBytes = kMeta + (size_t)4 * (4 * NW + 6 * C);
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ void atomic_add4(float *dst, float4 v)
{
    atomicAdd(reinterpret_cast<float4 *>(dst), v);
}

template <int D, int C>
__global__ void __launch_bounds__(TcBwd<D, C>::T, 1)
attn_bwd_tc_kernel(const __nv_bfloat16 *__restrict__ qk, const __nv_bfloat16 *__restrict__ v,
                   const int32_t *__restrict__ buckets, const int32_t *__restrict__ perm,
                   const float *__restrict__ inv_norm, const float *__restrict__ lse,
                   const float *__restrict__ g_out, const __nv_bfloat16 *__restrict__ g16,
                   const float *__restrict__ dsum, const float *__restrict__ g_lse, int L,
                   int n_rounds, int causal, float scale, float *__restrict__ dqk,
                   float *__restrict__ dv)
{
    using S = TcBwd<D, C>;
    constexpr int W = S::W, NW = S::NW, PB = S::PB, PW = S::PW, PS = S::PS;
    extern __shared__ __align__(128) uint8_t sm[];
    __nv_bfloat16 *Kb = reinterpret_cast<__nv_bfloat16 *>(sm + S::kK);
    __nv_bfloat16 *Gb = reinterpret_cast<__nv_bfloat16 *>(sm + S::kG);
    __nv_bfloat16 *E1 = reinterpret_cast<__nv_bfloat16 *>(sm + S::kE1);
    __nv_bfloat16 *E2 = reinterpret_cast<__nv_bfloat16 *>(sm + S::kE2);
    __nv_bfloat16 *Vb = reinterpret_cast<__nv_bfloat16 *>(sm + S::kV);
    __nv_bfloat16 *Pb = reinterpret_cast<__nv_bfloat16 *>(sm + S::kP);
    float *Gks = reinterpret_cast<float *>(sm + S::kGks);
    int *tok = reinterpret_cast<int *>(sm + S::kMeta);
    int *bkt = tok + NW;
    float *kin = reinterpret_cast<float *>(bkt + NW);
    int *used = reinterpret_cast<int *>(kin + NW);
    float *lq = reinterpret_cast<float *>(used + NW);
    int *has = reinterpret_cast<int *>(lq + C);
    int *qmeta = has + C;                                 // [C][2]: bucket, token of query q
    float *qf = reinterpret_cast<float *>(qmeta + 2 * C); // [C][2]: lse, D - g_lse

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float *stg_s = reinterpret_cast<float *>(sm + S::kStg) + warp * 512;
    float *stg_p = stg_s + 256;
    const long nch = L / C;
    const long seg = (long)blockIdx.x / nch;            // (batch, head, round)
    const int k = (int)((long)blockIdx.x - seg * nch);  // chunk
    const long bh = seg / n_rounds;
    const size_t head = (size_t)bh * L;
    const int32_t *P = perm + seg * L;

    // ---- 1. window rows (absent look-back rows of chunk 0 are zero and match nothing),
    //         every 16-byte piece issued before one wait ---------------------------------
    constexpr int PPR = D * 2 / 16;                     // 16-byte pieces per row
    for (int x = threadIdx.x; x < NW * PPR; x += S::T) {
        const int r = x / PPR, pc = x - r * PPR;
        const int s = k * C - C + r;                    // sorted index
        __nv_bfloat16 *dk = Kb + r * PB + pc * 8, *dvv = Vb + r * PB + pc * 8;
        if (s >= 0) {
            int j = P[s];
            if ((unsigned)j >= (unsigned)L) j = 0;
            cp_async16(smem_u32(dk), qk + (head + j) * D + pc * 8);
            cp_async16(smem_u32(dvv), v + (head + j) * D + pc * 8);
        } else {
            *reinterpret_cast<uint4 *>(dk) = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4 *>(dvv) = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    for (int x = threadIdx.x; x < C * PPR; x += S::T) {
        const int q = x / PPR, pc = x - q * PPR;
        int i = P[k * C + q];
        if ((unsigned)i >= (unsigned)L) i = 0;
        cp_async16(smem_u32(Gb + q * PB + pc * 8), g16 + (head + i) * D + pc * 8);
    }
    for (int r = threadIdx.x; r < NW; r += S::T) {
        const int s = k * C - C + r;
        const bool present = s >= 0;
        int j = present ? P[s] : 0;
        if ((unsigned)j >= (unsigned)L) j = 0;
        tok[r] = present ? j : INT_MAX;
        bkt[r] = present ? buckets[seg * L + j] : -1;
        kin[r] = present ? inv_norm[head + j] : 0.f;
        used[r] = 0;
        if (r >= C) {
            const int q = r - C;
            const float l = lse[head + j];
            lq[q] = l;
            qmeta[2 * q] = bkt[r];
            qmeta[2 * q + 1] = j;
            qf[2 * q] = l;
            qf[2 * q + 1] = dsum[head + j] - (g_lse ? g_lse[head + j] : 0.f);
            has[q] = 0;
        }
    }
    cp_async_wait_all();
    __syncthreads();

    // ---- 2. S = Q K^T and dP = G V^T per 16 x 16 tile; pi and ds with the masks ----------
    {
        constexpr int TK = NW / 16, TILES = (C / 16) * TK;
        for (int t = warp; t < TILES; t += W) {
            const int tq = t / TK, tk = t % TK;
            wmma::fragment<wmma::accumulator, 16, 16, 16, float> acc_s, acc_p;
            wmma::fill_fragment(acc_s, 0.f);
            wmma::fill_fragment(acc_p, 0.f);
#pragma unroll
            for (int dd = 0; dd < D / 16; ++dd) {
                wmma::fragment<wmma::matrix_a, 16, 16, 16, __nv_bfloat16, wmma::row_major> a;
                wmma::fragment<wmma::matrix_b, 16, 16, 16, __nv_bfloat16, wmma::col_major> b;
                wmma::load_matrix_sync(a, Kb + (C + 16 * tq) * PB + 16 * dd, PB);
                wmma::load_matrix_sync(b, Kb + (16 * tk) * PB + 16 * dd, PB);
                wmma::mma_sync(acc_s, a, b, acc_s);
                wmma::load_matrix_sync(a, Gb + (16 * tq) * PB + 16 * dd, PB);
                wmma::load_matrix_sync(b, Vb + (16 * tk) * PB + 16 * dd, PB);
                wmma::mma_sync(acc_p, a, b, acc_p);
            }
            wmma::store_matrix_sync(stg_s, acc_s, 16, wmma::mem_row_major);
            wmma::store_matrix_sync(stg_p, acc_p, 16, wmma::mem_row_major);
            __syncwarp();
            // lane: columns 2cp, 2cp+1 of the tile, rows rg, rg+4, rg+8, rg+12
            const int cp = lane & 7, rg = lane >> 3;
            const int r0 = 16 * tk + 2 * cp;
            const int2 bk = *reinterpret_cast<const int2 *>(bkt + r0);
            const int2 tk2 = *reinterpret_cast<const int2 *>(tok + r0);
            const float2 kn = *reinterpret_cast<const float2 *>(kin + r0);
            bool u0 = false, u1 = false;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int a = rg + 4 * m, q = 16 * tq + a, qi = C + q;
                const int2 bt = *reinterpret_cast<const int2 *>(qmeta + 2 * q);    // bucket, token
                const float2 lb = *reinterpret_cast<const float2 *>(qf + 2 * q);   // lse, D - g_lse
                const float2 sv = *reinterpret_cast<const float2 *>(stg_s + a * 16 + 2 * cp);
                const float2 pv = *reinterpret_cast<const float2 *>(stg_p + a * 16 + 2 * cp);
                const bool v0 = r0 != qi && bk.x == bt.x && bk.x >= 0 && (!causal || tk2.x < bt.y);
                const bool v1 = r0 + 1 != qi && bk.y == bt.x && bk.y >= 0 && (!causal || tk2.y < bt.y);
                const float p0 = v0 ? expf(sv.x * scale * kn.x - lb.x) : 0.f;
                const float p1 = v1 ? expf(sv.y * scale * kn.y - lb.x) : 0.f;
                const float d0 = p0 * (pv.x - lb.y), d1 = p1 * (pv.y - lb.y);
                *reinterpret_cast<__nv_bfloat162 *>(Pb + q * PW + r0) = __floats2bfloat162_rn(p0, p1);
                *reinterpret_cast<__nv_bfloat162 *>(E1 + q * PW + r0) =
                    __floats2bfloat162_rn(d0 * scale * kn.x, d1 * scale * kn.y);
                *reinterpret_cast<__nv_bfloat162 *>(E2 + q * PW + r0) =
                    __floats2bfloat162_rn(d0 * scale, d1 * scale);
                if (v0 || v1) has[q] = 1;
                u0 |= v0;
                u1 |= v1;
            }
            if (u0) used[r0] = 1;
            if (u1) used[r0 + 1] = 1;
            __syncwarp();
        }
    }
    __syncthreads();

    // ---- 3. dv_j += sum_i pi_ij g_out_i  (P^T G); tokens with no key in any round --------
    {
        constexpr int TR = NW / 16, TILES = TR * (D / 16);
        for (int t = warp; t < TILES; t += W) {
            const int tr = t % TR, tc = t / TR;
            wmma::fragment<wmma::accumulator, 16, 16, 16, float> acc;
            wmma::fill_fragment(acc, 0.f);
#pragma unroll
            for (int iq = 0; iq < C / 16; ++iq) {
                wmma::fragment<wmma::matrix_a, 16, 16, 16, __nv_bfloat16, wmma::col_major> a;
                wmma::fragment<wmma::matrix_b, 16, 16, 16, __nv_bfloat16, wmma::row_major> b;
                wmma::load_matrix_sync(a, Pb + (16 * iq) * PW + 16 * tr, PW);
                wmma::load_matrix_sync(b, Gb + (16 * iq) * PB + 16 * tc, PB);
                wmma::mma_sync(acc, a, b, acc);
            }
            wmma::store_matrix_sync(stg_s, acc, 16, wmma::mem_row_major);
            __syncwarp();
            const int r = 16 * tr + (lane >> 1), c0 = 8 * (lane & 1);
            if (used[r]) {
                float *dst = dv + (head + tok[r]) * D + 16 * tc + c0;
                const float *src = stg_s + (lane >> 1) * 16 + c0;
                atomic_add4(dst, make_float4(src[0], src[1], src[2], src[3]));
                atomic_add4(dst + 4, make_float4(src[4], src[5], src[6], src[7]));
            }
            __syncwarp();
        }
        const float wself = 1.0f / (float)n_rounds;
        for (int q = warp; q < C; q += W) {
            if (has[q] || !(lq[q] < 0.5f * kSelfLogit)) continue;
            const int i = tok[C + q];
            for (int c = lane * 4; c < D; c += 128) {
                const float4 g = *reinterpret_cast<const float4 *>(g_out + (head + i) * D + c);
                atomic_add4(dv + (head + i) * D + c,
                            make_float4(wself * g.x, wself * g.y, wself * g.z, wself * g.w));
            }
        }
    }
    __syncthreads();

    // ---- 4. key role: g_j = sum_i (ds_ij scale) qk_i, then the normalisation Jacobian ----
    {
        constexpr int TR = NW / 16, TILES = TR * (D / 16);
        for (int t = warp; t < TILES; t += W) {
            const int tr = t % TR, tc = t / TR;
            wmma::fragment<wmma::accumulator, 16, 16, 16, float> acc;
            wmma::fill_fragment(acc, 0.f);
#pragma unroll
            for (int iq = 0; iq < C / 16; ++iq) {
                wmma::fragment<wmma::matrix_a, 16, 16, 16, __nv_bfloat16, wmma::col_major> a;
                wmma::fragment<wmma::matrix_b, 16, 16, 16, __nv_bfloat16, wmma::row_major> b;
                wmma::load_matrix_sync(a, E2 + (16 * iq) * PW + 16 * tr, PW);
                wmma::load_matrix_sync(b, Kb + (C + 16 * iq) * PB + 16 * tc, PB);
                wmma::mma_sync(acc, a, b, acc);
            }
            wmma::store_matrix_sync(Gks + (16 * tr) * PS + 16 * tc, acc, PS, wmma::mem_row_major);
        }
        __syncthreads();
        for (int r = warp; r < NW; r += W) {
            if (!used[r]) continue;                     // also every absent row
            const float kr = kin[r];
            float proj = 0.f;
            float kh[4] = {0.f, 0.f, 0.f, 0.f}, g[4] = {0.f, 0.f, 0.f, 0.f};
            const int c = lane * 4;
            if (c < D) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    kh[e] = __bfloat162float(Kb[r * PB + c + e]) * kr;
                    g[e] = Gks[r * PS + c + e];
                    proj = fmaf(kh[e], g[e], proj);
                }
            }
            proj = warp_sum(proj);
            if (c < D)
                atomic_add4(dqk + (head + tok[r]) * D + c,
                            make_float4(kr * (g[0] - kh[0] * proj), kr * (g[1] - kh[1] * proj),
                                        kr * (g[2] - kh[2] * proj), kr * (g[3] - kh[3] * proj)));
        }
    }
    __syncthreads();

    // ---- 5. query role: dqk_i += sum_j (ds_ij scale / |k_j|) qk_j ------------------------
    {
        constexpr int TQ = C / 16, TILES = TQ * (D / 16);
        for (int t = warp; t < TILES; t += W) {
            const int tq = t % TQ, tc = t / TQ;
            wmma::fragment<wmma::accumulator, 16, 16, 16, float> acc;
            wmma::fill_fragment(acc, 0.f);
#pragma unroll
            for (int ir = 0; ir < NW / 16; ++ir) {
                wmma::fragment<wmma::matrix_a, 16, 16, 16, __nv_bfloat16, wmma::row_major> a;
                wmma::fragment<wmma::matrix_b, 16, 16, 16, __nv_bfloat16, wmma::row_major> b;
                wmma::load_matrix_sync(a, E1 + (16 * tq) * PW + 16 * ir, PW);
                wmma::load_matrix_sync(b, Kb + (16 * ir) * PB + 16 * tc, PB);
                wmma::mma_sync(acc, a, b, acc);
            }
            wmma::store_matrix_sync(stg_s, acc, 16, wmma::mem_row_major);
            __syncwarp();
            const int q = 16 * tq + (lane >> 1), c0 = 8 * (lane & 1);
            if (has[q]) {
                float *dst = dqk + (head + tok[C + q]) * D + 16 * tc + c0;
                const float *src = stg_s + (lane >> 1) * 16 + c0;
                atomic_add4(dst, make_float4(src[0], src[1], src[2], src[3]));
                atomic_add4(dst + 4, make_float4(src[4], src[5], src[6], src[7]));
            }
            __syncwarp();
        }
    }
}

template <int D, int C>
cudaError_t launch_tc(const Problem &p, const void *qk, const void *v, const int32_t *buckets,
                      const int32_t *perm, const float *inv_norm, const float *lse,
                      const float *g_out, const __nv_bfloat16 *g16, const float *dsum,
                      const float *g_lse, float *dqk, float *dv, cudaStream_t st)
{
    const size_t smem = TcBwd<D, C>::kBytes;
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_tc_kernel<D, C>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const long blocks = p.n_seg() * (p.L / C);
    attn_bwd_tc_kernel<D, C><<<(unsigned)blocks, TcBwd<D, C>::T, smem, st>>>(
        (const __nv_bfloat16 *)qk, (const __nv_bfloat16 *)v, buckets, perm, inv_norm, lse, g_out,
        g16, dsum, g_lse, p.L, p.n_rounds, p.causal, p.scale, dqk, dv);
    return cudaGetLastError();
}


// ---------------------------------------------------------------------------------------
// d = 128, chunk 64: the five contractions on the tcgen05 tensor cores.
//
// One unit per (head, round, 128-row tile): query rows = chunks 2t and 2t+1 of the sorted
// segment, window = chunks 2t-1 .. 2t+1 (192 rows; the first 64 absent for t = 0).
// Persistent CTAs, one per SM, take the units in turn (TMEM and the barriers set up once).  The
// operands live in shared memory as planes of 64 columns, each plane rows x 128 bytes
// with the 128-byte swizzle; one such tile serves as a K-major operand (rows = M or N,
// columns = K) and as an MN-major one (rows = K, columns = M or N) through its
// descriptor.  TMEM (512 columns):
//     phase 1   S = Q K^T   [0, 192)    dP = G V^T  [192, 384)        (M 128, N 192)
//     pass A    E1 = ds scale / |k|,  E2 = ds scale  (bf16 tiles; E2 over the V rows)
//               dQ = E1 K   [384, 512)                                 (M 128, N 128)
//     pass B    P = pi (bf16, over E1; kept in registers since pass A)
//     phase 2   dV^T = G^T P   [0, 192)     dK^T = Q^T E2   [192, 384) (M = d, N 192)
//     epilogue  dV^T, dK^T + dQ through the freed v / g_out / P tiles as fp32 rows, each
//               added to dv or dqk by one warp
// Warps w, w + 4, w + 8 and w + 12 share TMEM lane quarter w (a query row, or in phase 2
// a column d) and split the columns four ways; warp 4 also issues the MMAs and owns TMEM;
// all sixteen gather.
// A row's keys are one interval of the window (its bucket run, clipped to its window, and
// before it when causal), from run bounds computed once per unit.  One mbarrier takes a
// unit's first two commits (phase 1, then dQ: waited with parities 0 and 1 by warps that
// saw the one before), a second its last (phase 2: every MMA of the unit, waited with the
// unit's count mod 2), so no wait can alias a phase.  The next unit's permutation entries
// and row metadata are fetched (4-byte cp.async) while the current one computes.

// 2^x by the special-function unit (relative error near 2^-22).  Results below 2^-126
// flush to 0: the weights here are a token's softmax weights over the keys of all its
// rounds (their total is 1), so a flushed one is below 2^-126 of that total.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
constexpr int kT5Rows = 128, kT5Win = 192, kT5D = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kT5Threads = 512;
constexpr int kPlK = kT5Win * 128;                   // window-tile plane (192 rows)
constexpr int kPlQ = kT5Rows * 128;                  // query-tile plane (128 rows)
constexpr size_t kT5OffK = 0;                        // qk window rows, 2 planes
constexpr size_t kT5OffV = kT5OffK + 2 * kPlK;       // v window rows, 2 planes; then E2
constexpr size_t kT5OffG = kT5OffV + 2 * kPlK;       // g_out query rows, 2 planes
constexpr size_t kT5OffP = kT5OffG + 2 * kPlQ;       // E1, then P: 3 planes of 64 keys
constexpr size_t kT5OffMeta = kT5OffP + 3 * kPlQ;
static_assert(2 * kPlK == 3 * kPlQ, "E2 (3 key planes) fits the v rows (2 d planes)");
struct T5Meta {
    int tok[kT5Win], bkt[kT5Win];
    float kin[kT5Win], kcs[kT5Win];                  // 1/|k|, scale log2(e) / |k|
    int rs[kT5Win], re[kT5Win];                      // bucket run of each window row: [rs, re)
    float lq[kT5Rows], base[kT5Rows];                // lse log2(e), D - g_lse of each query row
    int has[kT5Rows];
    unsigned used[kT5Win / 32];
};
constexpr size_t kT5Smem = 1024 + kT5OffMeta + sizeof(T5Meta);

// byte offset of element (row, col) of a tile of `plane` bytes per 64-column plane
__device__ __forceinline__ uint32_t sw_off(int row, int col, int plane)
{
    return (uint32_t)((col >> 6) * plane + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4) + (col & 7) * 2);
}

// 16 consecutive columns [c0, c0 + 16) of row `row` of a 16-bit tile, from fp32 values
__device__ __forceinline__ void put_row16(uint8_t *tile, int plane, int row, int c0, const float (&x)[16])
{
#pragma unroll
    for (int g = 0; g < 2; ++g) {
        uint4 u;
        u.x = pack_bf16x2(x[8 * g], x[8 * g + 1]);
        u.y = pack_bf16x2(x[8 * g + 2], x[8 * g + 3]);
        u.z = pack_bf16x2(x[8 * g + 4], x[8 * g + 5]);
        u.w = pack_bf16x2(x[8 * g + 6], x[8 * g + 7]);
        *reinterpret_cast<uint4 *>(tile + sw_off(row, c0 + 8 * g, plane)) = u;
    }
}
// the same 16 columns from bf16 pairs already packed (word k = columns c0 + 2k, c0 + 2k + 1)
__device__ __forceinline__ void put_row16p(uint8_t *tile, int plane, int row, int c0, const uint32_t (&u)[8])
{
#pragma unroll
    for (int g = 0; g < 2; ++g)
        *reinterpret_cast<uint4 *>(tile + sw_off(row, c0 + 8 * g, plane)) =
            make_uint4(u[4 * g], u[4 * g + 1], u[4 * g + 2], u[4 * g + 3]);
}
__global__ void __launch_bounds__(kT5Threads, 1)
attn_bwd_tc5_kernel(const __nv_bfloat16 *__restrict__ qk, const __nv_bfloat16 *__restrict__ v,
                    const int32_t *__restrict__ buckets, const int32_t *__restrict__ perm,
                    const float *__restrict__ inv_norm, const float *__restrict__ lse,
                    const float *__restrict__ g_out, const __nv_bfloat16 *__restrict__ g16,
                    const float *__restrict__ dsum, const float *__restrict__ g_lse, int L,
                    int n_rounds, int causal, float scale, float *__restrict__ dqk,
                    float *__restrict__ dv, long n_units, StatusBlock *status)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t bar_mma, bar_done;            // phases 1 and pass A's MMA; phase 2
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag_s;
    // the next unit's permutation entries and row metadata, fetched while this one computes
    __shared__ int nx_tok[kT5Win], nx_bkt[kT5Win];
    __shared__ float nx_kin[kT5Win], nx_lse[kT5Win], nx_dsum[kT5Win], nx_glse[kT5Win];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *Kt = sm + kT5OffK, *Vt = sm + kT5OffV, *Gt = sm + kT5OffG, *Pt = sm + kT5OffP;
    T5Meta &mt = *reinterpret_cast<T5Meta *>(sm + kT5OffMeta);
    volatile int *abort_flag = &abort_flag_s;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tps = (L + kT5Rows - 1) / kT5Rows;

    if (threadIdx.x == 0) {
        mbar_init(&bar_mma, 1);
        mbar_init(&bar_done, 1);
        abort_flag_s = 0;
        mbar_fence_init();
    }
    if (warp == 4) tmem_alloc(&tmem_slot, 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = tmem_slot;
    const uint32_t kb = smem_u32(Kt), vb = smem_u32(Vt), gb = smem_u32(Gt), pb = smem_u32(Pt);

    // persistent: units u = seg * tps + t, strided over the grid
    int it = 0;
    bool failed = false;
    for (long u = blockIdx.x; u < n_units; u += gridDim.x, ++it) {
    const long seg = u / tps;
    const int t = (int)(u - seg * tps);
    const long bh = seg / n_rounds;
    const size_t head = (size_t)bh * L;
    const int32_t *Pm = perm + seg * L;
    const long un = u + gridDim.x;                 // this CTA's next unit
    const long seg2 = un / tps;
    const int t2 = (int)(un - seg2 * tps);
    LSH_SPAN_BEGIN(t_all);
    LSH_SPAN_BEGIN(t_gather);

    // ---- 1. gather: window rows w (sorted 128 t - 64 + w) and query rows q (128 t + q,
    // the window's rows 64 + q).  The permutation entries and row metadata of every unit
    // but a CTA's first were fetched during its previous unit (nx_*); the row copies are
    // issued from shared memory with no load on their path.
    const bool pre = it > 0;
    for (int w = threadIdx.x; w < kT5Win; w += kT5Threads) {
        const int s = kT5Rows * t - 64 + w;
        const bool in = s >= 0 && s < L;
        const int j = in ? (pre ? nx_tok[w] : Pm[s]) : INT_MAX;
        mt.tok[w] = in ? ((unsigned)j < (unsigned)L ? j : 0) : INT_MAX;
        if (w < kT5Win / 32) mt.used[w] = 0u;
    }
    __syncthreads();
    for (int x = threadIdx.x; x < kT5Win * 16; x += kT5Threads) {
        const int w = x >> 4, pc = x & 15;
        const uint32_t o = sw_off(w, 8 * pc, kPlK);
        const int j = mt.tok[w];
        if (j != INT_MAX) {
            cp_async16(smem_u32(Kt + o), qk + (head + j) * kT5D + 8 * pc);
            cp_async16(smem_u32(Vt + o), v + (head + j) * kT5D + 8 * pc);
        } else {
            *reinterpret_cast<uint4 *>(Kt + o) = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4 *>(Vt + o) = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    for (int x = threadIdx.x; x < kT5Rows * 16; x += kT5Threads) {
        const int q = x >> 4, pc = x & 15;
        const uint32_t o = sw_off(q, 8 * pc, kPlQ);
        const int i = mt.tok[64 + q];
        if (i != INT_MAX)
            cp_async16(smem_u32(Gt + o), g16 + (head + i) * kT5D + 8 * pc);
        else
            *reinterpret_cast<uint4 *>(Gt + o) = make_uint4(0u, 0u, 0u, 0u);
    }
    for (int w = threadIdx.x; w < kT5Win; w += kT5Threads) {
        const int j = mt.tok[w];
        const bool present = j != INT_MAX;
        const int jj = present ? j : 0;
        const float kn = present ? (pre ? nx_kin[w] : inv_norm[head + jj]) : 0.f;
        mt.bkt[w] = present ? (pre ? nx_bkt[w] : buckets[seg * L + jj]) : -1;
        mt.kin[w] = kn;
        mt.kcs[w] = scale * kLog2e * kn;
        if (w >= 64) {
            const int q = w - 64;
            const float l = pre ? nx_lse[w] : lse[head + jj];
            const float ds = pre ? nx_dsum[w] : dsum[head + jj];
            const float gl = g_lse ? (pre ? nx_glse[w] : g_lse[head + jj]) : 0.f;
            mt.lq[q] = present ? l * kLog2e : 0.f;
            mt.base[q] = present ? ds - gl : 0.f;
            mt.has[q] = 0;
        }
    }
    __syncthreads();
    LSH_SPAN_END(t_gather, 0xa01);
    LSH_SPAN_BEGIN(t_runs);
    // bucket runs of the window (sorted order keeps a bucket's rows together): warp 0 scans
    // the start flags forward and the end flags backward, 32 rows at a time
    if (warp == 0) {
        int carry = 0;
        for (int b0 = 0; b0 < kT5Win; b0 += 32) {
            const int w = b0 + lane;
            int x = (w == 0 || mt.bkt[w] != mt.bkt[w - 1]) ? w : 0;   // a run starts here
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) x = max(x, __shfl_up_sync(0xffffffffu, x, o));
            x = max(x, carry);
            mt.rs[w] = x;
            carry = __shfl_sync(0xffffffffu, x, 31);
        }
        carry = kT5Win;
        for (int b0 = kT5Win - 32; b0 >= 0; b0 -= 32) {
            const int w = b0 + lane;
            int x = (w == kT5Win - 1 || mt.bkt[w] != mt.bkt[w + 1]) ? w + 1 : kT5Win;   // ends here
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) x = min(x, __shfl_down_sync(0xffffffffu, x, o));
            x = min(x, carry);
            mt.re[w] = x;
            carry = __shfl_sync(0xffffffffu, x, 0);
        }
    }
    cp_async_wait_all();
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    LSH_SPAN_END(t_runs, 0xa02);

    // ---- 2. phase 1: S = Q K^T, dP = G V^T
    if (warp == 4) {
        const uint32_t idesc = idesc_bf16(kT5Rows, kT5Win, 0, 0);
        for (int ks = 0; ks < kT5D / 16; ++ks) {
            const int pl = ks >> 2, ko = (ks & 3) * 32;
            mma_ss(tmem, smem_desc(kb + pl * kPlK + 64 * 128 + ko, 16, 1024),
                   smem_desc(kb + pl * kPlK + ko, 16, 1024), idesc, ks > 0);
            mma_ss(tmem + kT5Win, smem_desc(gb + pl * kPlQ + ko, 16, 1024),
                   smem_desc(vb + pl * kPlK + ko, 16, 1024), idesc, ks > 0);
        }
        mma_commit(smem_u32(&bar_mma));
    }

    // rows: warps w, w + 4, w + 8, w + 12 share TMEM lane quarter w (query q = its lane)
    // and split the columns four ways (keys [48 p, 48 p + 48), d [32 p, 32 p + 32))
    const int quarter = warp & 3, part = warp >> 2;
    const int q = 32 * quarter + lane, qi = 64 + q;
    const bool qlive = kT5Rows * t + q < L;
    const uint32_t tl = tmem + ((uint32_t)(32 * quarter) << 16);
    // the row's keys: its bucket run inside its window ([0, 128) for chunk 2t, [64, 192) for
    // 2t+1), before it when causal (sorted order is position order inside a bucket), itself
    // excluded
    const int wlo = q < 64 ? 0 : 64;
    const int klo = qlive ? max(wlo, mt.rs[qi]) : 0;
    const int khi = qlive ? (causal ? qi : min(wlo + 128, mt.re[qi])) : 0;
    const float lq2 = qlive ? mt.lq[q] : 0.f, bs = qlive ? mt.base[q] : 0.f;
    bool ok = true;

    // the row's weights pi (and score gradients ds) of keys [16 c, 16 c + 16)
    auto row_batch = [&](int c, float (&pi)[16], float (&ds)[16]) -> unsigned {
        uint32_t sv[16], pv[16];
        tmem_ld16(tl + 16 * c, sv);
        tmem_ld16(tl + kT5Win + 16 * c, pv);
        tmem_wait_ld16(sv);
        tmem_tie16(pv);
        unsigned vm = 0u;
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
            const int w = 16 * c + jj;
            const bool valid = w >= klo && w < khi && w != qi;
            pi[jj] = valid ? ex2(fmaf(__uint_as_float(sv[jj]), mt.kcs[w], -lq2)) : 0.f;
            ds[jj] = pi[jj] * (__uint_as_float(pv[jj]) - bs);
            vm |= valid ? 1u << jj : 0u;
        }
        return vm;
    };

    // ---- 3. pass A: E1 = ds scale / |k| (over P), E2 = ds scale (over the v rows); the
    // row's P stays in registers (bf16 pairs) until dQ has read E1
    uint32_t pp[3][8];
    {
        ok = wait(&bar_mma, 0, abort_flag, status, 0x901);
        fence_after_sync();
        LSH_SPAN_BEGIN(t_pa);
        // the next unit's permutation entries (this thread's window row), in flight until
        // the epilogue
        if (un < n_units && threadIdx.x < kT5Win) {
            const int s2 = kT5Rows * t2 - 64 + (int)threadIdx.x;
            if (s2 >= 0 && s2 < L) cp_async4(smem_u32(&nx_tok[threadIdx.x]), perm + seg2 * L + s2);
        }
        bool any = false;
#pragma unroll
        for (int cc = 0; cc < 3; ++cc) {
            const int c = 3 * part + cc;
            float pi[16], ds[16], e1[16], e2[16];
            const unsigned vm = row_batch(c, pi, ds);
#pragma unroll
            for (int k = 0; k < 8; ++k) pp[cc][k] = pack_bf16x2(pi[2 * k], pi[2 * k + 1]);
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
                e2[jj] = ds[jj] * scale;
                e1[jj] = e2[jj] * mt.kin[16 * c + jj];
            }
            put_row16(Pt, kPlQ, q, 16 * c, e1);
            put_row16(Vt, kPlQ, q, 16 * c, e2);
            any |= vm != 0u;
            const unsigned col = __reduce_or_sync(0xffffffffu, vm);
            if (lane == 0 && col) atomicOr(&mt.used[c >> 1], col << (16 * (c & 1)));
        }
        if (any) atomicOr(&mt.has[q], 1);
        fence_proxy_async();
        LSH_SPAN_END(t_pa, 0xa03);
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();

    // ---- 4. dQ = E1 K (K-major E1 rows, the qk window rows as an MN-major operand)
    if (warp == 4) {
        const uint32_t idesc = idesc_bf16(kT5Rows, kT5D, 0, 1);
        for (int ks = 0; ks < kT5Win / 16; ++ks) {
            const int pl = ks >> 2, ko = (ks & 3) * 32;
            mma_ss(tmem + 2 * kT5Win, smem_desc(pb + pl * kPlQ + ko, 16, 1024),
                   smem_desc(kb + 16 * ks * 128, kPlK, 1024), idesc, ks > 0);
        }
        mma_commit(smem_u32(&bar_mma));
    }

    // ---- 5. pass B: P over E1 once dQ has read it
    {
        ok = wait(&bar_mma, 1, abort_flag, status, 0x902) && ok;
        fence_after_sync();
        LSH_SPAN_BEGIN(t_pb);
#pragma unroll
        for (int cc = 0; cc < 3; ++cc) put_row16p(Pt, kPlQ, q, 16 * (3 * part + cc), pp[cc]);
        fence_proxy_async();
        LSH_SPAN_END(t_pb, 0xa04);
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();

    // ---- 6. phase 2: dV^T = G^T P, dK^T = Q^T E2 (both operands MN-major)
    if (warp == 4) {
        const uint32_t idesc = idesc_bf16(kT5D, kT5Win, 1, 1);
        for (int ks = 0; ks < kT5Rows / 16; ++ks) {
            mma_ss(tmem, smem_desc(gb + 16 * ks * 128, kPlQ, 1024),
                   smem_desc(pb + 16 * ks * 128, kPlQ, 1024), idesc, ks > 0);
            mma_ss(tmem + kT5Win, smem_desc(kb + (64 + 16 * ks) * 128, kPlK, 1024),
                   smem_desc(vb + 16 * ks * 128, kPlQ, 1024), idesc, ks > 0);
        }
        mma_commit(smem_u32(&bar_done));
    }

    // ---- 7. epilogue (all eight warps).  After the last commit every MMA has read its
    // operands, so the v, g_out and P tiles (128 KB from kT5OffV) are free.  The gradients
    // pass through them as fp32 rows [window row][d] (528-byte pitch: the rows a warp
    // touches at once fall on distinct banks), and a warp adds a whole 512-byte row to dv
    // or dqk with one float4 atomic per lane (lane l: d = 4 l .. 4 l + 3), where one token
    // per lane would scatter 32 rows per instruction.  A token that is both a key (window
    // row 64 + q) and a query (row q) of the tile gets its two dqk terms summed here
    // first, so it costs one row update instead of two.
    {
        ok = wait(&bar_done, it & 1, abort_flag, status, 0x903) && ok;
        fence_after_sync();
        LSH_SPAN_BEGIN(t_eq);
        // the next unit's row metadata, from its permutation entries (landed by now)
        if (un < n_units && threadIdx.x < kT5Win) {
            const int w = threadIdx.x, s2 = kT5Rows * t2 - 64 + w;
            cp_async_wait_all();
            if (s2 >= 0 && s2 < L) {
                int j = nx_tok[w];
                j = (unsigned)j < (unsigned)L ? j : 0;
                const size_t head2 = (size_t)(seg2 / n_rounds) * L;
                cp_async4(smem_u32(&nx_bkt[w]), buckets + seg2 * L + j);
                cp_async4(smem_u32(&nx_kin[w]), inv_norm + head2 + j);
                if (w >= 64) {
                    cp_async4(smem_u32(&nx_lse[w]), lse + head2 + j);
                    cp_async4(smem_u32(&nx_dsum[w]), dsum + head2 + j);
                    if (g_lse) cp_async4(smem_u32(&nx_glse[w]), g_lse + head2 + j);
                }
            }
        }
        constexpr int kXs = kT5D + 4;
        float *X = reinterpret_cast<float *>(sm + kT5OffV);
        const int tq = qlive ? mt.tok[qi] : 0;
        const int d = 32 * quarter + lane;
        auto key_used = [&](int w) { return (mt.used[w >> 5] >> (w & 31)) & 1u; };
        // dV^T or dK^T (TMEM lane = d, columns = window keys) into the rows
        auto stage_keys = [&](uint32_t col0) {
#pragma unroll
            for (int cc = 0; cc < 3; ++cc) {
                const int c = 3 * part + cc;
                uint32_t r[16];
                tmem_ld16(tl + col0 + 16 * c, r);
                tmem_wait_ld16(r);
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) X[(16 * c + jj) * kXs + d] = __uint_as_float(r[jj]);
            }
        };
        stage_keys(0);
        __syncthreads();
        for (int w = warp; w < kT5Win; w += kT5Threads / 32)
            if (key_used(w) && ok)
                atomicAdd(reinterpret_cast<float4 *>(dv + (head + mt.tok[w]) * kT5D) + lane,
                          reinterpret_cast<const float4 *>(X + w * kXs)[lane]);
        __syncthreads();
        LSH_SPAN_END(t_eq, 0xa05);
        LSH_SPAN_BEGIN(t_ek);
        stage_keys(kT5Win);
        __syncthreads();
        // key role: dqk_j += (g - khat (khat . g)) / |k_j|, khat = k_j / |k_j|, the dot over
        // the row's d by the warp (lane l: d = 4 l .. 4 l + 3); rows of unused keys become 0
        for (int w = warp; w < kT5Win; w += kT5Threads / 32) {
            float4 *xr = reinterpret_cast<float4 *>(X + w * kXs);
            float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
            if (key_used(w)) {                                           // warp-uniform
                const float4 g = xr[lane];
                const uint2 kr = *reinterpret_cast<const uint2 *>(Kt + sw_off(w, 4 * lane, kPlK));
                const float2 k01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kr.x));
                const float2 k23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kr.y));
                const float kn = mt.kin[w];
                const float h0 = k01.x * kn, h1 = k01.y * kn, h2 = k23.x * kn, h3 = k23.y * kn;
                const float dot = warp_sum(h0 * g.x + h1 * g.y + h2 * g.z + h3 * g.w);
                val = make_float4(kn * (g.x - h0 * dot), kn * (g.y - h1 * dot),
                                  kn * (g.z - h2 * dot), kn * (g.w - h3 * dot));
            }
            xr[lane] = val;
        }
        __syncthreads();
        {
            // query role: dQ (TMEM lane = query row q, this warp's quarter of d) onto row
            // 64 + q
            uint32_t r0[32];
            tmem_ld32(tl + 2 * kT5Win + 32 * part, r0);
            tmem_wait_ld(r0);
            float4 *xr = reinterpret_cast<float4 *>(X + qi * kXs) + 8 * part;
#pragma unroll
            for (int g4 = 0; g4 < 8; ++g4) {
                float4 a = xr[g4];
                a.x += __uint_as_float(r0[4 * g4]);     a.y += __uint_as_float(r0[4 * g4 + 1]);
                a.z += __uint_as_float(r0[4 * g4 + 2]); a.w += __uint_as_float(r0[4 * g4 + 3]);
                xr[g4] = a;
            }
        }
        __syncthreads();
        for (int w = warp; w < kT5Win; w += kT5Threads / 32) {
            const int qq = w - 64;
            const bool qrow = qq >= 0 && kT5Rows * t + qq < L && mt.has[qq];
            if ((key_used(w) || qrow) && ok)                             // warp-uniform
                atomicAdd(reinterpret_cast<float4 *>(dqk + (head + mt.tok[w]) * kT5D) + lane,
                          reinterpret_cast<const float4 *>(X + w * kXs)[lane]);
        }
        LSH_SPAN_END(t_ek, 0xa06);
        // a token with no key in any round copies v_i: 1 / n_rounds of g_out from each round
        if (part == 0 && ok && qlive && !mt.has[q] && mt.lq[q] < 0.5f * kSelfLogit * kLog2e) {
            const float wself = 1.0f / (float)n_rounds;
            for (int c = 0; c < kT5D; c += 4) {
                const float4 g = *reinterpret_cast<const float4 *>(g_out + (head + tq) * kT5D + c);
                atomicAdd(reinterpret_cast<float4 *>(dv + (head + tq) * kT5D + c),
                          make_float4(wself * g.x, wself * g.y, wself * g.z, wself * g.w));
            }
        }
    }
    LSH_SPAN_END(t_all, 0xa0f);
    // the next unit overwrites the tiles, the staged rows and TMEM: every thread is done
    // with them, and its prefetched metadata has landed (a failed wait anywhere ends the
    // loop for the whole CTA)
    cp_async_wait_all();
    fence_before_sync();
    failed = __syncthreads_or(!ok) != 0;
    fence_after_sync();
    if (failed) break;
    }

    // ---- teardown.  Normally every MMA has completed (each unit waited for its last
    // commit); after a failed wait, give the unit's MMAs a bounded wait first.
    if (warp == 4 && failed) {
        int dummy = 0;
        wait_w(&bar_done, it & 1, &dummy, status, 0x904);
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 4) {
        fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

bool attn_bwd_tc_supported(const Problem &p)
{
    return p.dtype == LSH_BF16 && (p.d == 64 || p.d == 128) && (p.chunk == 32 || p.chunk == 64);
}

size_t attn_bwd_tc_scratch_bytes(const Problem &p)
{
    return attn_bwd_tc_supported(p) ? (size_t)p.n_tok() * (2 * p.d + 4) : 0;
}

cudaError_t attn_bwd_tc(const Problem &p, const void *qk, const void *v, const int32_t *buckets,
                        const int32_t *perm, const float *inv_norm, const float *out,
                        const float *lse, const float *g_out, const float *g_lse, float *dqk,
                        float *dv, void *scratch, StatusBlock *status, cudaStream_t st)
{
    __nv_bfloat16 *g16 = (__nv_bfloat16 *)scratch;
    float *dsum = (float *)((char *)scratch + (size_t)p.n_tok() * p.d * 2);
    const long n_tok = p.n_tok();
    const long warps = n_tok < 148L * 64 ? n_tok : 148L * 64;
    bwd_prep_kernel<<<(unsigned)((warps * 32 + 255) / 256), 256, 0, st>>>(g_out, out, g16, dsum,
                                                                          n_tok, p.d);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (p.d == 64 && p.chunk == 32)
        return launch_tc<64, 32>(p, qk, v, buckets, perm, inv_norm, lse, g_out, g16, dsum, g_lse, dqk, dv, st);
    if (p.d == 64 && p.chunk == 64)
        return launch_tc<64, 64>(p, qk, v, buckets, perm, inv_norm, lse, g_out, g16, dsum, g_lse, dqk, dv, st);
    if (p.d == 128 && p.chunk == 32)
        return launch_tc<128, 32>(p, qk, v, buckets, perm, inv_norm, lse, g_out, g16, dsum, g_lse, dqk, dv, st);
    if (p.d == 128 && p.chunk == 64) {
        e = cudaFuncSetAttribute(attn_bwd_tc5_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kT5Smem);
        if (e != cudaSuccess) return e;
        const long units = p.n_seg() * ((p.L + kT5Rows - 1) / kT5Rows);
        int dev = 0, sms = 148;
        if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        const long grid = units < sms ? units : sms;
        attn_bwd_tc5_kernel<<<(unsigned)grid, kT5Threads, kT5Smem, st>>>(
            (const __nv_bfloat16 *)qk, (const __nv_bfloat16 *)v, buckets, perm, inv_norm, lse, g_out,
            g16, dsum, g_lse, p.L, p.n_rounds, p.causal, p.scale, dqk, dv, units, status);
        return cudaGetLastError();
    }
    return cudaErrorInvalidValue;
}

}  // namespace lsh
