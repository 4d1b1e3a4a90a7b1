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
using sm100::cp_async16;
using sm100::cp_async_wait_all;
using sm100::smem_u32;

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
                        float *dv, void *scratch, cudaStream_t st)
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
    if (p.d == 128 && p.chunk == 64)
        return launch_tc<128, 64>(p, qk, v, buckets, perm, inv_norm, lse, g_out, g16, dsum, g_lse, dqk, dv, st);
    return cudaErrorInvalidValue;
}

}  // namespace lsh
