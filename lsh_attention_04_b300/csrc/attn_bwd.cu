// attn_bwd.cu -- backward pass of multi-round LSH attention (gradients in qk and v).
//
// The Reformer pages train the model by back-propagation (modulabs-hub notes,
// "Introduction") but print no gradient; this is the derivative of the forward pass for the
// loss  sum_i g_out_i . out_i + sum_i g_lse_i lse_i,  with the buckets held fixed (the hash
// is piecewise constant).  The rounds' logsumexp weighting makes every (round, candidate)
// pair of token i one entry of a single softmax with weight
//     pi_ij = exp(s_ij - LSE_i),   s_ij = scale * (qk_i . qk_j) / |qk_j|,
// LSE_i being the forward's combined lse.  Differentiating out_i = sum pi_ij v_j and LSE_i:
//     ds_ij   = pi_ij (g_out_i . v_j - D_i + g_lse_i),      D_i = g_out_i . out_i
//     dv_j   += pi_ij g_out_i
//     dqk_i  += scale * sum_j ds_ij khat_j                    (query role, khat = unit key)
//     dqk_j  += (g - khat_j (khat_j . g)) / |qk_j|,  g = scale * sum_i ds_ij qk_i  (key role)
// A round in which token i has no candidate copies v_i with weight exp(-1e5 - LSE_i): that
// is 1/n_rounds when every round of token i is like that (LSE_i = -1e5 + ln n_rounds,
// recognised as LSE_i < -5e4) and underflows to 0 otherwise.
//
// One CTA per (head, round, chunk).  Its query rows are the chunk's sorted rows, its keys
// the look-one-back window (previous chunk + own chunk), all staged in shared memory in
// fp32; pi and then ds live in a [chunk][2 chunk] tile.  Query-role gradients are added
// once per round, key-role and value gradients once per window holding the key (twice per
// round), by fp32 atomics into dqk and dv, which the caller clears first.  CUDA cores, fp32.
#include "internal.cuh"

namespace lsh {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <int D, int C>
struct BwdSmem {
    // row stride in floats: rows stay 16-byte aligned, and lanes reading float4s of
    // consecutive rows fall on distinct bank groups
    static constexpr int kStride = D + 4;
    float K[2 * C][kStride];  // window rows of qk
    float V[2 * C][kStride];  // window rows of v
    float G[C][kStride];      // g_out of the query rows
    float X[C][2 * C];        // pi, then ds
    float kin[2 * C];         // 1/|qk_j| of the window rows
    int tok[2 * C];           // original positions of the window rows
    int bkt[2 * C];           // their buckets in this round
    int used[2 * C];          // the key is a candidate of some query row
    float lse[C], Dq[C], glse[C];
    int has[C];               // the query row has a candidate
};

template <int N>
__device__ __forceinline__ float dot4(const float *a, const float *b)
{
    const float4 *x = reinterpret_cast<const float4 *>(a);
    const float4 *y = reinterpret_cast<const float4 *>(b);
    float s = 0.f;
#pragma unroll 8
    for (int c = 0; c < N / 4; ++c) {
        const float4 u = x[c], w = y[c];
        s = fmaf(u.x, w.x, s);
        s = fmaf(u.y, w.y, s);
        s = fmaf(u.z, w.z, s);
        s = fmaf(u.w, w.w, s);
    }
    return s;
}

template <typename T, int D, int C>
__global__ void __launch_bounds__(kThreads, 1)
attn_bwd_kernel(const T *__restrict__ qk, const T *__restrict__ v,
                const int32_t *__restrict__ buckets, const int32_t *__restrict__ perm,
                const float *__restrict__ inv_norm, const float *__restrict__ out,
                const float *__restrict__ lse, const float *__restrict__ g_out,
                const float *__restrict__ g_lse, int L, int n_rounds, int causal, float scale,
                float *__restrict__ dqk, float *__restrict__ dv)
{
    constexpr int EPL = D / 32;  // columns per lane: lane, lane + 32, ...
    extern __shared__ float4 smem_f4[];
    BwdSmem<D, C> &sm = *reinterpret_cast<BwdSmem<D, C> *>(smem_f4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const long nch = L / C;
    const long seg = (long)blockIdx.x / nch;          // (batch, head, round)
    const int k = (int)((long)blockIdx.x - seg * nch);  // chunk
    const long bh = seg / n_rounds;
    const int lo = k > 0 ? (k - 1) * C : 0;           // first sorted index of the window
    const int nW = (k + 1) * C - lo;                  // window rows: C or 2C
    const int qoff = k * C - lo;                      // window index of the first query row
    const int32_t *P = perm + seg * L;
    const size_t head = (size_t)bh * L;

    // ---- 1. stage the window rows and the query rows' gradients --------------------------
    for (int r = warp; r < nW; r += kWarps) {
        const int j = P[lo + r];
        const size_t row = (head + j) * D;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            sm.K[r][e * 32 + lane] = ld_f32(qk, row + e * 32 + lane);
            sm.V[r][e * 32 + lane] = ld_f32(v, row + e * 32 + lane);
        }
        if (lane == 0) {
            sm.tok[r] = j;
            sm.bkt[r] = buckets[seg * L + j];
            sm.kin[r] = inv_norm[head + j];
            sm.used[r] = 0;
        }
    }
    for (int q = warp; q < C; q += kWarps) {
        const int i = P[k * C + q];
        const size_t row = (head + i) * D;
        float dsum = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            const float g = g_out[row + e * 32 + lane];
            sm.G[q][e * 32 + lane] = g;
            dsum = fmaf(g, out[row + e * 32 + lane], dsum);
        }
        dsum = warp_sum(dsum);
        if (lane == 0) {
            sm.Dq[q] = dsum;
            sm.lse[q] = lse[head + i];
            sm.glse[q] = g_lse ? g_lse[head + i] : 0.f;
            sm.has[q] = 0;
        }
    }
    __syncthreads();

    // ---- 2. pi_ij for the candidates (own or previous chunk, same bucket, not self,
    //         earlier position when causal), 0 elsewhere ------------------------------------
    for (int q = warp; q < C; q += kWarps) {
        const int sq = qoff + q;
        const int ti = sm.tok[sq], bi = sm.bkt[sq];
        const float li = sm.lse[q];
        bool any = false;
        for (int r = lane; r < 2 * C; r += 32) {
            float x = 0.f;
            if (r < nW && r != sq && sm.bkt[r] == bi && (!causal || sm.tok[r] < ti)) {
                x = expf(scale * dot4<D>(sm.K[sq], sm.K[r]) * sm.kin[r] - li);
                any = true;
                sm.used[r] = 1;
            }
            sm.X[q][r] = x;
        }
        if (__any_sync(0xffffffffu, any) && lane == 0) sm.has[q] = 1;
    }
    __syncthreads();

    // ---- 3. dv_j += sum_i pi_ij g_out_i;  rows with no candidate in any round ----------------
    for (int r = warp; r < nW; r += kWarps) {
        if (!sm.used[r]) continue;
        float acc[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
        for (int q = 0; q < C; ++q) {
            const float x = sm.X[q][r];
            if (x == 0.f) continue;
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[e] = fmaf(x, sm.G[q][e * 32 + lane], acc[e]);
        }
        float *dst = dv + (head + sm.tok[r]) * D;
#pragma unroll
        for (int e = 0; e < EPL; ++e) atomicAdd(dst + e * 32 + lane, acc[e]);
    }
    const float wself = 1.0f / (float)n_rounds;
    for (int q = warp; q < C; q += kWarps) {
        if (sm.has[q] || !(sm.lse[q] < 0.5f * kSelfLogit)) continue;
        float *dst = dv + (head + sm.tok[qoff + q]) * D;
#pragma unroll
        for (int e = 0; e < EPL; ++e) atomicAdd(dst + e * 32 + lane, wself * sm.G[q][e * 32 + lane]);
    }
    __syncthreads();

    // ---- 4. ds_ij = pi_ij (g_out_i . v_j - D_i + g_lse_i), in place ---------------------------
    for (int q = warp; q < C; q += kWarps) {
        const float base = sm.glse[q] - sm.Dq[q];
        for (int r = lane; r < nW; r += 32) {
            const float x = sm.X[q][r];
            if (x == 0.f) continue;
            sm.X[q][r] = x * (dot4<D>(sm.G[q], sm.V[r]) + base);
        }
    }
    __syncthreads();

    // ---- 5. query role: dqk_i += scale * sum_j ds_ij khat_j --------------------------------
    for (int q = warp; q < C; q += kWarps) {
        if (!sm.has[q]) continue;
        float acc[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
        for (int r = 0; r < nW; ++r) {
            const float x = sm.X[q][r];
            if (x == 0.f) continue;
            const float w = x * sm.kin[r];
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[e] = fmaf(w, sm.K[r][e * 32 + lane], acc[e]);
        }
        float *dst = dqk + (head + sm.tok[qoff + q]) * D;
#pragma unroll
        for (int e = 0; e < EPL; ++e) atomicAdd(dst + e * 32 + lane, scale * acc[e]);
    }

    // ---- 6. key role: g = scale * sum_i ds_ij qk_i;  dqk_j += (g - khat (khat . g)) / |qk_j|
    for (int r = warp; r < nW; r += kWarps) {
        if (!sm.used[r]) continue;
        float g[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) g[e] = 0.f;
        for (int q = 0; q < C; ++q) {
            const float x = sm.X[q][r];
            if (x == 0.f) continue;
#pragma unroll
            for (int e = 0; e < EPL; ++e) g[e] = fmaf(x, sm.K[qoff + q][e * 32 + lane], g[e]);
        }
        const float kin = sm.kin[r];
        float proj = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            g[e] *= scale;
            proj = fmaf(sm.K[r][e * 32 + lane] * kin, g[e], proj);
        }
        proj = warp_sum(proj);
        float *dst = dqk + (head + sm.tok[r]) * D;
#pragma unroll
        for (int e = 0; e < EPL; ++e)
            atomicAdd(dst + e * 32 + lane, kin * (g[e] - sm.K[r][e * 32 + lane] * kin * proj));
    }
}

template <typename T, int D, int C>
cudaError_t launch(const Problem &p, const void *qk, const void *v, const int32_t *buckets,
                   const int32_t *perm, const float *inv_norm, const float *out, const float *lse,
                   const float *g_out, const float *g_lse, float *dqk, float *dv, cudaStream_t st)
{
    const size_t smem = sizeof(BwdSmem<D, C>);
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_kernel<T, D, C>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const long blocks = p.n_seg() * (p.L / C);
    attn_bwd_kernel<T, D, C><<<(unsigned)blocks, kThreads, smem, st>>>(
        (const T *)qk, (const T *)v, buckets, perm, inv_norm, out, lse, g_out, g_lse, p.L,
        p.n_rounds, p.causal, p.scale, dqk, dv);
    return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch(const Problem &p, const void *qk, const void *v, const int32_t *buckets,
                     const int32_t *perm, const float *inv_norm, const float *out,
                     const float *lse, const float *g_out, const float *g_lse, float *dqk,
                     float *dv, cudaStream_t st)
{
    if (p.d == 64 && p.chunk == 32)
        return launch<T, 64, 32>(p, qk, v, buckets, perm, inv_norm, out, lse, g_out, g_lse, dqk, dv, st);
    if (p.d == 64 && p.chunk == 64)
        return launch<T, 64, 64>(p, qk, v, buckets, perm, inv_norm, out, lse, g_out, g_lse, dqk, dv, st);
    if (p.d == 128 && p.chunk == 32)
        return launch<T, 128, 32>(p, qk, v, buckets, perm, inv_norm, out, lse, g_out, g_lse, dqk, dv, st);
    if (p.d == 128 && p.chunk == 64)
        return launch<T, 128, 64>(p, qk, v, buckets, perm, inv_norm, out, lse, g_out, g_lse, dqk, dv, st);
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t attn_bwd(const Problem &p, const void *qk, const void *v, const int32_t *buckets,
                     const int32_t *perm, const float *inv_norm, const float *out, const float *lse,
                     const float *g_out, const float *g_lse, float *dqk, float *dv, cudaStream_t st)
{
    if (p.dtype == LSH_BF16)
        return dispatch<__nv_bfloat16>(p, qk, v, buckets, perm, inv_norm, out, lse, g_out, g_lse,
                                       dqk, dv, st);
    if (p.dtype == LSH_F16)
        return dispatch<__half>(p, qk, v, buckets, perm, inv_norm, out, lse, g_out, g_lse, dqk,
                                dv, st);
    return dispatch<float>(p, qk, v, buckets, perm, inv_norm, out, lse, g_out, g_lse, dqk, dv, st);
}

}  // namespace lsh
