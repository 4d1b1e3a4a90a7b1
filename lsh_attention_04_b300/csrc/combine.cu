// combine.cu -- un-sort the per-round outputs and combine the rounds.
//
// Each round r produced an output row o_r and its log-normaliser lse_r per token, in
// sorted order (token i's row of round r at sorted index inv_r[i]) or, inside the fused
// forward, already in token order (at i; no index lookups).  The rounds are weighted by
// their share of the total softmax mass:
//   lse_i = logsumexp_r lse_r(i),   out_i = sum_r exp(lse_r(i) - lse_i) * o_r(i).
// (Rounds run in parallel per the "Reformer" glossary, section "Atencion LSH"; the
// logsumexp weighting is the standard way to merge softmax results computed over
// separate key sets.)
//
// One warp per token.  Lane r fetches inv_r[i] and lse_r of round r (all rounds at
// once, so the index lookups cost one dependent round trip, not one per round), the
// warp reduces the weights with shuffles, and then every round's row is requested
// before any is accumulated (up to 8 rows in flight per warp).  Each lane owns D/32
// consecutive elements of a row: one 4- to 16-byte vector load per row.
#include <math.h>

#include "internal.cuh"

namespace lsh {
namespace {

constexpr int kWarps = 8;
constexpr int kRowsInFlight = 8;

// A caller's inverse-permutation entry as a row index: entries outside [0, L) (a
// corrupt or foreign inv) are replaced by 0, so no read leaves the round's rows.
__device__ __forceinline__ int safe_row(int s, int L) { return (unsigned)s < (unsigned)L ? s : 0; }

template <int EPL>
__device__ __forceinline__ void load_row(const float *p, float (&x)[EPL]) {
    if constexpr (EPL == 4) {
        const float4 t = __ldg(reinterpret_cast<const float4 *>(p));
        x[0] = t.x; x[1] = t.y; x[2] = t.z; x[3] = t.w;
    } else {
        const float2 t = __ldg(reinterpret_cast<const float2 *>(p));
        x[0] = t.x; x[1] = t.y;
    }
}
template <int EPL>
__device__ __forceinline__ void load_row(const __nv_bfloat16 *p, float (&x)[EPL]) {
    if constexpr (EPL == 4) {
        const uint2 t = __ldg(reinterpret_cast<const uint2 *>(p));
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&t.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&t.y));
        x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
    } else {
        const uint32_t t = __ldg(reinterpret_cast<const unsigned int *>(p));
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&t));
        x[0] = a.x; x[1] = a.y;
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32)
combine_kernel(const T *__restrict__ o_r, const float *__restrict__ lse_r,
               const int32_t *__restrict__ inv, long n_tok, int L, int n_rounds,
               int token_order, float *__restrict__ out, float *__restrict__ lse)
{
    constexpr int EPL = D / 32;  // elements per lane, contiguous
    const int lane = threadIdx.x & 31;
    const long tok = (long)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (tok >= n_tok) return;
    const long bh = tok / L;
    const int i = (int)(tok % L);
    const size_t seg0 = (size_t)bh * n_rounds;

    // pass 1: lane r looks up round r (rounds beyond 32 are folded in 32 at a time)
    float mx = -INFINITY;
    for (int r0 = 0; r0 < n_rounds; r0 += 32) {
        const int r = r0 + lane;
        if (r < n_rounds) {
            const size_t base = (seg0 + r) * L;
            mx = fmaxf(mx, __ldg(lse_r + base + (token_order ? i : safe_row(__ldg(inv + base + i), L))));
        }
    }
    mx = warp_max(mx);
    float acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
    float sum = 0.f;
    for (int r0 = 0; r0 < n_rounds; r0 += 32) {
        const int r = r0 + lane;
        int s = 0;
        float w = 0.f;
        if (r < n_rounds) {
            const size_t base = (seg0 + r) * L;
            s = token_order ? i : safe_row(__ldg(inv + base + i), L);
            w = expf(__ldg(lse_r + base + s) - mx);
        }
        sum += warp_sum(w);
        const int nr = min(32, n_rounds - r0);
        // pass 2: rows of up to kRowsInFlight rounds requested before any is used
        for (int q0 = 0; q0 < nr; q0 += kRowsInFlight) {
            float x[kRowsInFlight][EPL];
            float wq[kRowsInFlight];
#pragma unroll
            for (int q = 0; q < kRowsInFlight; ++q) {
                const int rr = q0 + q;
                const int sq = __shfl_sync(0xffffffffu, s, rr & 31);
                wq[q] = __shfl_sync(0xffffffffu, w, rr & 31);
                if (rr < nr) {
                    load_row<EPL>(o_r + ((seg0 + r0 + rr) * L + sq) * D + lane * EPL, x[q]);
                } else {
                    wq[q] = 0.f;
#pragma unroll
                    for (int e = 0; e < EPL; ++e) x[q][e] = 0.f;
                }
            }
#pragma unroll
            for (int q = 0; q < kRowsInFlight; ++q)
#pragma unroll
                for (int e = 0; e < EPL; ++e) acc[e] = fmaf(wq[q], x[q][e], acc[e]);
        }
    }
    const float rs = 1.0f / sum;
    float *dst = out + (size_t)tok * D + lane * EPL;
    if constexpr (EPL == 4) {
        __stcs(reinterpret_cast<float4 *>(dst), make_float4(acc[0] * rs, acc[1] * rs, acc[2] * rs, acc[3] * rs));
    } else {
        __stcs(reinterpret_cast<float2 *>(dst), make_float2(acc[0] * rs, acc[1] * rs));
    }
    if (lane == 0) lse[tok] = mx + logf(sum);
}

// Token-order rows (the fused forward), up to kTokRounds rounds: nothing depends on the
// weights until the sum, so every round's row and log-normaliser is requested at once
// (one memory round trip per token), then the warp reduces.  Two tokens per warp keep
// more bytes in flight.
constexpr int kTokRounds = 8;
constexpr int kTokPerWarp = 2;

template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32)
combine_tok_kernel(const T *__restrict__ o_r, const float *__restrict__ lse_r, long n_tok, int L,
                   int n_rounds, float *__restrict__ out, float *__restrict__ lse)
{
    constexpr int EPL = D / 32;
    const int lane = threadIdx.x & 31;
    const long tok0 = ((long)blockIdx.x * kWarps + (threadIdx.x >> 5)) * kTokPerWarp;
    float x[kTokPerWarp][kTokRounds][EPL];
    float lr[kTokPerWarp];
#pragma unroll
    for (int u = 0; u < kTokPerWarp; ++u) {
        const long tok = tok0 + u;
        const bool ok = tok < n_tok;
        const long bh = ok ? tok / L : 0;
        const int i = ok ? (int)(tok % L) : 0;
        const size_t seg0 = (size_t)bh * n_rounds;
        lr[u] = ok && lane < n_rounds ? __ldg(lse_r + (seg0 + lane) * L + i) : -INFINITY;
#pragma unroll
        for (int r = 0; r < kTokRounds; ++r) {
            if (ok && r < n_rounds) {
                load_row<EPL>(o_r + ((seg0 + r) * L + i) * D + lane * EPL, x[u][r]);
            } else {
#pragma unroll
                for (int e = 0; e < EPL; ++e) x[u][r][e] = 0.f;
            }
        }
    }
#pragma unroll
    for (int u = 0; u < kTokPerWarp; ++u) {
        const long tok = tok0 + u;
        if (tok >= n_tok) break;
        const float mx = warp_max(lr[u]);
        const float w = lane < n_rounds ? expf(lr[u] - mx) : 0.f;
        const float sum = warp_sum(w);
        float acc[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
#pragma unroll
        for (int r = 0; r < kTokRounds; ++r) {
            const float wr = __shfl_sync(0xffffffffu, w, r);
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[e] = fmaf(wr, x[u][r][e], acc[e]);
        }
        const float rs = 1.0f / sum;
        float *dst = out + (size_t)tok * D + lane * EPL;
        if constexpr (EPL == 4) {
            __stcs(reinterpret_cast<float4 *>(dst), make_float4(acc[0] * rs, acc[1] * rs, acc[2] * rs, acc[3] * rs));
        } else {
            __stcs(reinterpret_cast<float2 *>(dst), make_float2(acc[0] * rs, acc[1] * rs));
        }
        if (lane == 0) lse[tok] = mx + logf(sum);
    }
}

template <typename T, int D>
cudaError_t launch(const Problem &p, const void *o_r, const float *lse_r, const int32_t *inv,
                   float *out, float *lse, cudaStream_t st)
{
    const long n = p.n_tok();
    if (p.token_order && p.n_rounds <= kTokRounds) {
        const long per_block = (long)kWarps * kTokPerWarp;
        const unsigned grid = (unsigned)((n + per_block - 1) / per_block);
        combine_tok_kernel<T, D><<<grid, kWarps * 32, 0, st>>>((const T *)o_r, lse_r, n, p.L,
                                                               p.n_rounds, out, lse);
        return cudaGetLastError();
    }
    const unsigned grid = (unsigned)((n + kWarps - 1) / kWarps);
    combine_kernel<T, D><<<grid, kWarps * 32, 0, st>>>((const T *)o_r, lse_r, inv, n, p.L,
                                                       p.n_rounds, p.token_order, out, lse);
    return cudaGetLastError();
}

}  // namespace

cudaError_t combine_launch(const Problem &p, const void *o_r, const float *lse_r,
                           const int32_t *inv, float *out, float *lse, cudaStream_t st,
                           StatusBlock *status)
{
    if (combine_tma_supported(p)) return combine_tma(p, o_r, lse_r, out, lse, status, st);
    if (p.dtype == LSH_F32)
        return p.d == 64 ? launch<float, 64>(p, o_r, lse_r, inv, out, lse, st)
                         : launch<float, 128>(p, o_r, lse_r, inv, out, lse, st);
    return p.d == 64 ? launch<__nv_bfloat16, 64>(p, o_r, lse_r, inv, out, lse, st)
                     : launch<__nv_bfloat16, 128>(p, o_r, lse_r, inv, out, lse, st);
}

}  // namespace lsh
