// internal.cuh -- shared declarations of the LSH-attention CUDA library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "lsh_attn.h"

namespace lsh {

// Logit given to a token's own key when it is the only key left (the "self only when
// nothing else exists" rule of the modulabs-hub notes, section "LSH attention").
constexpr float kSelfLogit = -1.0e5f;

// First 256 bytes of every workspace.  Kernels that wait on hardware barriers give up
// after a bounded time, record where in `detail`, and set `code` to 1.
struct StatusBlock {
    int code;
    int detail;
    int pad[62];
};
static_assert(sizeof(StatusBlock) == 256, "status block is 256 bytes");

// status-block detail written by the bounded-wait self test
constexpr int kSelftestWaitCode = 0xF01;

constexpr size_t kAlign = 1024;
inline size_t align_up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }

// Sort tile: keys per CTA of the counting-sort passes.
constexpr int kSortTile = 4096;
inline int sort_tiles(int L) { return (L + kSortTile - 1) / kSortTile; }
// dynamic shared memory the one-launch segment sort may use
constexpr size_t kSortSegSmemMax = 220 * 1024;

// Element loads widened to fp32.
__device__ __forceinline__ float ld_f32(const float *p, size_t i) { return p[i]; }
__device__ __forceinline__ float ld_f32(const __nv_bfloat16 *p, size_t i) {
    return __bfloat162float(p[i]);
}
__device__ __forceinline__ float ld_f32(const __half *p, size_t i) { return __half2float(p[i]); }
// 16-bit inputs (bf16 or fp16) keep their per-round rows in bf16.
inline bool is16(lsh_dtype_t t) { return t == LSH_BF16 || t == LSH_F16; }
__device__ __forceinline__ void st_elem(float *p, size_t i, float x) { p[i] = x; }
__device__ __forceinline__ void st_elem(__nv_bfloat16 *p, size_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Problem description passed to every launcher.
struct Problem {
    int B, H, L, d, nb, n_rounds, chunk, causal;
    float scale;
    lsh_dtype_t dtype;
    // Attention output rows (o_r, lse_r) at the token's original position instead of its
    // sorted index; the round combination then reads them without the inverse
    // permutation.  Internal to the fused forward.
    int token_order = 0;
    long n_tok() const { return (long)B * H * L; }
    long n_seg() const { return (long)B * H * n_rounds; }
};

// ---- launchers (each returns the launch error, if any) ----
cudaError_t hash_simt(const Problem &p, const void *qk, const void *R, int32_t *buckets,
                      float *inv_norm, cudaStream_t st);
// tensor-core hash: R is first packed into `rpack` (bytes from hash_tc_pack_bytes)
size_t hash_tc_pack_bytes(const Problem &p);
cudaError_t hash_tc(const Problem &p, const void *qk, const void *R, void *rpack,
                    int32_t *buckets, float *inv_norm, StatusBlock *status, cudaStream_t st);
bool hash_tc_supported(const Problem &p);
int hash_tc_launches(const Problem &p);

int sort_launches(const Problem &p);   // kernels one sort_launch call launches
cudaError_t sort_launch(const Problem &p, const int32_t *buckets, int32_t *perm, int32_t *inv,
                        int32_t *bstart, int32_t *counts, cudaStream_t st);

cudaError_t attn_simt(const Problem &p, const void *qk, const void *v, const int32_t *buckets,
                      const int32_t *perm, const int32_t *bstart, const float *inv_norm,
                      void *o_r, float *lse_r, cudaStream_t st);
// chunk 128 on the tensor cores (bf16 / fp16, d = 128, L a multiple of 128)
bool attn_c128_supported(const Problem &p);
cudaError_t attn_c128(const Problem &p, const void *qk, const void *v, const int32_t *buckets,
                      const int32_t *perm, const float *inv_norm, void *o_r, float *lse_r,
                      StatusBlock *status, cudaStream_t st);
bool attn_tc_supported(const Problem &p);
cudaError_t attn_tc(const Problem &p, const void *qk, const void *v, const int32_t *buckets,
                    const int32_t *perm, const int32_t *bstart, const float *inv_norm, void *o_r,
                    float *lse_r, StatusBlock *status, cudaStream_t st);

// backward of attention + combination; dqk and dv (fp32) are accumulated into
cudaError_t attn_bwd(const Problem &p, const void *qk, const void *v, const int32_t *buckets,
                     const int32_t *perm, const float *inv_norm, const float *out, const float *lse,
                     const float *g_out, const float *g_lse, float *dqk, float *dv, cudaStream_t st);
// bf16 inputs, d in {64, 128}, chunk in {32, 64}: the tensor-core backward, which needs
// attn_bwd_tc_scratch_bytes() of scratch (g_out in bf16 and g_out . out per token) and
// 16-byte aligned out, g_out, dqk and dv.
bool attn_bwd_tc_supported(const Problem &p);
size_t attn_bwd_tc_scratch_bytes(const Problem &p);
cudaError_t attn_bwd_tc(const Problem &p, const void *qk, const void *v, const int32_t *buckets,
                        const int32_t *perm, const float *inv_norm, const float *out,
                        const float *lse, const float *g_out, const float *g_lse, float *dqk,
                        float *dv, void *scratch, StatusBlock *status, cudaStream_t st);

cudaError_t selftest_wait_launch(StatusBlock *status, cudaStream_t st);

// Dense projection on the tensor cores: C = epilogue(A W^T), A [M][K], W [N][K] bf16.
// Epilogue: + bias[n] (optional), ReLU (optional), out = res + res_sign * x (optional
// residual, fp32 [M][N]); written to out_f32 [M][N] and/or out_bf16 ([M][N], or split into
// heads [M / split_L][N / split_d][split_L][split_d] when split_heads).
struct GemmArgs {
    const __nv_bfloat16 *A = nullptr, *W = nullptr;
    int M = 0, N = 0, K = 0;
    const float *bias = nullptr;
    int relu = 0;
    const float *res = nullptr;
    float res_sign = 1.f;
    float *out_f32 = nullptr;
    __nv_bfloat16 *out_bf16 = nullptr;
    int split_heads = 0, split_L = 1, split_d = 1;
};
bool gemm_tc_supported(int M, int N, int K);
cudaError_t gemm_tc(const GemmArgs &g, StatusBlock *status, cudaStream_t st);

// LSH k-nearest-neighbour search: per-round lists (cand_idx, cand_sim: [seg][L][k]), then
// the merged top k per token (nn_idx, nn_sim: [B][H][L][k])
cudaError_t knn_launch(const Problem &p, int k, const void *qk, const int32_t *buckets,
                       const int32_t *perm, const float *inv_norm, int32_t *cand_idx,
                       float *cand_sim, int32_t *nn_idx, float *nn_sim, cudaStream_t st);

cudaError_t combine_launch(const Problem &p, const void *o_r, const float *lse_r,
                           const int32_t *inv, float *out, float *lse, cudaStream_t st,
                           StatusBlock *status = nullptr);
// token-order rows, bf16, <= 8 rounds: the TMA-fed combination (status may be null)
bool combine_tma_supported(const Problem &p);
cudaError_t combine_tma(const Problem &p, const void *o_r, const float *lse_r, float *out,
                        float *lse, StatusBlock *status, cudaStream_t st);

}  // namespace lsh
