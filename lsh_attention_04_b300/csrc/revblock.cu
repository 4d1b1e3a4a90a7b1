// revblock.cu -- the reversible residual block around the LSH attention, forward and
// inverse, on random weights supplied by the caller.
//
// ai-scholar.tech Reformer article, sections "什么是可逆残余层？" and "RevNet 中的反向传播";
// "Reformer" glossary (ultralytics.com, es), section "Capas reversibles y división en
// fragmentos"; modulabs-hub notes, "Reversible Transformer" and "Chunking":
//     y1 = x1 + Attention(x2),        y2 = x2 + FeedForward(y1)
//     x2 = y2 - FeedForward(y1),      x1 = y1 - Attention(x2)
// Attention(x) = LSHAttention(x Wqk^T, x Wv^T) Wo^T over one shared query/key projection,
// heads split from and merged back into the model dimension; FeedForward(y) =
// relu(y W1^T + b1) W2^T + b2, run over chunks of positions so the hidden activations of
// only one chunk exist at a time.
// The residual stream (x1, x2, y1, y2) is fp32.  Matrix products take bf16 copies of their
// inputs (the activation entering a projection, the per-head projections, the merged
// attention output and the hidden layer) and accumulate in fp32 on the tensor cores
// (gemm_tc.cu); the attention is lsh_attn_forward itself.
#include <string.h>

#include "internal.cuh"

namespace lsh {
namespace {

__global__ void f32_to_bf16_kernel(const float *__restrict__ x, __nv_bfloat16 *__restrict__ y, long n4)
{
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n4; i += (long)gridDim.x * blockDim.x) {
        const float4 v = reinterpret_cast<const float4 *>(x)[i];
        __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
        uint2 o;
        o.x = *reinterpret_cast<uint32_t *>(&a);
        o.y = *reinterpret_cast<uint32_t *>(&b);
        reinterpret_cast<uint2 *>(y)[i] = o;
    }
}

// [B][H][L][d] fp32 -> [B*L][H*d] bf16
__global__ void merge_heads_kernel(const float *__restrict__ x, __nv_bfloat16 *__restrict__ y, int H,
                                   int L, int d, long n4)
{
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n4; i += (long)gridDim.x * blockDim.x) {
        const long e = i * 4;                     // element of the output, row-major [B*L][H*d]
        const long row = e / ((long)H * d);
        const int col = (int)(e % ((long)H * d));
        const long b = row / L, l = row % L;
        const int h = col / d, c = col % d;
        const float4 v = *reinterpret_cast<const float4 *>(x + (((b * H + h) * L + l) * d + c));
        __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), bb = __floats2bfloat162_rn(v.z, v.w);
        uint2 o;
        o.x = *reinterpret_cast<uint32_t *>(&a);
        o.y = *reinterpret_cast<uint32_t *>(&bb);
        reinterpret_cast<uint2 *>(y)[i] = o;
    }
}

// Keep the first failure: copy the attention's status block into the block's, unless the
// block's already records one.
__global__ void status_merge_kernel(StatusBlock *dst, const StatusBlock *src)
{
    if (threadIdx.x == 0 && dst->code == 0 && src->code != 0) {
        dst->code = src->code;
        dst->detail = src->detail;
    }
}

unsigned grid_for(long n) { return (unsigned)(n < 148L * 16 * 256 ? (n + 255) / 256 : 148L * 16); }

struct RevShape {
    int B, L, dm, H, d, dff, nb, R, chunk, causal, ff_chunk;
    float scale;
    long M() const { return (long)B * L; }
};

struct RevLayout {
    size_t attn_ws, attn_ws_bytes, qk, v, attn_out, lse, act16, merged, hidden, total;
};

bool rev_valid(const RevShape &s)
{
    if (s.B <= 0 || s.L <= 0 || s.dm <= 0 || s.H <= 0 || s.dff <= 0 || s.ff_chunk <= 0) return false;
    if (s.dm % s.H != 0) return false;
    if (s.dm % 128 != 0 || s.dff % 128 != 0) return false;          // 128-wide output tiles
    if ((long)s.B * s.L * s.dm >= (1L << 31) || (long)s.ff_chunk * s.dff >= (1L << 31)) return false;
    return lsh_attn_workspace_bytes(s.B, s.H, s.L, s.d, s.nb, s.R, s.chunk, LSH_BF16) > 0;
}

RevLayout rev_layout(const RevShape &s)
{
    RevLayout w;
    size_t o = align_up(sizeof(StatusBlock));
    const size_t n_hd = (size_t)s.B * s.H * s.L * s.d;
    w.attn_ws = o;
    w.attn_ws_bytes = lsh_attn_workspace_bytes(s.B, s.H, s.L, s.d, s.nb, s.R, s.chunk, LSH_BF16);
    o = align_up(o + w.attn_ws_bytes);
    w.qk = o;       o = align_up(o + 2 * n_hd);
    w.v = o;        o = align_up(o + 2 * n_hd);
    w.attn_out = o; o = align_up(o + 4 * n_hd);
    w.lse = o;      o = align_up(o + 4 * (size_t)s.B * s.H * s.L);
    w.act16 = o;    o = align_up(o + 2 * (size_t)s.M() * s.dm);
    w.merged = o;   o = align_up(o + 2 * (size_t)s.M() * s.dm);
    w.hidden = o;   o = align_up(o + 2 * (size_t)s.ff_chunk * s.dff);
    w.total = o;
    return w;
}

template <typename T> T *at(void *base, size_t off) { return (T *)((char *)base + off); }

struct RevWeights {
    const __nv_bfloat16 *Wqk, *Wv, *Wo, *W1, *W2, *R;
    const float *b1, *b2;
};

// out = x_res + sign * Attention(x) (x fp32 [M][dm])
cudaError_t attention_residual(const RevShape &s, const RevWeights &w, const float *x,
                               const float *res, float sign, float *out, void *ws,
                               const RevLayout &lay, cudaStream_t st)
{
    StatusBlock *status = (StatusBlock *)ws;
    const long M = s.M();
    __nv_bfloat16 *x16 = at<__nv_bfloat16>(ws, lay.act16);
    f32_to_bf16_kernel<<<grid_for(M * s.dm / 4), 256, 0, st>>>(x, x16, M * s.dm / 4);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    GemmArgs g;
    g.A = x16; g.M = (int)M; g.N = s.dm; g.K = s.dm;
    g.split_heads = 1; g.split_L = s.L; g.split_d = s.d;
    g.W = w.Wqk; g.out_bf16 = at<__nv_bfloat16>(ws, lay.qk);
    if ((e = gemm_tc(g, status, st)) != cudaSuccess) return e;
    g.W = w.Wv; g.out_bf16 = at<__nv_bfloat16>(ws, lay.v);
    if ((e = gemm_tc(g, status, st)) != cudaSuccess) return e;
    void *aws = at<void>(ws, lay.attn_ws);
    const lsh_status_t a = lsh_attn_forward(at<void>(ws, lay.qk), at<void>(ws, lay.v), w.R, LSH_BF16,
                                            s.B, s.H, s.L, s.d, s.nb, s.R, s.chunk, s.causal, s.scale,
                                            at<float>(ws, lay.attn_out), at<float>(ws, lay.lse), aws,
                                            lay.attn_ws_bytes, st);
    if (a != LSH_OK) return a == LSH_ERR_CUDA ? cudaErrorLaunchFailure : cudaErrorInvalidValue;
    status_merge_kernel<<<1, 32, 0, st>>>(status, (const StatusBlock *)aws);
    __nv_bfloat16 *merged = at<__nv_bfloat16>(ws, lay.merged);
    merge_heads_kernel<<<grid_for(M * s.dm / 4), 256, 0, st>>>(at<float>(ws, lay.attn_out), merged,
                                                                s.H, s.L, s.d, M * s.dm / 4);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    GemmArgs o;
    o.A = merged; o.W = w.Wo; o.M = (int)M; o.N = s.dm; o.K = s.dm;
    o.res = res; o.res_sign = sign; o.out_f32 = out;
    return gemm_tc(o, status, st);
}

// out = res + sign * FeedForward(y), chunks of ff_chunk positions (rows of [M][dm])
cudaError_t feed_forward_residual(const RevShape &s, const RevWeights &w, const float *y,
                                  const float *res, float sign, float *out, void *ws,
                                  const RevLayout &lay, cudaStream_t st)
{
    StatusBlock *status = (StatusBlock *)ws;
    const long M = s.M();
    __nv_bfloat16 *y16 = at<__nv_bfloat16>(ws, lay.act16);
    __nv_bfloat16 *hid = at<__nv_bfloat16>(ws, lay.hidden);
    f32_to_bf16_kernel<<<grid_for(M * s.dm / 4), 256, 0, st>>>(y, y16, M * s.dm / 4);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    for (long c0 = 0; c0 < M; c0 += s.ff_chunk) {
        const int cm = (int)(M - c0 < s.ff_chunk ? M - c0 : s.ff_chunk);
        GemmArgs h;
        h.A = y16 + c0 * s.dm; h.W = w.W1; h.M = cm; h.N = s.dff; h.K = s.dm;
        h.bias = w.b1; h.relu = 1; h.out_bf16 = hid;
        if ((e = gemm_tc(h, status, st)) != cudaSuccess) return e;
        GemmArgs o;
        o.A = hid; o.W = w.W2; o.M = cm; o.N = s.dm; o.K = s.dff;
        o.bias = w.b2; o.res = res + c0 * s.dm; o.res_sign = sign; o.out_f32 = out + c0 * s.dm;
        if ((e = gemm_tc(o, status, st)) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace
}  // namespace lsh

using namespace lsh;

namespace {

RevShape make_rev(int B, int L, int d_model, int heads, int d_ff, int nb, int n_rounds, int chunk,
                  int causal, float scale, int ff_chunk)
{
    RevShape s;
    s.B = B; s.L = L; s.dm = d_model; s.H = heads; s.d = heads > 0 ? d_model / heads : 0;
    s.dff = d_ff; s.nb = nb; s.R = n_rounds; s.chunk = chunk; s.causal = causal; s.scale = scale;
    s.ff_chunk = ff_chunk;
    return s;
}

lsh_status_t rev_common(const RevShape &s, const void *ptrs[], int n_ptrs, void *ws, size_t ws_bytes,
                        RevLayout &lay)
{
    if (!rev_valid(s) || (s.causal != 0 && s.causal != 1)) return LSH_ERR_INVALID_ARGUMENT;
    // every array is read with 16-byte vectors or by TMA; the four residual-stream arrays
    // (the last two pointers are the outputs) must be distinct
    for (int i = 0; i < n_ptrs; ++i)
        if (!ptrs[i] || ((uintptr_t)ptrs[i]) % 16 != 0) return LSH_ERR_INVALID_ARGUMENT;
    const void *stream4[] = {ptrs[0], ptrs[1], ptrs[n_ptrs - 2], ptrs[n_ptrs - 1]};
    for (int i = 0; i < 4; ++i)
        for (int j = i + 1; j < 4; ++j)
            if (stream4[i] == stream4[j]) return LSH_ERR_INVALID_ARGUMENT;
    if (!ws || ((uintptr_t)ws) % 256 != 0) return LSH_ERR_INVALID_ARGUMENT;
    lay = rev_layout(s);
    if (ws_bytes < lay.total) return LSH_ERR_WORKSPACE_TOO_SMALL;
    return LSH_OK;
}

lsh_status_t cuda_st(cudaError_t e) { return e == cudaSuccess ? LSH_OK : LSH_ERR_CUDA; }

}  // namespace

extern "C" {

size_t lsh_revblock_workspace_bytes(int B, int L, int d_model, int heads, int d_ff, int n_buckets,
                                    int n_rounds, int chunk, int ff_chunk)
{
    const RevShape s = make_rev(B, L, d_model, heads, d_ff, n_buckets, n_rounds, chunk, 0, 1.f, ff_chunk);
    return rev_valid(s) ? rev_layout(s).total : 0;
}

lsh_status_t lsh_revblock_workspace_layout(int B, int L, int d_model, int heads, int d_ff,
                                           int n_buckets, int n_rounds, int chunk, int ff_chunk,
                                           size_t *off_attn_ws, size_t *off_qk, size_t *off_v,
                                           size_t *off_attn_out, size_t *off_merged)
{
    const RevShape s = make_rev(B, L, d_model, heads, d_ff, n_buckets, n_rounds, chunk, 0, 1.f, ff_chunk);
    if (!rev_valid(s)) return LSH_ERR_INVALID_ARGUMENT;
    const RevLayout w = rev_layout(s);
    if (off_attn_ws) *off_attn_ws = w.attn_ws;
    if (off_qk) *off_qk = w.qk;
    if (off_v) *off_v = w.v;
    if (off_attn_out) *off_attn_out = w.attn_out;
    if (off_merged) *off_merged = w.merged;
    return LSH_OK;
}

lsh_status_t lsh_revblock_forward(const float *x1, const float *x2, const void *Wqk, const void *Wv,
                                  const void *Wo, const void *W1, const float *b1, const void *W2,
                                  const float *b2, const void *R, int B, int L, int d_model,
                                  int heads, int d_ff, int n_buckets, int n_rounds, int chunk,
                                  int causal, float scale, int ff_chunk, float *y1, float *y2,
                                  void *workspace, size_t workspace_bytes, void *stream)
{
    const RevShape s = make_rev(B, L, d_model, heads, d_ff, n_buckets, n_rounds, chunk, causal, scale, ff_chunk);
    const void *ptrs[] = {x1, x2, Wqk, Wv, Wo, W1, b1, W2, b2, R, y1, y2};
    RevLayout lay;
    lsh_status_t st = rev_common(s, ptrs, 12, workspace, workspace_bytes, lay);
    if (st != LSH_OK) return st;
    const RevWeights w = {(const __nv_bfloat16 *)Wqk, (const __nv_bfloat16 *)Wv, (const __nv_bfloat16 *)Wo,
                          (const __nv_bfloat16 *)W1, (const __nv_bfloat16 *)W2, (const __nv_bfloat16 *)R,
                          b1, b2};
    cudaStream_t cs = (cudaStream_t)stream;
    if ((st = cuda_st(cudaMemsetAsync(workspace, 0, sizeof(StatusBlock), cs))) != LSH_OK) return st;
    if ((st = cuda_st(attention_residual(s, w, x2, x1, 1.f, y1, workspace, lay, cs))) != LSH_OK) return st;
    return cuda_st(feed_forward_residual(s, w, y1, x2, 1.f, y2, workspace, lay, cs));
}

lsh_status_t lsh_revblock_inverse(const float *y1, const float *y2, const void *Wqk, const void *Wv,
                                  const void *Wo, const void *W1, const float *b1, const void *W2,
                                  const float *b2, const void *R, int B, int L, int d_model,
                                  int heads, int d_ff, int n_buckets, int n_rounds, int chunk,
                                  int causal, float scale, int ff_chunk, float *x1, float *x2,
                                  void *workspace, size_t workspace_bytes, void *stream)
{
    const RevShape s = make_rev(B, L, d_model, heads, d_ff, n_buckets, n_rounds, chunk, causal, scale, ff_chunk);
    const void *ptrs[] = {y1, y2, Wqk, Wv, Wo, W1, b1, W2, b2, R, x1, x2};
    RevLayout lay;
    lsh_status_t st = rev_common(s, ptrs, 12, workspace, workspace_bytes, lay);
    if (st != LSH_OK) return st;
    const RevWeights w = {(const __nv_bfloat16 *)Wqk, (const __nv_bfloat16 *)Wv, (const __nv_bfloat16 *)Wo,
                          (const __nv_bfloat16 *)W1, (const __nv_bfloat16 *)W2, (const __nv_bfloat16 *)R,
                          b1, b2};
    cudaStream_t cs = (cudaStream_t)stream;
    if ((st = cuda_st(cudaMemsetAsync(workspace, 0, sizeof(StatusBlock), cs))) != LSH_OK) return st;
    if ((st = cuda_st(feed_forward_residual(s, w, y1, y2, -1.f, x2, workspace, lay, cs))) != LSH_OK) return st;
    return cuda_st(attention_residual(s, w, x2, y1, -1.f, x1, workspace, lay, cs));
}

}  // extern "C"
