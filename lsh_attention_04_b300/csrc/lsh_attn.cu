// lsh_attn.cu -- the C ABI: argument validation, workspace layout and the launch
// sequence of the forward pass.  No allocation, no host synchronisation, no global state.
#include <string.h>

#include "internal.cuh"

using namespace lsh;

namespace {

bool nonpos(int x) { return x <= 0; }

// check_chunk = false for the hash stage, which does not depend on the chunk size.
lsh_status_t validate(const Problem &p, bool check_chunk = true)
{
    if (nonpos(p.B) || nonpos(p.H) || nonpos(p.L) || nonpos(p.d) || nonpos(p.nb) ||
        nonpos(p.n_rounds) || (check_chunk && nonpos(p.chunk)))
        return LSH_ERR_INVALID_ARGUMENT;
    if (p.dtype != LSH_F32 && !is16(p.dtype)) return LSH_ERR_INVALID_ARGUMENT;
    if (p.nb % 2 != 0) return LSH_ERR_INVALID_ARGUMENT;          // R has nb/2 columns
    if (check_chunk && p.L % p.chunk != 0) return LSH_ERR_INVALID_ARGUMENT;  // equal chunks
    if (p.causal != 0 && p.causal != 1) return LSH_ERR_INVALID_ARGUMENT;
    if (p.d != 64 && p.d != 128) return LSH_ERR_UNSUPPORTED;
    if (check_chunk && p.chunk != 32 && p.chunk != 64 && p.chunk != 128) return LSH_ERR_UNSUPPORTED;
    // chunk 128: the forward pass only, on the CUDA cores; fp32 rows at d = 128 do not fit
    if (check_chunk && p.chunk == 128 && p.d == 128 && p.dtype == LSH_F32) return LSH_ERR_UNSUPPORTED;
    if (p.nb > 2048) return LSH_ERR_UNSUPPORTED;
    if (is16(p.dtype) && p.nb % 16 != 0) return LSH_ERR_UNSUPPORTED;
    if ((long long)p.B * p.H * p.n_rounds * p.L >= (1LL << 31)) return LSH_ERR_UNSUPPORTED;
    return LSH_OK;
}

Problem make_problem(int B, int H, int L, int d, int nb, int n_rounds, int chunk, int causal,
                     float scale, lsh_dtype_t dtype)
{
    Problem p;
    p.B = B; p.H = H; p.L = L; p.d = d; p.nb = nb; p.n_rounds = n_rounds;
    p.chunk = chunk; p.causal = causal; p.scale = scale; p.dtype = dtype;
    return p;
}

size_t esize(lsh_dtype_t t) { return t == LSH_F32 ? 4 : 2; }

size_t rpack_bytes(const Problem &p) { return hash_tc_supported(p) ? hash_tc_pack_bytes(p) : 0; }
size_t counts_bytes(const Problem &p) { return sizeof(int32_t) * p.n_seg() * p.nb * sort_tiles(p.L); }

// Workspace of the whole forward pass; the backward pass uses the same layout without
// the per-round outputs (round_outputs = false).
struct Layout {
    size_t rpack, counts, buckets, inv_norm, perm, inv, bstart, o_r, lse_r, total;
};

Layout layout(const Problem &p, bool round_outputs = true)
{
    Layout w;
    size_t o = align_up(sizeof(StatusBlock));
    const size_t SL = (size_t)p.n_seg() * p.L;
    w.rpack = o;    o = align_up(o + rpack_bytes(p));
    w.counts = o;   o = align_up(o + counts_bytes(p));
    w.buckets = o;  o = align_up(o + sizeof(int32_t) * SL);
    w.inv_norm = o; o = align_up(o + sizeof(float) * p.n_tok());
    w.perm = o;     o = align_up(o + sizeof(int32_t) * SL);
    w.inv = o;      o = align_up(o + sizeof(int32_t) * SL);
    w.bstart = o;   o = align_up(o + sizeof(int32_t) * p.n_seg() * (p.nb + 1));
    w.o_r = o;      o = align_up(o + (round_outputs ? esize(p.dtype) * SL * p.d : 0));
    w.lse_r = o;    o = align_up(o + (round_outputs ? sizeof(float) * SL : 0));
    w.total = o;
    return w;
}

template <typename T> T *at(void *base, size_t off) { return (T *)((char *)base + off); }

lsh_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? LSH_OK : LSH_ERR_CUDA; }

lsh_status_t clear_status(void *ws, cudaStream_t st)
{
    return cuda_status(cudaMemsetAsync(ws, 0, sizeof(StatusBlock), st));
}

lsh_status_t run_hash(const Problem &p, const void *qk, const void *R, int32_t *buckets,
                      float *inv_norm, void *ws, void *rpack, cudaStream_t st)
{
    if (hash_tc_supported(p))
        return cuda_status(hash_tc(p, qk, R, rpack, buckets, inv_norm, (StatusBlock *)ws, st));
    return cuda_status(hash_simt(p, qk, R, buckets, inv_norm, st));
}

lsh_status_t run_attn(const Problem &p, const void *qk, const void *v, const int32_t *buckets,
                      const int32_t *perm, const int32_t *bstart, const float *inv_norm,
                      void *o_r, float *lse_r, void *ws, cudaStream_t st)
{
    if (attn_c128_supported(p))
        return cuda_status(attn_c128(p, qk, v, buckets, perm, inv_norm, o_r, lse_r,
                                     (StatusBlock *)ws, st));
    if (attn_tc_supported(p))
        return cuda_status(attn_tc(p, qk, v, buckets, perm, bstart, inv_norm, o_r, lse_r,
                                   (StatusBlock *)ws, st));
    return cuda_status(attn_simt(p, qk, v, buckets, perm, bstart, inv_norm, o_r, lse_r, st));
}

}  // namespace

extern "C" {

const char *lsh_status_string(lsh_status_t s)
{
    switch (s) {
    case LSH_OK: return "LSH_OK";
    case LSH_ERR_INVALID_ARGUMENT: return "LSH_ERR_INVALID_ARGUMENT";
    case LSH_ERR_UNSUPPORTED: return "LSH_ERR_UNSUPPORTED";
    case LSH_ERR_WORKSPACE_TOO_SMALL: return "LSH_ERR_WORKSPACE_TOO_SMALL";
    case LSH_ERR_CUDA: return "LSH_ERR_CUDA";
    case LSH_ERR_DEVICE_CHECK: return "LSH_ERR_DEVICE_CHECK";
    }
    return "LSH_ERR_UNKNOWN";
}

size_t lsh_attn_workspace_bytes(int B, int H, int L, int d, int n_buckets, int n_rounds,
                                int chunk, lsh_dtype_t dtype)
{
    const Problem p = make_problem(B, H, L, d, n_buckets, n_rounds, chunk, 0, 1.f, dtype);
    if (validate(p) != LSH_OK) return 0;
    return layout(p).total;
}

lsh_status_t lsh_attn_workspace_layout(int B, int H, int L, int d, int n_buckets, int n_rounds,
                                       int chunk, lsh_dtype_t dtype, size_t *off_buckets,
                                       size_t *off_inv_norm, size_t *off_perm, size_t *off_inv,
                                       size_t *off_bstart, size_t *off_o_r, size_t *off_lse_r)
{
    const Problem p = make_problem(B, H, L, d, n_buckets, n_rounds, chunk, 0, 1.f, dtype);
    const lsh_status_t s = validate(p);
    if (s != LSH_OK) return s;
    const Layout w = layout(p);
    if (off_buckets) *off_buckets = w.buckets;
    if (off_inv_norm) *off_inv_norm = w.inv_norm;
    if (off_perm) *off_perm = w.perm;
    if (off_inv) *off_inv = w.inv;
    if (off_bstart) *off_bstart = w.bstart;
    if (off_o_r) *off_o_r = w.o_r;
    if (off_lse_r) *off_lse_r = w.lse_r;
    return LSH_OK;
}

}  // extern "C"

namespace {

lsh_status_t record(void *const *events, int i, cudaStream_t st)
{
    if (!events) return LSH_OK;
    return cuda_status(cudaEventRecord((cudaEvent_t)events[i], st));
}

lsh_status_t forward(const void *qk, const void *v, const void *R, lsh_dtype_t dtype, int B,
                     int H, int L, int d, int n_buckets, int n_rounds, int chunk, int causal,
                     float scale, float *out, float *lse, void *workspace,
                     size_t workspace_bytes, void *stream, void *const *events)
{
    Problem p = make_problem(B, H, L, d, n_buckets, n_rounds, chunk, causal, scale, dtype);
    lsh_status_t s = validate(p);
    if (s != LSH_OK) return s;
    if (!qk || !v || !R || !out || !lse || !workspace) return LSH_ERR_INVALID_ARGUMENT;
    // attention writes each round's rows at the tokens' own positions, so the round
    // combination streams them (no inverse-permutation gather)
    p.token_order = 1;
    if (((uintptr_t)workspace) % 256 != 0) return LSH_ERR_INVALID_ARGUMENT;
    const Layout w = layout(p);
    if (workspace_bytes < w.total) return LSH_ERR_WORKSPACE_TOO_SMALL;
    cudaStream_t st = (cudaStream_t)stream;
    int32_t *buckets = at<int32_t>(workspace, w.buckets);
    float *inv_norm = at<float>(workspace, w.inv_norm);
    int32_t *perm = at<int32_t>(workspace, w.perm);
    int32_t *inv = at<int32_t>(workspace, w.inv);
    int32_t *bstart = at<int32_t>(workspace, w.bstart);
    void *o_r = at<void>(workspace, w.o_r);
    float *lse_r = at<float>(workspace, w.lse_r);

    if ((s = clear_status(workspace, st)) != LSH_OK) return s;
    if ((s = record(events, 0, st)) != LSH_OK) return s;
    if ((s = run_hash(p, qk, R, buckets, inv_norm, workspace, at<void>(workspace, w.rpack), st)) != LSH_OK)
        return s;
    if ((s = record(events, 1, st)) != LSH_OK) return s;
    if ((s = cuda_status(sort_launch(p, buckets, perm, inv, bstart, at<int32_t>(workspace, w.counts), st))) != LSH_OK)
        return s;
    if ((s = record(events, 2, st)) != LSH_OK) return s;
    if ((s = run_attn(p, qk, v, buckets, perm, bstart, inv_norm, o_r, lse_r, workspace, st)) != LSH_OK)
        return s;
    if ((s = record(events, 3, st)) != LSH_OK) return s;
    if ((s = cuda_status(combine_launch(p, o_r, lse_r, inv, out, lse, st, (StatusBlock *)workspace))) != LSH_OK)
        return s;
    return record(events, 4, st);
}

// Workspace of the backward pass: the forward's layout without per-round outputs, then
// the tensor-core kernel's scratch.
size_t backward_bytes(const Problem &p)
{
    return align_up(layout(p, false).total + attn_bwd_tc_scratch_bytes(p));
}

// The backward pass; `events`, when not null, are recorded before the hash, the sort and
// the backward kernel, and after it.
lsh_status_t backward(const void *qk, const void *v, const void *R, lsh_dtype_t dtype, int B,
                      int H, int L, int d, int n_buckets, int n_rounds, int chunk, int causal,
                      float scale, const float *out, const float *lse, const float *g_out,
                      const float *g_lse, float *dqk, float *dv, void *workspace,
                      size_t workspace_bytes, void *stream, void *const *events)
{
    const Problem p = make_problem(B, H, L, d, n_buckets, n_rounds, chunk, causal, scale, dtype);
    lsh_status_t s = validate(p);
    if (s != LSH_OK) return s;
    if (chunk == 128) return LSH_ERR_UNSUPPORTED;            // forward only
    if (!qk || !v || !R || !out || !lse || !g_out || !dqk || !dv || !workspace)
        return LSH_ERR_INVALID_ARGUMENT;
    if (((uintptr_t)workspace) % 256 != 0) return LSH_ERR_INVALID_ARGUMENT;
    const Layout w = layout(p, false);
    const bool tc = attn_bwd_tc_supported(p);
    if (tc) {
        const auto a16 = [](const void *x) { return ((uintptr_t)x) % 16 == 0; };
        if (!a16(qk) || !a16(v) || !a16(out) || !a16(g_out) || !a16(dqk) || !a16(dv))
            return LSH_ERR_INVALID_ARGUMENT;
    }
    if (workspace_bytes < backward_bytes(p)) return LSH_ERR_WORKSPACE_TOO_SMALL;
    cudaStream_t st = (cudaStream_t)stream;
    int32_t *buckets = at<int32_t>(workspace, w.buckets);
    float *inv_norm = at<float>(workspace, w.inv_norm);
    int32_t *perm = at<int32_t>(workspace, w.perm);
    const size_t grad_bytes = sizeof(float) * (size_t)p.n_tok() * p.d;
    if ((s = clear_status(workspace, st)) != LSH_OK) return s;
    if ((s = cuda_status(cudaMemsetAsync(dqk, 0, grad_bytes, st))) != LSH_OK) return s;
    if ((s = cuda_status(cudaMemsetAsync(dv, 0, grad_bytes, st))) != LSH_OK) return s;
    if ((s = record(events, 0, st)) != LSH_OK) return s;
    // the same deterministic kernels as the forward pass: the same buckets and order
    if ((s = run_hash(p, qk, R, buckets, inv_norm, workspace, at<void>(workspace, w.rpack), st)) != LSH_OK)
        return s;
    if ((s = record(events, 1, st)) != LSH_OK) return s;
    if ((s = cuda_status(sort_launch(p, buckets, perm, at<int32_t>(workspace, w.inv),
                                     at<int32_t>(workspace, w.bstart),
                                     at<int32_t>(workspace, w.counts), st))) != LSH_OK)
        return s;
    if ((s = record(events, 2, st)) != LSH_OK) return s;
    if (tc)
        s = cuda_status(attn_bwd_tc(p, qk, v, buckets, perm, inv_norm, out, lse, g_out, g_lse, dqk,
                                    dv, at<void>(workspace, w.total), (StatusBlock *)workspace, st));
    else
        s = cuda_status(attn_bwd(p, qk, v, buckets, perm, inv_norm, out, lse, g_out, g_lse, dqk,
                                 dv, st));
    if (s != LSH_OK) return s;
    return record(events, 3, st);
}

}  // namespace

extern "C" {

lsh_status_t lsh_attn_forward(const void *qk, const void *v, const void *R, lsh_dtype_t dtype,
                              int B, int H, int L, int d, int n_buckets, int n_rounds,
                              int chunk, int causal, float scale, float *out, float *lse,
                              void *workspace, size_t workspace_bytes, void *stream)
{
    return forward(qk, v, R, dtype, B, H, L, d, n_buckets, n_rounds, chunk, causal, scale, out,
                   lse, workspace, workspace_bytes, stream, nullptr);
}

lsh_status_t lsh_attn_forward_timed(const void *qk, const void *v, const void *R,
                                    lsh_dtype_t dtype, int B, int H, int L, int d,
                                    int n_buckets, int n_rounds, int chunk, int causal,
                                    float scale, float *out, float *lse, void *workspace,
                                    size_t workspace_bytes, void *stream,
                                    void *const *stage_events)
{
    if (!stage_events) return LSH_ERR_INVALID_ARGUMENT;
    for (int i = 0; i < 5; ++i)
        if (!stage_events[i]) return LSH_ERR_INVALID_ARGUMENT;
    return forward(qk, v, R, dtype, B, H, L, d, n_buckets, n_rounds, chunk, causal, scale, out,
                   lse, workspace, workspace_bytes, stream, stage_events);
}

size_t lsh_attn_backward_workspace_bytes(int B, int H, int L, int d, int n_buckets,
                                         int n_rounds, int chunk, lsh_dtype_t dtype)
{
    const Problem p = make_problem(B, H, L, d, n_buckets, n_rounds, chunk, 0, 1.f, dtype);
    if (validate(p) != LSH_OK || chunk == 128) return 0;
    return backward_bytes(p);
}

lsh_status_t lsh_attn_backward(const void *qk, const void *v, const void *R, lsh_dtype_t dtype,
                               int B, int H, int L, int d, int n_buckets, int n_rounds,
                               int chunk, int causal, float scale, const float *out,
                               const float *lse, const float *g_out, const float *g_lse,
                               float *dqk, float *dv, void *workspace, size_t workspace_bytes,
                               void *stream)
{
    return backward(qk, v, R, dtype, B, H, L, d, n_buckets, n_rounds, chunk, causal, scale, out,
                    lse, g_out, g_lse, dqk, dv, workspace, workspace_bytes, stream, nullptr);
}

lsh_status_t lsh_attn_backward_timed(const void *qk, const void *v, const void *R,
                                     lsh_dtype_t dtype, int B, int H, int L, int d,
                                     int n_buckets, int n_rounds, int chunk, int causal,
                                     float scale, const float *out, const float *lse,
                                     const float *g_out, const float *g_lse, float *dqk,
                                     float *dv, void *workspace, size_t workspace_bytes,
                                     void *stream, void *const *stage_events)
{
    if (!stage_events) return LSH_ERR_INVALID_ARGUMENT;
    for (int i = 0; i < 4; ++i)
        if (!stage_events[i]) return LSH_ERR_INVALID_ARGUMENT;
    return backward(qk, v, R, dtype, B, H, L, d, n_buckets, n_rounds, chunk, causal, scale, out,
                    lse, g_out, g_lse, dqk, dv, workspace, workspace_bytes, stream, stage_events);
}

int lsh_attn_kernel_launches(int B, int H, int L, int d, int n_buckets, int n_rounds, int chunk,
                             lsh_dtype_t dtype)
{
    const Problem p = make_problem(B, H, L, d, n_buckets, n_rounds, chunk, 0, 1.f, dtype);
    if (validate(p) != LSH_OK) return 0;
    const int hash = hash_tc_supported(p) ? hash_tc_launches(p) : 1;
    const int sort = sort_launches(p);
    const int attn = 1;
    const int combine = 1;
    return hash + sort + attn + combine;
}

size_t lsh_hash_workspace_bytes(int n_rounds, int d, int n_buckets, lsh_dtype_t dtype)
{
    const Problem p = make_problem(1, 1, 128, d, n_buckets, n_rounds, 0, 0, 1.f, dtype);
    if (validate(p, false) != LSH_OK) return 0;
    return align_up(sizeof(StatusBlock)) + align_up(rpack_bytes(p));
}

lsh_status_t lsh_hash(const void *qk, const void *R, lsh_dtype_t dtype, int B, int H, int L,
                      int d, int n_buckets, int n_rounds, int32_t *buckets, float *inv_norm,
                      void *workspace, size_t workspace_bytes, void *stream)
{
    const Problem p = make_problem(B, H, L, d, n_buckets, n_rounds, 0, 0, 1.f, dtype);
    lsh_status_t s = validate(p, false);
    if (s != LSH_OK) return s;
    if (!qk || !R || !buckets || !inv_norm || !workspace) return LSH_ERR_INVALID_ARGUMENT;
    if (((uintptr_t)workspace) % 256 != 0) return LSH_ERR_INVALID_ARGUMENT;
    if (workspace_bytes < lsh_hash_workspace_bytes(n_rounds, d, n_buckets, dtype))
        return LSH_ERR_WORKSPACE_TOO_SMALL;
    cudaStream_t st = (cudaStream_t)stream;
    if ((s = clear_status(workspace, st)) != LSH_OK) return s;
    return run_hash(p, qk, R, buckets, inv_norm, workspace,
                    at<void>(workspace, align_up(sizeof(StatusBlock))), st);
}

size_t lsh_bucket_sort_workspace_bytes(int B, int H, int L, int n_buckets, int n_rounds)
{
    if (B <= 0 || H <= 0 || L <= 0 || n_buckets <= 0 || n_rounds <= 0 || n_buckets > 2048) return 0;
    Problem p = make_problem(B, H, L, 64, n_buckets, n_rounds, 32, 0, 1.f, LSH_F32);
    return align_up(sizeof(StatusBlock)) + align_up(counts_bytes(p));
}

lsh_status_t lsh_bucket_sort(const int32_t *buckets, int B, int H, int L, int n_buckets,
                             int n_rounds, int32_t *perm, int32_t *inv, int32_t *bstart,
                             void *workspace, size_t workspace_bytes, void *stream)
{
    if (B <= 0 || H <= 0 || L <= 0 || n_buckets <= 0 || n_rounds <= 0) return LSH_ERR_INVALID_ARGUMENT;
    if (!buckets || !perm || !inv || !bstart || !workspace) return LSH_ERR_INVALID_ARGUMENT;
    if (((uintptr_t)workspace) % 256 != 0) return LSH_ERR_INVALID_ARGUMENT;
    if (n_buckets > 2048) return LSH_ERR_UNSUPPORTED;
    if ((long long)B * H * n_rounds * L >= (1LL << 31)) return LSH_ERR_UNSUPPORTED;
    if (workspace_bytes < lsh_bucket_sort_workspace_bytes(B, H, L, n_buckets, n_rounds))
        return LSH_ERR_WORKSPACE_TOO_SMALL;
    const Problem p = make_problem(B, H, L, 64, n_buckets, n_rounds, 32, 0, 1.f, LSH_F32);
    cudaStream_t st = (cudaStream_t)stream;
    lsh_status_t s = clear_status(workspace, st);
    if (s != LSH_OK) return s;
    return cuda_status(sort_launch(p, buckets, perm, inv, bstart,
                                   at<int32_t>(workspace, align_up(sizeof(StatusBlock))), st));
}

size_t lsh_chunk_attn_workspace_bytes(void) { return align_up(sizeof(StatusBlock)); }

lsh_status_t lsh_chunk_attn(const void *qk, const void *v, lsh_dtype_t dtype,
                            const int32_t *buckets, const int32_t *perm, const int32_t *bstart,
                            const float *inv_norm, int B, int H, int L, int d, int n_buckets,
                            int n_rounds, int chunk, int causal, float scale, void *o_r,
                            float *lse_r, void *workspace, size_t workspace_bytes,
                            void *stream)
{
    const Problem p = make_problem(B, H, L, d, n_buckets, n_rounds, chunk, causal, scale, dtype);
    lsh_status_t s = validate(p);
    if (s != LSH_OK) return s;
    if (!qk || !v || !buckets || !perm || !bstart || !inv_norm || !o_r || !lse_r || !workspace)
        return LSH_ERR_INVALID_ARGUMENT;
    if (((uintptr_t)workspace) % 256 != 0) return LSH_ERR_INVALID_ARGUMENT;
    if (workspace_bytes < lsh_chunk_attn_workspace_bytes()) return LSH_ERR_WORKSPACE_TOO_SMALL;
    cudaStream_t st = (cudaStream_t)stream;
    if ((s = clear_status(workspace, st)) != LSH_OK) return s;
    return run_attn(p, qk, v, buckets, perm, bstart, inv_norm, o_r, lse_r, workspace, st);
}

lsh_status_t lsh_unsort_combine(const void *o_r, const float *lse_r, const int32_t *inv,
                                lsh_dtype_t dtype, int B, int H, int L, int d, int n_rounds,
                                float *out, float *lse, void *stream)
{
    if (B <= 0 || H <= 0 || L <= 0 || n_rounds <= 0) return LSH_ERR_INVALID_ARGUMENT;
    if (dtype != LSH_F32 && !is16(dtype)) return LSH_ERR_INVALID_ARGUMENT;
    if (!o_r || !lse_r || !inv || !out || !lse) return LSH_ERR_INVALID_ARGUMENT;
    if (d != 64 && d != 128) return LSH_ERR_UNSUPPORTED;
    if ((long long)B * H * n_rounds * L >= (1LL << 31)) return LSH_ERR_UNSUPPORTED;
    const Problem p = make_problem(B, H, L, d, 2, n_rounds, 32, 0, 1.f, dtype);
    return cuda_status(combine_launch(p, o_r, lse_r, inv, out, lse, (cudaStream_t)stream));
}

}  // extern "C"

namespace {

// Workspace of the k-nearest-neighbour search: the backward pass's (hash and sort
// outputs, no per-round attention outputs) followed by the per-round candidate lists.
struct KnnLayout {
    Layout base;
    size_t cand_idx, cand_sim, total;
};

bool knn_k_ok(int n_rounds, int k) { return k >= 1 && k <= 32 && (long)n_rounds * k <= 256; }

KnnLayout knn_layout(const Problem &p, int k)
{
    KnnLayout w;
    w.base = layout(p, false);
    const size_t n = (size_t)p.n_seg() * p.L * k;
    size_t o = w.base.total;
    w.cand_idx = o; o = align_up(o + sizeof(int32_t) * n);
    w.cand_sim = o; o = align_up(o + sizeof(float) * n);
    w.total = o;
    return w;
}

}  // namespace

extern "C" {

size_t lsh_knn_workspace_bytes(int B, int H, int L, int d, int n_buckets, int n_rounds, int chunk,
                               int k, lsh_dtype_t dtype)
{
    const Problem p = make_problem(B, H, L, d, n_buckets, n_rounds, chunk, 0, 1.f, dtype);
    if (validate(p) != LSH_OK || !knn_k_ok(n_rounds, k) || dtype == LSH_F16 || chunk == 128) return 0;
    return knn_layout(p, k).total;
}

lsh_status_t lsh_knn(const void *qk, const void *R, lsh_dtype_t dtype, int B, int H, int L, int d,
                     int n_buckets, int n_rounds, int chunk, int k, int32_t *nn_idx, float *nn_sim,
                     void *workspace, size_t workspace_bytes, void *stream)
{
    const Problem p = make_problem(B, H, L, d, n_buckets, n_rounds, chunk, 0, 1.f, dtype);
    lsh_status_t s = validate(p);
    if (s != LSH_OK) return s;
    if (dtype == LSH_F16 || chunk == 128) return LSH_ERR_UNSUPPORTED;   // bf16 / fp32, window <= 128
    if (!knn_k_ok(n_rounds, k)) return LSH_ERR_INVALID_ARGUMENT;
    if (!qk || !R || !nn_idx || !nn_sim || !workspace) return LSH_ERR_INVALID_ARGUMENT;
    if (((uintptr_t)workspace) % 256 != 0) return LSH_ERR_INVALID_ARGUMENT;
    const KnnLayout w = knn_layout(p, k);
    if (workspace_bytes < w.total) return LSH_ERR_WORKSPACE_TOO_SMALL;
    cudaStream_t st = (cudaStream_t)stream;
    int32_t *buckets = at<int32_t>(workspace, w.base.buckets);
    float *inv_norm = at<float>(workspace, w.base.inv_norm);
    int32_t *perm = at<int32_t>(workspace, w.base.perm);
    if ((s = clear_status(workspace, st)) != LSH_OK) return s;
    if ((s = run_hash(p, qk, R, buckets, inv_norm, workspace, at<void>(workspace, w.base.rpack), st)) != LSH_OK)
        return s;
    if ((s = cuda_status(sort_launch(p, buckets, perm, at<int32_t>(workspace, w.base.inv),
                                     at<int32_t>(workspace, w.base.bstart),
                                     at<int32_t>(workspace, w.base.counts), st))) != LSH_OK)
        return s;
    return cuda_status(knn_launch(p, k, qk, buckets, perm, inv_norm, at<int32_t>(workspace, w.cand_idx),
                                  at<float>(workspace, w.cand_sim), nn_idx, nn_sim, st));
}

lsh_status_t lsh_selftest_wait_timeout(void *workspace, size_t workspace_bytes, void *stream)
{
    if (!workspace || workspace_bytes < sizeof(StatusBlock)) return LSH_ERR_INVALID_ARGUMENT;
    if (((uintptr_t)workspace) % 256 != 0) return LSH_ERR_INVALID_ARGUMENT;
    cudaStream_t st = (cudaStream_t)stream;
    lsh_status_t s = clear_status(workspace, st);
    if (s != LSH_OK) return s;
    return cuda_status(selftest_wait_launch((StatusBlock *)workspace, st));
}

lsh_status_t lsh_workspace_status(const void *workspace, int *detail, void *stream)
{
    if (!workspace) return LSH_ERR_INVALID_ARGUMENT;
    StatusBlock h;
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return LSH_ERR_CUDA;
    e = cudaMemcpy(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return LSH_ERR_CUDA;
    if (detail) *detail = h.detail;
    return h.code == 0 ? LSH_OK : LSH_ERR_DEVICE_CHECK;
}

}  // extern "C"
