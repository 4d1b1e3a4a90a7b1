/*
 * lsh_attn.h -- C ABI of the B300 (sm_103a) multi-round LSH attention: the forward pass
 * and its backward pass.
 *
 * The method is Reformer's LSH attention over a shared query/key projection
 * (Kitaev, Kaiser & Levskaya, "Reformer: The Efficient Transformer", ICLR 2020), as
 * described by the "Reformer" glossary entry of ultralytics.com, section "Atencion
 * LSH", and the modulabs-hub Reformer notes, sections "Locality sensitive hashing",
 * "LSH attention" and "Multi-round LSH attention":
 *
 *   1. hash     bucket = argmax([xR_r, -xR_r]) for every token and round r;
 *   2. sort     order the tokens of each (batch, head, round) by (bucket, position);
 *   3. chunk    cut the sorted sequence into equal chunks of `chunk` tokens;
 *   4. attend   every token attends to its own chunk and the previous one, only to
 *               keys of its own bucket, only to earlier positions when causal, and to
 *               itself only when no other key is left;
 *   5. un-sort  move each round's result back to the original order;
 *   6. combine  weight the rounds by exp(lse_r - logsumexp_r lse_r).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every array pointer is DEVICE memory owned by the caller.  The library never
 *    allocates or frees memory and keeps no global state; calls on different
 *    streams with different buffers are independent.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and never synchronise the host.  The return code reports argument
 *    validation and launch errors only; faults inside a kernel surface at the
 *    caller's next synchronisation.
 *  - Layouts are dense, row-major:
 *        qk, v     [B][H][L][d]        element type `dtype`
 *        R         [n_rounds][d][n_buckets/2]   element type `dtype`, shared by all (b, h)
 *        buckets   int32 [B][H][n_rounds][L]
 *        inv_norm  fp32  [B][H][L]     1/|qk_j| (0 for a zero row)
 *        perm      int32 [B][H][n_rounds][L]   sorted index -> original position
 *        inv       int32 [B][H][n_rounds][L]   original position -> sorted index
 *        bstart    int32 [B][H][n_rounds][n_buckets+1]  first sorted index of each
 *                  bucket; bstart[n_buckets] = L
 *        o_r       [B][H][n_rounds][L][d] in SORTED order; bf16 when dtype is
 *                  LSH_BF16 or LSH_F16, fp32 when dtype is LSH_F32
 *        lse_r     fp32 [B][H][n_rounds][L] in sorted order (natural log)
 *        out       fp32 [B][H][L][d];  lse fp32 [B][H][L]
 *  - Keys are L2-normalised and queries are not: the score of query i and key j is
 *    scale * (qk_i . qk_j) / |qk_j|.  The usual choice is scale = 1/sqrt(d).
 *  - A token with no key left gets o = v_i and lse_r = -1e5 for that round, so the
 *    round combination gives that round a weight of about exp(-1e5) unless every
 *    round is like that.  This assumes |scale * |qk|| is far below 1e5.
 *  - Results for NaN or Inf inputs are undefined.
 *  - Workspaces are device buffers of at least the size the matching
 *    *_workspace_bytes() call returns, 256-byte aligned.  Their first 256 bytes hold
 *    a status block that kernels with bounded waits write when a wait gives up;
 *    lsh_workspace_status() reads it.
 */
#ifndef LSH_ATTN_H
#define LSH_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LSH_OK = 0,
    LSH_ERR_INVALID_ARGUMENT = 1,  /* null pointer, non-positive size, L % chunk != 0, odd n_buckets */
    LSH_ERR_UNSUPPORTED = 2,       /* valid but outside what the kernels implement (see below) */
    LSH_ERR_WORKSPACE_TOO_SMALL = 3,
    LSH_ERR_CUDA = 4,              /* a CUDA runtime call or kernel launch failed */
    LSH_ERR_DEVICE_CHECK = 5       /* a kernel gave up a bounded wait (from lsh_workspace_status) */
} lsh_status_t;

typedef enum {
    LSH_F32 = 0,   /* fp32 inputs; CUDA-core arithmetic in fp32 */
    LSH_BF16 = 1,  /* bf16 inputs; tensor-core products with fp32 accumulation */
    LSH_F16 = 2    /* fp16 inputs; as LSH_BF16 with fp16 operands (the softmax weights are
                      packed to fp16 for P V, and rows whose score bound exceeds 7 in log2
                      units take the exact row maximum, so the weights that matter stay
                      normal fp16 numbers, >= 2^-14); per-round rows (o_r) are bf16 as for
                      LSH_BF16.  Not taken by lsh_knn (LSH_ERR_UNSUPPORTED); the backward
                      pass runs it on the CUDA cores in fp32. */
} lsh_dtype_t;

/*
 * Supported range (anything else returns LSH_ERR_UNSUPPORTED):
 *   d in {64, 128};  chunk in {32, 64, 128};  2 <= n_buckets <= 2048;
 *   chunk 128: the forward pass and the staged steps only (lsh_attn_backward and lsh_knn
 *   return LSH_ERR_UNSUPPORTED); on the tensor cores for 16-bit inputs at d = 128 with
 *   L % 128 == 0, on the CUDA cores otherwise, and not for LSH_F32 at d = 128;
 *   n_buckets % 16 == 0 for LSH_BF16 and LSH_F16;  B*H*n_rounds*L < 2^31.
 */

/* Human-readable name of a status code (static storage). */
const char *lsh_status_string(lsh_status_t status);

/*
 * Bytes of device workspace lsh_attn_forward needs for this problem (0 when the
 * arguments are invalid or unsupported).
 */
size_t lsh_attn_workspace_bytes(int B, int H, int L, int d, int n_buckets, int n_rounds,
                                int chunk, lsh_dtype_t dtype);

/*
 * The whole forward pass: steps 1-6 above, on `stream`, through the caller's
 * workspace (which then holds buckets, perm, inv, bstart, o_r and lse_r; see
 * lsh_attn_workspace_layout).  Inside this call the attention step writes o_r and
 * lse_r in TOKEN order (round r's row of token i at position i, not at its sorted
 * index), so the round combination reads them as a stream; lsh_chunk_attn alone
 * keeps the sorted order documented above.
 *   qk, v     [B][H][L][d] dtype;  R [n_rounds][d][n_buckets/2] dtype
 *   causal    0 or 1;  scale  multiplies every score (see conventions)
 *   out       fp32 [B][H][L][d];  lse  fp32 [B][H][L]: logsumexp over rounds of lse_r
 * out and lse must not alias the inputs or the workspace.
 */
lsh_status_t lsh_attn_forward(const void *qk, const void *v, const void *R, lsh_dtype_t dtype,
                              int B, int H, int L, int d, int n_buckets, int n_rounds,
                              int chunk, int causal, float scale, float *out, float *lse,
                              void *workspace, size_t workspace_bytes, void *stream);

/*
 * lsh_attn_forward that also records five caller-created CUDA events (cudaEvent_t) on
 * `stream` at the stage boundaries: stage_events[0] before the hash, [1] before the
 * sort, [2] before the attention, [3] before the combination and [4] after it.  For
 * timing each kernel inside the real call.  A NULL array or event is
 * LSH_ERR_INVALID_ARGUMENT.
 */
lsh_status_t lsh_attn_forward_timed(const void *qk, const void *v, const void *R,
                                    lsh_dtype_t dtype, int B, int H, int L, int d,
                                    int n_buckets, int n_rounds, int chunk, int causal,
                                    float scale, float *out, float *lse, void *workspace,
                                    size_t workspace_bytes, void *stream,
                                    void *const *stage_events);

/*
 * Bytes of device workspace lsh_attn_backward needs (0 when the arguments are invalid
 * or unsupported): the forward's without per-round outputs, plus, for LSH_BF16, g_out in
 * bf16 and one fp32 per token.
 */
size_t lsh_attn_backward_workspace_bytes(int B, int H, int L, int d, int n_buckets,
                                         int n_rounds, int chunk, lsh_dtype_t dtype);

/*
 * Backward pass: the gradients in qk and v of the loss
 *     sum(g_out * out) + sum(g_lse * lse)
 * of the lsh_attn_forward call with the same arguments.  The Reformer pages train the
 * model by back-propagation (modulabs-hub notes, "Introduction") but give no gradient
 * formula; this is the derivative of steps 4-6 above with the buckets held fixed.  The
 * hash is piecewise constant, so neither the hash nor the sort is differentiated.
 * Steps 1-2 are recomputed here with the forward's kernels, which are deterministic and
 * so give the forward's buckets and order.  Every (round, candidate) pair of token i is
 * one entry of a single softmax with weight exp(s_ij - lse_i), which is why `out` and
 * `lse` from the forward are all that is kept of it.
 *   qk, v, R  as given to lsh_attn_forward (same dtype, sizes, causal and scale)
 *   out, lse  fp32 [B][H][L][d] and [B][H][L]: that call's outputs, unchanged.  lse
 *             must be the forward's own combined lse: the kernel uses it as the softmax
 *             normaliser of every (round, candidate) weight, and it reads a value below
 *             -5e4 (half the self logit) as "no key in any round".  A recomputed or
 *             shifted lse gives wrong gradients without an error.
 *   g_out     fp32 [B][H][L][d]: the loss's gradient in out
 *   g_lse     fp32 [B][H][L]: the loss's gradient in lse, or NULL for zero
 *   dqk, dv   fp32 [B][H][L][d]: overwritten with the gradients in qk and v
 * A zero row of qk has a constant score 0 as a key and gets no gradient through that
 * role.  A token with no key left in any round gets 1/n_rounds of its output gradient
 * in dv from each round (it copies v_i).  dqk and dv must not alias any input or the
 * workspace.  The gradients are summed with fp32 atomics, so the order of additions,
 * and with it the last bits, can change from call to call.
 * Arithmetic: LSH_F32 runs in fp32 on the CUDA cores.  LSH_BF16 (d in {64, 128}, chunk
 * in {32, 64}) runs its five contractions on the tensor cores with bf16 operands and
 * fp32 accumulation: g_out, the weights exp(s_ij - lse_i) and the score gradients are
 * rounded to bf16 for the products (scores, their softmax and g_out . out stay fp32);
 * qk, v, out, g_out, dqk and dv must then be 16-byte aligned (else
 * LSH_ERR_INVALID_ARGUMENT).  At d = 128 and chunk 64 the contractions run on tcgen05
 * (shared-memory operands, TMEM accumulators); the other shapes on warp-level MMA.
 */
lsh_status_t lsh_attn_backward(const void *qk, const void *v, const void *R, lsh_dtype_t dtype,
                               int B, int H, int L, int d, int n_buckets, int n_rounds,
                               int chunk, int causal, float scale, const float *out,
                               const float *lse, const float *g_out, const float *g_lse,
                               float *dqk, float *dv, void *workspace, size_t workspace_bytes,
                               void *stream);

/*
 * lsh_attn_backward that also records four caller-created CUDA events (cudaEvent_t) on
 * `stream`: stage_events[0] before the hash, [1] before the sort, [2] before the backward
 * kernel and [3] after it (the clearing of dqk and dv comes before [0]).  A NULL array or
 * event is LSH_ERR_INVALID_ARGUMENT.
 */
lsh_status_t lsh_attn_backward_timed(const void *qk, const void *v, const void *R,
                                     lsh_dtype_t dtype, int B, int H, int L, int d,
                                     int n_buckets, int n_rounds, int chunk, int causal,
                                     float scale, const float *out, const float *lse,
                                     const float *g_out, const float *g_lse, float *dqk,
                                     float *dv, void *workspace, size_t workspace_bytes,
                                     void *stream, void *const *stage_events);

/*
 * Number of kernels one lsh_attn_forward call launches for this problem (0 when the
 * arguments are invalid or unsupported).  The workspace status clear is a memset, not
 * a kernel, and is not counted.
 */
int lsh_attn_kernel_launches(int B, int H, int L, int d, int n_buckets, int n_rounds,
                             int chunk, lsh_dtype_t dtype);

/*
 * Byte offsets of the intermediates inside lsh_attn_forward's workspace, for
 * callers that want to inspect them.  Any pointer may be NULL.
 */
lsh_status_t lsh_attn_workspace_layout(int B, int H, int L, int d, int n_buckets, int n_rounds,
                                       int chunk, lsh_dtype_t dtype, size_t *off_buckets,
                                       size_t *off_inv_norm, size_t *off_perm, size_t *off_inv,
                                       size_t *off_bstart, size_t *off_o_r, size_t *off_lse_r);

/* ---------------------------------------------------------------- stages */

/*
 * Step 1, angular LSH ("Atencion LSH": the bucket is the position of the largest
 * entry of [xR, -xR]; modulabs-hub "Locality sensitive hashing": R has half as many
 * columns as there are buckets).  Ties go to the first index of the concatenation.
 * Writes buckets [B][H][n_rounds][L] and inv_norm [B][H][L].
 */
size_t lsh_hash_workspace_bytes(int n_rounds, int d, int n_buckets, lsh_dtype_t dtype);
lsh_status_t lsh_hash(const void *qk, const void *R, lsh_dtype_t dtype, int B, int H, int L,
                      int d, int n_buckets, int n_rounds, int32_t *buckets, float *inv_norm,
                      void *workspace, size_t workspace_bytes, void *stream);

/*
 * Step 2, stable sort of each (b, h, r) segment by bucket (ai-scholar.tech article,
 * "LSH attention": sort each LSH bucket; modulabs-hub: "ordering" the bucketed
 * keys).  Ties keep position order.  Writes perm, inv and bstart (layouts above).
 * Every bucket id must lie in [0, n_buckets).  An id outside that range is skipped:
 * its token gets no sorted slot, so perm, inv and bstart are then undefined, but no
 * memory outside them is written.
 */
size_t lsh_bucket_sort_workspace_bytes(int B, int H, int L, int n_buckets, int n_rounds);
lsh_status_t lsh_bucket_sort(const int32_t *buckets, int B, int H, int L, int n_buckets,
                             int n_rounds, int32_t *perm, int32_t *inv, int32_t *bstart,
                             void *workspace, size_t workspace_bytes, void *stream);

/*
 * lsh_bucket_sort for callers that cannot allocate device memory (frameworks whose
 * allocator they do not own, runtimes that forbid allocation after start-up, code that
 * must not risk cudaMalloc's implicit synchronisation or failure).  The paper has no
 * counterpart: this is a packaging choice of this library.  Same inputs, outputs and
 * results as lsh_bucket_sort, but the sort's scratch comes from an 8 MiB array that
 * the library holds on every GPU that loads it, until the process exits.
 *  - Needs 4 * B*H*n_rounds * n_buckets * ceil(L/4096) <= 8 MiB; larger problems return
 *    LSH_ERR_WORKSPACE_TOO_SMALL and launch nothing.
 *  - All calls on a device share that array: calls that overlap on the GPU race and
 *    corrupt each other; order them on one stream.
 *  - The first call on a device looks the array's address up with that device
 *    current; make it before any stream capture, with the stream's device current.
 *    The address is kept for the life of the process: after cudaDeviceReset (or any
 *    teardown of the device's primary context) this entry point must not be called
 *    again on that device.
 *  - Allocates nothing and takes no workspace.
 */
lsh_status_t lsh_bucket_sort_noalloc(const int32_t *buckets, int B, int H, int L, int n_buckets,
                                     int n_rounds, int32_t *perm, int32_t *inv, int32_t *bstart,
                                     void *stream);

/*
 * Steps 3-4, chunked attention of every round ("Atencion LSH": equal chunks, each
 * token attends to its own and the previous chunk; modulabs-hub "LSH attention":
 * same-bucket, self and causal masks).  Sorted row s sees the sorted rows
 * [(s/chunk - 1)*chunk, (s/chunk + 1)*chunk) clipped to [0, L); chunk 0 has no
 * previous chunk.  Writes o_r and lse_r in sorted order (layouts above).
 * buckets, perm and bstart must come from one sort of the same buckets (as
 * lsh_bucket_sort writes them).  The bf16 tensor-core path finds each row's bucket run
 * from the sorted rows' buckets, and the other paths read bstart, so inconsistent
 * arrays give path-dependent results.  Permutation entries outside [0, L) are
 * replaced by 0 (no out-of-range reads) and then the results are meaningless.
 */
size_t lsh_chunk_attn_workspace_bytes(void);
lsh_status_t lsh_chunk_attn(const void *qk, const void *v, lsh_dtype_t dtype,
                            const int32_t *buckets, const int32_t *perm, const int32_t *bstart,
                            const float *inv_norm, int B, int H, int L, int d, int n_buckets,
                            int n_rounds, int chunk, int causal, float scale, void *o_r,
                            float *lse_r, void *workspace, size_t workspace_bytes,
                            void *stream);

/*
 * Steps 5-6, un-sort and combine rounds: for token i,
 * lse_i = logsumexp_r lse_r[inv_r[i]] and out_i = sum_r exp(lse_r[inv_r[i]] - lse_i)
 * o_r[inv_r[i]].  o_r is bf16 when dtype is LSH_BF16 or LSH_F16 and fp32 when LSH_F32.
 * Every inv entry must lie in [0, L), as lsh_bucket_sort writes it.  An entry outside
 * that range is replaced by 0 (no read leaves the round's rows); that token's results
 * are then meaningless.
 */
lsh_status_t lsh_unsort_combine(const void *o_r, const float *lse_r, const int32_t *inv,
                                lsh_dtype_t dtype, int B, int H, int L, int d, int n_rounds,
                                float *out, float *lse, void *stream);

/* ---------------------------------------------------------------- k-NN search */

/*
 * LSH bucketing as approximate k-nearest-neighbour search ("Reformer" glossary,
 * ultralytics.com, section "Atencion LSH", the paragraph after the algorithm: LSH is the
 * classic approximate nearest-neighbour method and finds most of a query's nearest
 * neighbours at a fraction of the cost of an exhaustive search).  Steps 1-2 above, then:
 * the candidates of token i are the union over the rounds of the tokens sharing its
 * bucket in its chunk window (own chunk in both directions and the previous chunk, i
 * itself left out); they are ranked by cosine similarity x_i.x_j / (|x_i| |x_j|) (0 when
 * either vector is zero), ties to the smaller j, and the first k are written.
 *   qk        [B][H][L][d] dtype;  R [n_rounds][d][n_buckets/2] dtype
 *   k         1..32, with n_rounds * k <= 256
 *   nn_idx    int32 [B][H][L][k]: token positions in [0, L), -1 where fewer than k exist
 *   nn_sim    fp32  [B][H][L][k]: their similarities, descending; -2 beside a -1
 * Sizes, dtype and chunk follow lsh_attn_forward's rules.  The workspace (device,
 * 256-byte aligned, caller-owned, lsh_knn_workspace_bytes() bytes) holds the buckets,
 * the sort and the per-round candidate lists.  Asynchronous on `stream`; returns
 * argument and launch errors only.
 */
size_t lsh_knn_workspace_bytes(int B, int H, int L, int d, int n_buckets, int n_rounds,
                               int chunk, int k, lsh_dtype_t dtype);
lsh_status_t lsh_knn(const void *qk, const void *R, lsh_dtype_t dtype, int B, int H, int L,
                     int d, int n_buckets, int n_rounds, int chunk, int k, int32_t *nn_idx,
                     float *nn_sim, void *workspace, size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------- reversible block */

/*
 * The dense projections of the reversible block (below) on the tensor cores, exported on
 * their own:  C = epilogue(A W^T),  A bf16 [M][K], W bf16 [N][K] (K contiguous in both,
 * row = output feature as in a linear layer's weight), accumulated in fp32.  Epilogue, in
 * this order: + bias[N] (fp32, optional); ReLU (relu = 1); with res (fp32 [M][N],
 * optional) out = res + res_sign * value.  The result goes to out_f32 (fp32 [M][N]) and/or
 * out_bf16 (bf16, rounded to nearest even): row-major [M][N] when split_L = split_d = 0,
 * else split into heads, row m = (b, l) = (m / split_L, m % split_L) and column
 * n = (h, c) = (n / split_d, n % split_d) stored at [b][h][l][c] (M % split_L == 0,
 * N % split_d == 0, split_d % 32 == 0).  N % 128 == 0 and K % 64 == 0, else
 * LSH_ERR_UNSUPPORTED; any M >= 1.  A, W, res and the outputs 16-byte aligned.
 * Workspace: device, 256-byte aligned, >= 256 bytes (the status block only).
 * The matrix products of the pages' attention and feed-forward layers are plain linear
 * layers; nothing in the pages fixes their arithmetic beyond that.
 */
lsh_status_t lsh_gemm_bf16(const void *A, const void *W, int M, int N, int K,
                           const float *bias, int relu, const float *res, float res_sign,
                           float *out_f32, void *out_bf16, int split_L, int split_d,
                           void *workspace, size_t workspace_bytes, void *stream);

/*
 * The reversible residual block around the LSH attention (ai-scholar.tech Reformer
 * article, sections "什么是可逆残余层？" and "RevNet 中的反向传播"; "Reformer" glossary,
 * ultralytics.com, section "Capas reversibles y división en fragmentos"; modulabs-hub
 * notes, "Reversible Transformer" and "Chunking"):
 *     y1 = x1 + Attention(x2),        y2 = x2 + FeedForward(y1)          (forward)
 *     x2 = y2 - FeedForward(y1),      x1 = y1 - Attention(x2)            (inverse)
 * Attention(x) = LSHAttention(x Wqk^T, x Wv^T) Wo^T: one shared query/key projection, the
 * d_model columns split into `heads` heads of d = d_model / heads (64 or 128), steps 1-6
 * above on each head (n_buckets, n_rounds, chunk, causal, scale as lsh_attn_forward), the
 * heads merged back.  FeedForward(y) = relu(y W1^T + b1) W2^T + b2, evaluated over chunks
 * of ff_chunk positions (rows of [B*L][d_model]), so only one chunk's hidden layer exists.
 *   x1, x2, y1, y2   fp32 [B][L][d_model]   (the residual stream; four distinct arrays)
 * Every pointer must be 16-byte aligned (b1 and b2 included); a NULL or misaligned pointer,
 * or two residual-stream arguments that are the same array, give LSH_ERR_INVALID_ARGUMENT.
 *   Wqk, Wv, Wo      bf16 [d_model][d_model]   (row = output feature, [out][in])
 *   W1               bf16 [d_ff][d_model];  b1 fp32 [d_ff]
 *   W2               bf16 [d_model][d_ff];  b2 fp32 [d_model]
 *   R                bf16 [n_rounds][d][n_buckets/2]
 * d_model and d_ff must be multiples of 128.  Matrix products take bf16 copies of their
 * inputs and accumulate in fp32 on the tensor cores; the attention runs in bf16 as
 * lsh_attn_forward does.  The inverse recomputes the forward's inputs up to the rounding
 * of the fp32 residual additions (and, where a recomputed input rounds differently to
 * bf16, the near-tie effects of that on the hash).  Workspace: device, 256-byte aligned,
 * caller-owned, lsh_revblock_workspace_bytes() bytes (0: invalid sizes); its first 256
 * bytes are the status block lsh_workspace_status reads.  Asynchronous on `stream`.
 */
size_t lsh_revblock_workspace_bytes(int B, int L, int d_model, int heads, int d_ff,
                                    int n_buckets, int n_rounds, int chunk, int ff_chunk);
lsh_status_t lsh_revblock_forward(const float *x1, const float *x2, const void *Wqk,
                                  const void *Wv, const void *Wo, const void *W1,
                                  const float *b1, const void *W2, const float *b2,
                                  const void *R, int B, int L, int d_model, int heads, int d_ff,
                                  int n_buckets, int n_rounds, int chunk, int causal,
                                  float scale, int ff_chunk, float *y1, float *y2,
                                  void *workspace, size_t workspace_bytes, void *stream);
lsh_status_t lsh_revblock_inverse(const float *y1, const float *y2, const void *Wqk,
                                  const void *Wv, const void *Wo, const void *W1,
                                  const float *b1, const void *W2, const float *b2,
                                  const void *R, int B, int L, int d_model, int heads, int d_ff,
                                  int n_buckets, int n_rounds, int chunk, int causal,
                                  float scale, int ff_chunk, float *x1, float *x2,
                                  void *workspace, size_t workspace_bytes, void *stream);
/*
 * Byte offsets of the block's intermediates inside its workspace, for callers (and
 * tests) that inspect them: the attention's own workspace (lsh_attn_forward's layout,
 * status block first), the per-head projections qk and v (bf16 [B][heads][L][d]), the
 * attention output (fp32 [B][heads][L][d]) and the merged heads (bf16 [B*L][d_model]),
 * as left by the last forward or inverse call.  Any pointer may be NULL.
 */
lsh_status_t lsh_revblock_workspace_layout(int B, int L, int d_model, int heads, int d_ff,
                                           int n_buckets, int n_rounds, int chunk, int ff_chunk,
                                           size_t *off_attn_ws, size_t *off_qk, size_t *off_v,
                                           size_t *off_attn_out, size_t *off_merged);

/*
 * Self test of the bounded waits the tensor-core kernels use (the pages have no
 * counterpart: it exists to test this library's failure reporting).  Clears the status
 * block at the start of `workspace` (>= 256 bytes, 256-byte aligned, device memory) and
 * launches one warp that waits on an mbarrier nothing ever arrives on.  After the wait
 * limit (1 s) the wait gives up, records detail 0xF01 in the status block and the
 * kernel returns: nothing traps or hangs, and the context stays usable.  A following
 * lsh_workspace_status() on the same stream then returns LSH_ERR_DEVICE_CHECK with
 * detail 0xF01.  Returns launch errors only, like every entry point.
 */
lsh_status_t lsh_selftest_wait_timeout(void *workspace, size_t workspace_bytes, void *stream);

/*
 * Waits for `stream`, then reads the status block at the start of `workspace`:
 * LSH_OK, or LSH_ERR_DEVICE_CHECK when a kernel gave up a bounded wait since the
 * block was last cleared (each entry point that takes a workspace clears it).
 * `detail`, when not NULL, receives the kernel's code for where it gave up.
 */
lsh_status_t lsh_workspace_status(const void *workspace, int *detail, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* LSH_ATTN_H */
