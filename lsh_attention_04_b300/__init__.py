"""Python binding of the LSH-attention C ABI (include/lsh_attn.h).

Argument marshalling only: every step of the forward pass runs in the CUDA kernels of
``liblshattn.so``.  torch supplies device memory and the current stream.  When the
library cannot be loaded, every call raises; there is no fallback.

Functions carry the C names: lsh_attn_forward, lsh_attn_backward, lsh_hash,
lsh_bucket_sort, lsh_chunk_attn, lsh_unsort_combine, lsh_attn_workspace_bytes,
lsh_status_string, lsh_workspace_status.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "liblshattn.so")

LSH_OK = 0
LSH_ERR_INVALID_ARGUMENT = 1
LSH_ERR_UNSUPPORTED = 2
LSH_ERR_WORKSPACE_TOO_SMALL = 3
LSH_ERR_CUDA = 4
LSH_ERR_DEVICE_CHECK = 5

LSH_F32 = 0
LSH_BF16 = 1
LSH_F16 = 2

#: Every symbol the header declares.
EXPORTS = (
    "lsh_status_string", "lsh_attn_workspace_bytes", "lsh_attn_forward",
    "lsh_attn_workspace_layout", "lsh_hash_workspace_bytes", "lsh_hash",
    "lsh_bucket_sort_workspace_bytes", "lsh_bucket_sort", "lsh_chunk_attn_workspace_bytes",
    "lsh_chunk_attn", "lsh_unsort_combine", "lsh_workspace_status", "lsh_attn_forward_timed",
    "lsh_attn_kernel_launches", "lsh_bucket_sort_noalloc", "lsh_selftest_wait_timeout",
    "lsh_attn_backward_workspace_bytes", "lsh_attn_backward", "lsh_attn_backward_timed",
    "lsh_knn_workspace_bytes", "lsh_knn", "lsh_revblock_workspace_bytes", "lsh_revblock_forward",
    "lsh_revblock_inverse", "lsh_revblock_workspace_layout", "lsh_gemm_bf16",
)

_lib = None


class LshError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {lsh_status_string(status)}")


def load():
    """Load liblshattn.so (raises OSError when it is missing: build it first)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise OSError(f"{LIB_PATH} is missing; run python -m lsh_attention_04_b300.build")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.lsh_status_string.argtypes = [I]
    lib.lsh_status_string.restype = ctypes.c_char_p
    lib.lsh_attn_workspace_bytes.argtypes = [I] * 7 + [I]
    lib.lsh_attn_workspace_bytes.restype = S
    lib.lsh_attn_forward.argtypes = [P, P, P, I] + [I] * 8 + [F, P, P, P, S, P]
    lib.lsh_attn_forward.restype = I
    lib.lsh_attn_forward_timed.argtypes = [P, P, P, I] + [I] * 8 + [F, P, P, P, S, P, P]
    lib.lsh_attn_forward_timed.restype = I
    lib.lsh_attn_kernel_launches.argtypes = [I] * 8
    lib.lsh_attn_kernel_launches.restype = I
    lib.lsh_attn_workspace_layout.argtypes = [I] * 8 + [ctypes.POINTER(S)] * 7
    lib.lsh_attn_workspace_layout.restype = I
    lib.lsh_hash_workspace_bytes.argtypes = [I, I, I, I]
    lib.lsh_hash_workspace_bytes.restype = S
    lib.lsh_hash.argtypes = [P, P, I] + [I] * 6 + [P, P, P, S, P]
    lib.lsh_hash.restype = I
    lib.lsh_bucket_sort_workspace_bytes.argtypes = [I] * 5
    lib.lsh_bucket_sort_workspace_bytes.restype = S
    lib.lsh_bucket_sort.argtypes = [P] + [I] * 5 + [P, P, P, P, S, P]
    lib.lsh_bucket_sort.restype = I
    lib.lsh_chunk_attn_workspace_bytes.argtypes = []
    lib.lsh_chunk_attn_workspace_bytes.restype = S
    lib.lsh_chunk_attn.argtypes = [P, P, I, P, P, P, P] + [I] * 8 + [F, P, P, P, S, P]
    lib.lsh_chunk_attn.restype = I
    lib.lsh_knn_workspace_bytes.argtypes = [I] * 8 + [I]
    lib.lsh_knn_workspace_bytes.restype = S
    lib.lsh_knn.argtypes = [P, P, I] + [I] * 8 + [P, P, P, S, P]
    lib.lsh_knn.restype = I
    lib.lsh_revblock_workspace_bytes.argtypes = [I] * 9
    lib.lsh_revblock_workspace_bytes.restype = S
    rev = [P] * 10 + [I] * 9 + [F, I, P, P, P, S, P]
    lib.lsh_revblock_forward.argtypes = rev
    lib.lsh_revblock_forward.restype = I
    lib.lsh_revblock_inverse.argtypes = rev
    lib.lsh_revblock_inverse.restype = I
    lib.lsh_revblock_workspace_layout.argtypes = [I] * 9 + [ctypes.POINTER(S)] * 5
    lib.lsh_revblock_workspace_layout.restype = I
    lib.lsh_gemm_bf16.argtypes = [P, P, I, I, I, P, I, P, F, P, P, I, I, P, S, P]
    lib.lsh_gemm_bf16.restype = I
    lib.lsh_unsort_combine.argtypes = [P, P, P, I] + [I] * 5 + [P, P, P]
    lib.lsh_unsort_combine.restype = I
    lib.lsh_workspace_status.argtypes = [P, ctypes.POINTER(I), P]
    lib.lsh_workspace_status.restype = I
    lib.lsh_attn_backward_workspace_bytes.argtypes = [I] * 8
    lib.lsh_attn_backward_workspace_bytes.restype = S
    lib.lsh_attn_backward.argtypes = [P, P, P, I] + [I] * 8 + [F, P, P, P, P, P, P, P, S, P]
    lib.lsh_attn_backward.restype = I
    lib.lsh_attn_backward_timed.argtypes = [P, P, P, I] + [I] * 8 + [F, P, P, P, P, P, P, P, S, P, P]
    lib.lsh_attn_backward_timed.restype = I
    lib.lsh_selftest_wait_timeout.argtypes = [P, S, P]
    lib.lsh_selftest_wait_timeout.restype = I
    _lib = lib
    return lib


def lsh_status_string(status: int) -> str:
    return load().lsh_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != LSH_OK:
        raise LshError(status, what)


# ---- torch marshalling -------------------------------------------------------------

def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return LSH_F32
    if t.dtype == torch.bfloat16:
        return LSH_BF16
    if t.dtype == torch.float16:
        return LSH_F16
    raise TypeError(f"unsupported dtype {t.dtype}; use float32, bfloat16 or float16")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def lsh_attn_workspace_bytes(B, H, L, d, n_buckets, n_rounds, chunk, dtype_code) -> int:
    return int(load().lsh_attn_workspace_bytes(B, H, L, d, n_buckets, n_rounds, chunk, dtype_code))


def workspace(B, H, L, d, n_buckets, n_rounds, chunk, dtype_code, device="cuda"):
    """A device workspace tensor (uint8) for lsh_attn_forward."""
    torch = _torch()
    n = lsh_attn_workspace_bytes(B, H, L, d, n_buckets, n_rounds, chunk, dtype_code)
    if n == 0:
        raise LshError(LSH_ERR_INVALID_ARGUMENT, "lsh_attn_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device)


def lsh_attn_workspace_layout(B, H, L, d, n_buckets, n_rounds, chunk, dtype_code) -> dict:
    offs = [ctypes.c_size_t() for _ in range(7)]
    _check(load().lsh_attn_workspace_layout(B, H, L, d, n_buckets, n_rounds, chunk, dtype_code,
                                            *[ctypes.byref(o) for o in offs]),
           "lsh_attn_workspace_layout")
    names = ("buckets", "inv_norm", "perm", "inv", "bstart", "o_r", "lse_r")
    return {n: o.value for n, o in zip(names, offs)}


def lsh_attn_forward(qk, v, R, n_buckets, chunk, causal, scale, out=None, lse=None,
                     ws=None, stream=None):
    """Forward pass.  qk, v [B, H, L, d]; R [n_rounds, d, n_buckets/2] (same dtype).

    Returns (out fp32 [B, H, L, d], lse fp32 [B, H, L]).  ``ws`` is an optional
    workspace from ``workspace(...)`` (allocated here when absent)."""
    torch = _torch()
    B, H, L, d = qk.shape
    n_rounds = R.shape[0]
    dt = _dtype_code(qk)
    if v.dtype != qk.dtype or R.dtype != qk.dtype:
        raise TypeError("qk, v and R must share one dtype")
    if out is None:
        out = torch.empty((B, H, L, d), dtype=torch.float32, device=qk.device)
    if lse is None:
        lse = torch.empty((B, H, L), dtype=torch.float32, device=qk.device)
    if ws is None:
        ws = workspace(B, H, L, d, n_buckets, n_rounds, chunk, dt, qk.device)
    _check(load().lsh_attn_forward(_ptr(qk), _ptr(v), _ptr(R), dt, B, H, L, d, n_buckets,
                                   n_rounds, chunk, int(causal), float(scale), _ptr(out),
                                   _ptr(lse), _ptr(ws), ws.numel(), _stream(stream)),
           "lsh_attn_forward")
    return out, lse


def lsh_attn_forward_timed(qk, v, R, n_buckets, chunk, causal, scale, out, lse, ws, events,
                           stream=None):
    """lsh_attn_forward recording five torch.cuda.Event objects at the stage boundaries
    (before hash, sort, attention, combination, and after it)."""
    B, H, L, d = qk.shape
    s = _stream(stream)
    handles = (ctypes.c_void_p * 5)()
    for k, ev in enumerate(events):
        if ev.cuda_event == 0:  # torch creates the event on its first record
            ev.record()
        handles[k] = ev.cuda_event
    _check(load().lsh_attn_forward_timed(_ptr(qk), _ptr(v), _ptr(R), _dtype_code(qk), B, H, L,
                                         d, n_buckets, R.shape[0], chunk, int(causal),
                                         float(scale), _ptr(out), _ptr(lse), _ptr(ws),
                                         ws.numel(), s, handles),
           "lsh_attn_forward_timed")
    return out, lse


def lsh_attn_backward(qk, v, R, n_buckets, chunk, causal, scale, out, lse, g_out, g_lse=None,
                      dqk=None, dv=None, ws=None, stream=None):
    """Backward pass: gradients in qk and v of sum(g_out * out) + sum(g_lse * lse), where
    out and lse are lsh_attn_forward's outputs for the same arguments (buckets held fixed).

    g_out fp32 [B, H, L, d]; g_lse fp32 [B, H, L] or None (zero).  Returns (dqk, dv),
    fp32 [B, H, L, d]."""
    torch = _torch()
    B, H, L, d = qk.shape
    n_rounds = R.shape[0]
    dt = _dtype_code(qk)
    if v.dtype != qk.dtype or R.dtype != qk.dtype:
        raise TypeError("qk, v and R must share one dtype")
    for name, t in (("out", out), ("lse", lse), ("g_out", g_out), ("g_lse", g_lse)):
        if t is not None and t.dtype != torch.float32:
            raise TypeError(f"{name} must be float32")
    if dqk is None:
        dqk = torch.empty((B, H, L, d), dtype=torch.float32, device=qk.device)
    if dv is None:
        dv = torch.empty((B, H, L, d), dtype=torch.float32, device=qk.device)
    if ws is None:
        n = int(load().lsh_attn_backward_workspace_bytes(B, H, L, d, n_buckets, n_rounds, chunk, dt))
        if n == 0:
            raise LshError(LSH_ERR_INVALID_ARGUMENT, "lsh_attn_backward_workspace_bytes")
        ws = torch.empty(n, dtype=torch.uint8, device=qk.device)
    _check(load().lsh_attn_backward(_ptr(qk), _ptr(v), _ptr(R), dt, B, H, L, d, n_buckets,
                                    n_rounds, chunk, int(causal), float(scale), _ptr(out),
                                    _ptr(lse), _ptr(g_out),
                                    None if g_lse is None else _ptr(g_lse), _ptr(dqk), _ptr(dv),
                                    _ptr(ws), ws.numel(), _stream(stream)),
           "lsh_attn_backward")
    return dqk, dv


def lsh_attn_backward_timed(qk, v, R, n_buckets, chunk, causal, scale, out, lse, g_out, g_lse,
                            dqk, dv, ws, events, stream=None):
    """lsh_attn_backward recording four torch.cuda.Event objects at the stage boundaries
    (before hash, sort, backward kernel, and after it)."""
    B, H, L, d = qk.shape
    s = _stream(stream)
    handles = (ctypes.c_void_p * 4)()
    for k, ev in enumerate(events):
        if ev.cuda_event == 0:  # torch creates the event on its first record
            ev.record()
        handles[k] = ev.cuda_event
    _check(load().lsh_attn_backward_timed(_ptr(qk), _ptr(v), _ptr(R), _dtype_code(qk), B, H, L,
                                          d, n_buckets, R.shape[0], chunk, int(causal),
                                          float(scale), _ptr(out), _ptr(lse), _ptr(g_out),
                                          None if g_lse is None else _ptr(g_lse), _ptr(dqk),
                                          _ptr(dv), _ptr(ws), ws.numel(), s, handles),
           "lsh_attn_backward_timed")
    return dqk, dv


def lsh_knn(qk, R, n_buckets, chunk, k, nn_idx=None, nn_sim=None, ws=None, stream=None):
    """LSH bucketing as approximate k-nearest-neighbour search over qk [B, H, L, d] with
    R [n_rounds, d, n_buckets/2] (same dtype).  Returns (nn_idx int32 [B, H, L, k],
    nn_sim fp32 [B, H, L, k]): per token the k most cosine-similar tokens of the union of
    its rounds' bucket-and-chunk-window candidates, padded with (-1, -2)."""
    torch = _torch()
    B, H, L, d = qk.shape
    n_rounds = R.shape[0]
    dt = _dtype_code(qk)
    if R.dtype != qk.dtype:
        raise TypeError("qk and R must share one dtype")
    if nn_idx is None:
        nn_idx = torch.empty((B, H, L, k), dtype=torch.int32, device=qk.device)
    if nn_sim is None:
        nn_sim = torch.empty((B, H, L, k), dtype=torch.float32, device=qk.device)
    if ws is None:
        n = int(load().lsh_knn_workspace_bytes(B, H, L, d, n_buckets, n_rounds, chunk, k, dt))
        if n == 0:
            raise LshError(LSH_ERR_INVALID_ARGUMENT, "lsh_knn_workspace_bytes")
        ws = torch.empty(n, dtype=torch.uint8, device=qk.device)
    _check(load().lsh_knn(_ptr(qk), _ptr(R), dt, B, H, L, d, n_buckets, n_rounds, chunk, k,
                          _ptr(nn_idx), _ptr(nn_sim), _ptr(ws), ws.numel(), _stream(stream)),
           "lsh_knn")
    return nn_idx, nn_sim


def lsh_gemm_bf16(A, W, bias=None, relu=False, res=None, res_sign=1.0, f32=True, bf16=False,
                  split=None, out_f32=None, out_bf16=None, ws=None, stream=None):
    """C = epilogue(A W^T) on the tensor cores: A bf16 [M, K], W bf16 [N, K]; + bias (fp32
    [N]), ReLU, then res + res_sign * value (res fp32 [M, N]).  Returns (fp32 [M, N] or
    None, bf16 or None); the bf16 result is [M, N], or with split = (L, d) the heads
    layout [M / L, N / d, L, d]."""
    torch = _torch()
    if A.dtype != torch.bfloat16 or W.dtype != torch.bfloat16:
        raise TypeError("A and W must be bfloat16")
    M, K = A.shape
    N = W.shape[0]
    if f32 and out_f32 is None:
        out_f32 = torch.empty((M, N), dtype=torch.float32, device=A.device)
    if bf16 and out_bf16 is None:
        shape = (M, N) if split is None else (M // split[0], N // split[1], split[0], split[1])
        out_bf16 = torch.empty(shape, dtype=torch.bfloat16, device=A.device)
    if ws is None:
        ws = torch.empty(256, dtype=torch.uint8, device=A.device)
    sL, sd = (0, 0) if split is None else split
    _check(load().lsh_gemm_bf16(_ptr(A), _ptr(W), M, N, K, _ptr(bias), int(relu), _ptr(res),
                                float(res_sign), _ptr(out_f32), _ptr(out_bf16), sL, sd, _ptr(ws),
                                ws.numel(), _stream(stream)), "lsh_gemm_bf16")
    return out_f32, out_bf16


def revblock_workspace(B, L, d_model, heads, d_ff, n_buckets, n_rounds, chunk, ff_chunk,
                       device="cuda"):
    """A device workspace tensor (uint8) for lsh_revblock_forward / lsh_revblock_inverse."""
    torch = _torch()
    n = int(load().lsh_revblock_workspace_bytes(B, L, d_model, heads, d_ff, n_buckets, n_rounds,
                                                chunk, ff_chunk))
    if n == 0:
        raise LshError(LSH_ERR_INVALID_ARGUMENT, "lsh_revblock_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device)


def lsh_revblock_workspace_layout(B, L, d_model, heads, d_ff, n_buckets, n_rounds, chunk,
                                  ff_chunk) -> dict:
    offs = [ctypes.c_size_t() for _ in range(5)]
    _check(load().lsh_revblock_workspace_layout(B, L, d_model, heads, d_ff, n_buckets, n_rounds,
                                                chunk, ff_chunk, *[ctypes.byref(o) for o in offs]),
           "lsh_revblock_workspace_layout")
    return dict(zip(("attn_ws", "qk", "v", "attn_out", "merged"), (o.value for o in offs)))


def _revblock(fn, a1, a2, w, heads, n_buckets, chunk, causal, scale, ff_chunk, o1, o2, ws,
              stream):
    torch = _torch()
    B, L, dm = a1.shape
    for t in (a1, a2):
        if t.dtype != torch.float32:
            raise TypeError("the residual stream is float32")
    for k in ("Wqk", "Wv", "Wo", "W1", "W2", "R"):
        if w[k].dtype != torch.bfloat16:
            raise TypeError(f"{k} must be bfloat16")
    d_ff, n_rounds = w["W1"].shape[0], w["R"].shape[0]
    o1 = torch.empty_like(a1) if o1 is None else o1
    o2 = torch.empty_like(a2) if o2 is None else o2
    if ws is None:
        ws = revblock_workspace(B, L, dm, heads, d_ff, n_buckets, n_rounds, chunk, ff_chunk, a1.device)
    _check(fn(_ptr(a1), _ptr(a2), _ptr(w["Wqk"]), _ptr(w["Wv"]), _ptr(w["Wo"]), _ptr(w["W1"]),
              _ptr(w["b1"]), _ptr(w["W2"]), _ptr(w["b2"]), _ptr(w["R"]), B, L, dm, heads, d_ff,
              n_buckets, n_rounds, chunk, int(causal), float(scale), ff_chunk, _ptr(o1), _ptr(o2),
              _ptr(ws), ws.numel(), _stream(stream)), fn.__name__)
    return o1, o2


def lsh_revblock_forward(x1, x2, w, heads, n_buckets, chunk, causal, scale, ff_chunk, y1=None,
                         y2=None, ws=None, stream=None):
    """Reversible block forward: (y1, y2) = (x1 + Attention(x2), x2 + FeedForward(y1)).
    x1, x2 fp32 [B, L, d_model]; w: dict of Wqk, Wv, Wo [d_model, d_model], W1 [d_ff,
    d_model], W2 [d_model, d_ff], R [n_rounds, d, n_buckets/2] (bf16) and b1, b2 (fp32)."""
    return _revblock(load().lsh_revblock_forward, x1, x2, w, heads, n_buckets, chunk, causal,
                     scale, ff_chunk, y1, y2, ws, stream)


def lsh_revblock_inverse(y1, y2, w, heads, n_buckets, chunk, causal, scale, ff_chunk, x1=None,
                         x2=None, ws=None, stream=None):
    """Reversible block inverse: x2 = y2 - FeedForward(y1), x1 = y1 - Attention(x2)."""
    return _revblock(load().lsh_revblock_inverse, y1, y2, w, heads, n_buckets, chunk, causal,
                     scale, ff_chunk, x1, x2, ws, stream)


def lsh_attn_kernel_launches(B, H, L, d, n_buckets, n_rounds, chunk, dtype_code) -> int:
    return int(load().lsh_attn_kernel_launches(B, H, L, d, n_buckets, n_rounds, chunk, dtype_code))


def lsh_hash(qk, R, n_buckets, buckets=None, inv_norm=None, ws=None, stream=None):
    """Step 1.  Returns (buckets int32 [B, H, n_rounds, L], inv_norm fp32 [B, H, L])."""
    torch = _torch()
    B, H, L, d = qk.shape
    n_rounds = R.shape[0]
    dt = _dtype_code(qk)
    if buckets is None:
        buckets = torch.empty((B, H, n_rounds, L), dtype=torch.int32, device=qk.device)
    if inv_norm is None:
        inv_norm = torch.empty((B, H, L), dtype=torch.float32, device=qk.device)
    if ws is None:
        n = int(load().lsh_hash_workspace_bytes(n_rounds, d, n_buckets, dt))
        ws = torch.empty(max(n, 256), dtype=torch.uint8, device=qk.device)
    _check(load().lsh_hash(_ptr(qk), _ptr(R), dt, B, H, L, d, n_buckets, n_rounds,
                           _ptr(buckets), _ptr(inv_norm), _ptr(ws), ws.numel(), _stream(stream)),
           "lsh_hash")
    return buckets, inv_norm


def lsh_bucket_sort(buckets, n_buckets, perm=None, inv=None, bstart=None, ws=None, stream=None):
    """Step 2.  buckets int32 [B, H, n_rounds, L] -> (perm, inv, bstart)."""
    torch = _torch()
    B, H, n_rounds, L = buckets.shape
    if perm is None:
        perm = torch.empty_like(buckets)
    if inv is None:
        inv = torch.empty_like(buckets)
    if bstart is None:
        bstart = torch.empty((B, H, n_rounds, n_buckets + 1), dtype=torch.int32,
                             device=buckets.device)
    if ws is None:
        n = int(load().lsh_bucket_sort_workspace_bytes(B, H, L, n_buckets, n_rounds))
        ws = torch.empty(max(n, 256), dtype=torch.uint8, device=buckets.device)
    _check(load().lsh_bucket_sort(_ptr(buckets), B, H, L, n_buckets, n_rounds, _ptr(perm),
                                  _ptr(inv), _ptr(bstart), _ptr(ws), ws.numel(), _stream(stream)),
           "lsh_bucket_sort")
    return perm, inv, bstart


def lsh_chunk_attn(qk, v, buckets, perm, bstart, inv_norm, n_buckets, chunk, causal, scale,
                   o_r=None, lse_r=None, ws=None, stream=None):
    """Steps 3-4.  Returns (o_r [B, H, n_rounds, L, d] sorted order, lse_r fp32)."""
    torch = _torch()
    B, H, L, d = qk.shape
    n_rounds = perm.shape[2]
    dt = _dtype_code(qk)
    if o_r is None:
        # per-round rows: fp32 for fp32 inputs, bf16 for both 16-bit input types
        o_r = torch.empty((B, H, n_rounds, L, d),
                          dtype=torch.float32 if qk.dtype == torch.float32 else torch.bfloat16,
                          device=qk.device)
    if lse_r is None:
        lse_r = torch.empty((B, H, n_rounds, L), dtype=torch.float32, device=qk.device)
    if ws is None:
        ws = torch.empty(int(load().lsh_chunk_attn_workspace_bytes()), dtype=torch.uint8,
                         device=qk.device)
    _check(load().lsh_chunk_attn(_ptr(qk), _ptr(v), dt, _ptr(buckets), _ptr(perm), _ptr(bstart),
                                 _ptr(inv_norm), B, H, L, d, n_buckets, n_rounds, chunk,
                                 int(causal), float(scale), _ptr(o_r), _ptr(lse_r), _ptr(ws),
                                 ws.numel(), _stream(stream)),
           "lsh_chunk_attn")
    return o_r, lse_r


def lsh_unsort_combine(o_r, lse_r, inv, out=None, lse=None, stream=None):
    """Steps 5-6.  o_r [B, H, n_rounds, L, d] (sorted order) -> (out, lse)."""
    torch = _torch()
    B, H, n_rounds, L, d = o_r.shape
    if o_r.dtype == torch.float16:
        raise TypeError("per-round rows are float32 or bfloat16 (also for float16 inputs)")
    dt = _dtype_code(o_r)
    if out is None:
        out = torch.empty((B, H, L, d), dtype=torch.float32, device=o_r.device)
    if lse is None:
        lse = torch.empty((B, H, L), dtype=torch.float32, device=o_r.device)
    _check(load().lsh_unsort_combine(_ptr(o_r), _ptr(lse_r), _ptr(inv), dt, B, H, L, d,
                                     n_rounds, _ptr(out), _ptr(lse), _stream(stream)),
           "lsh_unsort_combine")
    return out, lse


SELFTEST_WAIT_CODE = 0xF01


def lsh_selftest_wait_timeout(ws, stream=None):
    """Launch the bounded-wait self test into the status block of `ws` (a CUDA uint8
    tensor of >= 256 bytes); lsh_workspace_status(ws) then reports the timeout."""
    _check(load().lsh_selftest_wait_timeout(_ptr(ws), ws.numel() * ws.element_size(),
                                            _stream(stream)), "lsh_selftest_wait_timeout")


def lsh_workspace_status(ws, stream=None):
    """(status, detail) of the status block at the start of a workspace (synchronises)."""
    detail = ctypes.c_int(0)
    st = load().lsh_workspace_status(_ptr(ws), ctypes.byref(detail), _stream(stream))
    return int(st), int(detail.value)
