"""The oracle: a plain fp64 CPU restatement of multi-round LSH attention.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the benchmark's CPU-baseline leg import this package.  The CUDA library never
imports, links or calls it, and it shares no code with the library.

The arithmetic lives in ``lsh_oracle.c`` (plain C, fp64, compiled here with
gcc on first use).  This module only marshals numpy arrays into it.

Each function follows the Reformer pages:
  * hash     -- angular LSH, bucket = first argmax of [xR, -xR]
                ("Reformer" glossary, ultralytics.com, section "Atencion LSH";
                 modulabs-hub Reformer notes, "Locality sensitive hashing")
  * sort     -- order tokens by (bucket, position)
                (ai-scholar.tech Reformer article, "LSH attention")
  * attend   -- own chunk + previous chunk, same bucket, causal, self only
                when nothing else is left (modulabs-hub notes, "LSH attention")
  * combine  -- un-sort and logsumexp-weighted sum of rounds
  * forward  -- all of the above for B*H heads
  * backward -- gradients of the forward in qk and v by the chain rule, buckets
                held fixed (the pages train by back-propagation but print no
                gradient formula; modulabs-hub notes, "Introduction")
  * knn      -- LSH bucketing as approximate nearest-neighbour search: the k
                most cosine-similar tokens among the union of the rounds'
                candidate sets ("Reformer" glossary, "Atencion LSH", the
                paragraph after the algorithm); exact_knn is the exhaustive
                search it is measured against
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lsh_oracle.c")
_LIB = os.path.join(_HERE, "liblsh_oracle.so")
_lock = threading.Lock()
_default = None

SELF_LOGIT = -1.0e5


def compile_source(src_path: str, lib_path: str) -> str:
    """Compile one C source into a shared library (IEEE fp64, no fast-math)."""
    tmp = lib_path + ".tmp%d" % os.getpid()
    subprocess.check_call(
        ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
         "-o", tmp, src_path, "-lm", "-lpthread"])
    os.replace(tmp, lib_path)
    return lib_path


def build(force: bool = False) -> str:
    """Compile lsh_oracle.c into liblsh_oracle.so when missing or stale."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        compile_source(_SRC, _LIB)
    return _LIB


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """numpy front end of one compiled copy of the oracle's C code."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int, ctypes.c_long, ctypes.c_double
        lib.oracle_hash.argtypes = [P, i64, i32, P, i32, P, P]
        lib.oracle_hash.restype = None
        lib.oracle_sort.argtypes = [P, i32, i32, P, P, P]
        lib.oracle_sort.restype = None
        lib.oracle_inv_norm.argtypes = [P, i32, i32, P]
        lib.oracle_inv_norm.restype = None
        lib.oracle_attend.argtypes = [P, P, P, P, P, i32, i32, i32, i32, f64, P, i32, P, P]
        lib.oracle_attend.restype = None
        lib.oracle_combine.argtypes = [P, P, P, i32, i32, i32, P, i32, P, P]
        lib.oracle_combine.restype = None
        lib.oracle_forward.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32, i32,
                                       f64, i32] + [P] * 9
        lib.oracle_forward.restype = ctypes.c_int
        lib.oracle_combine_backward.argtypes = [P, P, P, i32, i32, i32, P, P, P, P, P, P]
        lib.oracle_combine_backward.restype = None
        lib.oracle_attend_backward.argtypes = [P, P, P, P, P, i32, i32, i32, i32, f64,
                                               P, P, P, P, P, P, P]
        lib.oracle_attend_backward.restype = None
        lib.oracle_key_norm_backward.argtypes = [P, P, P, i32, i32, P]
        lib.oracle_key_norm_backward.restype = None
        lib.oracle_backward.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32, i32, f64,
                                        P, P, P, P]
        lib.oracle_backward.restype = ctypes.c_int
        lib.oracle_knn.argtypes = [P, i32, i32, P, P, P, i32, i32, i32, P, i32, P, P]
        lib.oracle_knn.restype = None
        lib.oracle_exact_knn.argtypes = [P, i32, i32, i32, P, i32, P, P]
        lib.oracle_exact_knn.restype = None
        lib.oracle_self_logit.argtypes = []
        lib.oracle_self_logit.restype = f64
        self.lib = lib
        self.SELF_LOGIT = lib.oracle_self_logit()

    def hash(self, x, R_r, n_buckets):
        """Buckets and top-1/top-2 margins of rows x [n, d] under one round R_r [d, nb/2]."""
        lib = self.lib
        x = _f64(x)
        R_r = _f64(R_r)
        n, d = x.shape
        assert R_r.shape == (d, n_buckets // 2)
        bucket = np.empty(n, np.int32)
        margin = np.empty(n, np.float64)
        lib.oracle_hash(_p(x), n, d, _p(R_r), n_buckets, _p(bucket), _p(margin))
        return bucket, margin

    def hash_rounds(self, x, R, n_buckets):
        """Buckets [n_rounds, n] and margins for every round of R [n_rounds, d, nb/2]."""
        R = _f64(R)
        out_b = np.empty((R.shape[0], len(x)), np.int32)
        out_m = np.empty((R.shape[0], len(x)), np.float64)
        for r in range(R.shape[0]):
            out_b[r], out_m[r] = self.hash(x, R[r], n_buckets)
        return out_b, out_m

    def sort(self, bucket, n_buckets):
        """perm (sorted -> original), inv (original -> sorted), bstart [nb+1] of one segment."""
        lib = self.lib
        bucket = _i32(bucket)
        L = bucket.shape[0]
        perm = np.empty(L, np.int32)
        inv = np.empty(L, np.int32)
        bstart = np.empty(n_buckets + 1, np.int32)
        lib.oracle_sort(_p(bucket), L, n_buckets, _p(perm), _p(inv), _p(bstart))
        return perm, inv, bstart

    def inv_norm(self, qk):
        lib = self.lib
        qk = _f64(qk)
        L, d = qk.shape
        out = np.empty(L, np.float64)
        lib.oracle_inv_norm(_p(qk), L, d, _p(out))
        return out

    def attend(self, qk, v, bucket, perm, chunk, causal, scale, rows=None):
        """One round of chunked attention for one head.

        Returns (o, lse) in SORTED order: o [L, d], lse [L].  When ``rows`` (sorted
        indices) is given, only those rows are computed and returned, in that order.
        """
        lib = self.lib
        qk = _f64(qk)
        v = _f64(v)
        bucket = _i32(bucket)
        perm = _i32(perm)
        L, d = qk.shape
        inorm = self.inv_norm(qk)
        o = np.zeros((L, d), np.float64)
        lse = np.zeros(L, np.float64)
        if rows is None:
            lib.oracle_attend(_p(qk), _p(v), _p(inorm), _p(bucket), _p(perm), L, d, chunk,
                              int(causal), float(scale), None, 0, _p(o), _p(lse))
            return o, lse
        rows = _i32(rows)
        lib.oracle_attend(_p(qk), _p(v), _p(inorm), _p(bucket), _p(perm), L, d, chunk,
                          int(causal), float(scale), _p(rows), len(rows), _p(o), _p(lse))
        return o[rows], lse[rows]

    def combine(self, o_r, lse_r, inv, tokens=None):
        """Un-sort and combine rounds of one head.

        o_r [R, L, d] and lse_r [R, L] are in sorted order, inv [R, L].  Returns
        (out [n, d], lse [n]) for ``tokens`` (original positions; all when None).
        """
        lib = self.lib
        o_r = _f64(o_r)
        lse_r = _f64(lse_r)
        inv = _i32(inv)
        R, L, d = o_r.shape
        if tokens is None:
            out = np.empty((L, d), np.float64)
            lse = np.empty(L, np.float64)
            lib.oracle_combine(_p(o_r), _p(lse_r), _p(inv), R, L, d, None, 0, _p(out), _p(lse))
            return out, lse
        tokens = _i32(tokens)
        out = np.empty((len(tokens), d), np.float64)
        lse = np.empty(len(tokens), np.float64)
        lib.oracle_combine(_p(o_r), _p(lse_r), _p(inv), R, L, d, _p(tokens), len(tokens),
                           _p(out), _p(lse))
        return out, lse

    def knn(self, x, bucket, perm, inv, chunk, k, tokens=None):
        """Approximate k nearest neighbours of one head from its LSH buckets.

        x [L, d]; bucket, perm, inv [n_rounds, L] of one head.  Returns (idx [n, k] int32,
        sim [n, k]) for ``tokens`` (all when None): the k most cosine-similar tokens of the
        union of the rounds' non-causal candidate sets, ties to the smaller index, padded
        with -1 / -2.
        """
        x = _f64(x)
        L, d = x.shape
        bucket, perm, inv = _i32(bucket), _i32(perm), _i32(inv)
        n_rounds = bucket.shape[0]
        tok = None if tokens is None else _i32(tokens)
        n = L if tok is None else len(tok)
        idx = np.empty((n, k), np.int32)
        sim = np.empty((n, k), np.float64)
        self.lib.oracle_knn(_p(x), L, d, _p(bucket), _p(perm), _p(inv), n_rounds, chunk, k,
                            _p(tok), 0 if tok is None else n, _p(idx), _p(sim))
        return idx, sim

    def exact_knn(self, x, k, tokens=None):
        """Exact k nearest neighbours by cosine similarity over every other token of x."""
        x = _f64(x)
        L, d = x.shape
        tok = None if tokens is None else _i32(tokens)
        n = L if tok is None else len(tok)
        idx = np.empty((n, k), np.int32)
        sim = np.empty((n, k), np.float64)
        self.lib.oracle_exact_knn(_p(x), L, d, k, _p(tok), 0 if tok is None else n, _p(idx),
                                  _p(sim))
        return idx, sim

    def forward(self, qk, v, R, n_buckets, chunk, causal, scale, threads=None, intermediates=False):
        """Full forward pass.  qk, v: [B, H, L, d] (or [n_heads, L, d]); R [n_rounds, d, nb/2].

        Returns (out [..., L, d], lse [..., L]) and, with ``intermediates``, a dict
        with bucket, perm, inv, bstart, margin, o_r, lse_r (per head and round).
        """
        lib = self.lib
        shape = qk.shape
        L, d = shape[-2], shape[-1]
        n_heads = int(np.prod(shape[:-2]))
        qk = _f64(qk).reshape(n_heads, L, d)
        v = _f64(v).reshape(n_heads, L, d)
        R = _f64(R)
        n_rounds = R.shape[0]
        assert R.shape == (n_rounds, d, n_buckets // 2)
        if threads is None:
            threads = os.cpu_count() or 1
        out = np.empty((n_heads, L, d), np.float64)
        lse = np.empty((n_heads, L), np.float64)
        inter = None
        if intermediates:
            inter = dict(
                bucket=np.empty((n_heads, n_rounds, L), np.int32),
                perm=np.empty((n_heads, n_rounds, L), np.int32),
                inv=np.empty((n_heads, n_rounds, L), np.int32),
                bstart=np.empty((n_heads, n_rounds, n_buckets + 1), np.int32),
                margin=np.empty((n_heads, n_rounds, L), np.float64),
                o_r=np.empty((n_heads, n_rounds, L, d), np.float64),
                lse_r=np.empty((n_heads, n_rounds, L), np.float64),
            )
        g = (lambda k: _p(inter[k])) if inter else (lambda k: None)
        rc = lib.oracle_forward(_p(qk), _p(v), _p(R), n_heads, L, d, n_buckets, n_rounds, chunk,
                                int(causal), float(scale), int(threads), _p(out), _p(lse),
                                g("bucket"), g("perm"), g("inv"), g("bstart"), g("margin"),
                                g("o_r"), g("lse_r"))
        if rc != 0:
            raise MemoryError("oracle_forward ran out of host memory")
        out = out.reshape(shape)
        lse = lse.reshape(shape[:-1])
        if intermediates:
            lead = shape[:-2]
            inter = {k: a.reshape(lead + a.shape[1:]) for k, a in inter.items()}
            return out, lse, inter
        return out, lse

    def backward(self, qk, v, R, n_buckets, chunk, causal, scale, g_out, g_lse):
        """Gradients of  sum(g_out * out) + sum(g_lse * lse)  in qk and v, with the
        buckets held fixed.  Shapes as in ``forward``; returns (dqk, dv)."""
        lib = self.lib
        shape = qk.shape
        L, d = shape[-2], shape[-1]
        n_heads = int(np.prod(shape[:-2]))
        qk = _f64(qk).reshape(n_heads, L, d)
        v = _f64(v).reshape(n_heads, L, d)
        g_out = _f64(g_out).reshape(n_heads, L, d)
        g_lse = _f64(g_lse).reshape(n_heads, L)
        R = _f64(R)
        n_rounds = R.shape[0]
        assert R.shape == (n_rounds, d, n_buckets // 2)
        dqk = np.empty((n_heads, L, d), np.float64)
        dv = np.empty((n_heads, L, d), np.float64)
        rc = lib.oracle_backward(_p(qk), _p(v), _p(R), n_heads, L, d, n_buckets, n_rounds,
                                 chunk, int(causal), float(scale), _p(g_out), _p(g_lse),
                                 _p(dqk), _p(dv))
        if rc != 0:
            raise MemoryError("oracle_backward ran out of host memory")
        return dqk.reshape(shape), dv.reshape(shape)

    def combine_backward(self, o_r, lse_r, inv, out, lse, g_out, g_lse):
        """Backward of the round combination of one head: (g_o [R, L, d], g_lse_r [R, L])
        in sorted order, from the forward's sorted o_r/lse_r and token-order out/lse."""
        o_r = _f64(o_r)
        lse_r = _f64(lse_r)
        inv = _i32(inv)
        out, lse, g_out, g_lse = _f64(out), _f64(lse), _f64(g_out), _f64(g_lse)
        R, L, d = o_r.shape
        g_o = np.zeros((R, L, d), np.float64)
        g_lse_r = np.zeros((R, L), np.float64)
        self.lib.oracle_combine_backward(_p(o_r), _p(lse_r), _p(inv), R, L, d, _p(out), _p(lse),
                                         _p(g_out), _p(g_lse), _p(g_o), _p(g_lse_r))
        return g_o, g_lse_r

    def attend_backward(self, qk, v, bucket, perm, chunk, causal, scale, o, lse, g_o, g_lse):
        """Backward of one round's attention of one head (all arrays of the round in sorted
        order).  Returns (dq, dkhat, dv): the gradients through qk as query, through the
        normalised key, and in v."""
        qk, v = _f64(qk), _f64(v)
        bucket, perm = _i32(bucket), _i32(perm)
        o, lse, g_o, g_lse = _f64(o), _f64(lse), _f64(g_o), _f64(g_lse)
        L, d = qk.shape
        inorm = self.inv_norm(qk)
        dq = np.zeros((L, d), np.float64)
        dkhat = np.zeros((L, d), np.float64)
        dv = np.zeros((L, d), np.float64)
        self.lib.oracle_attend_backward(_p(qk), _p(v), _p(inorm), _p(bucket), _p(perm), L, d,
                                        chunk, int(causal), float(scale), _p(o), _p(lse),
                                        _p(g_o), _p(g_lse), _p(dq), _p(dkhat), _p(dv))
        return dq, dkhat, dv

    def key_norm_backward(self, qk, dkhat):
        """Gradient in qk through the unit key qk / |qk|, for the gradient dkhat in it."""
        qk, dkhat = _f64(qk), _f64(dkhat)
        L, d = qk.shape
        inorm = self.inv_norm(qk)
        dqk = np.zeros((L, d), np.float64)
        self.lib.oracle_key_norm_backward(_p(qk), _p(inorm), _p(dkhat), L, d, _p(dqk))
        return dqk

    def backward_given_buckets(self, qk, v, bucket, n_buckets, chunk, causal, scale, g_out,
                               g_lse):
        """Forward and backward of one head with the given buckets [n_rounds, L] instead of
        the oracle's own hash (so that hash near-ties of another implementation do not
        enter a comparison).  Returns (out, lse, dqk, dv)."""
        qk, v = _f64(qk), _f64(v)
        bucket = _i32(bucket)
        n_rounds = bucket.shape[0]
        perm, inv, o_r, lse_r = [], [], [], []
        for r in range(n_rounds):
            p, i, _ = self.sort(bucket[r], n_buckets)
            o, l = self.attend(qk, v, bucket[r], p, chunk, causal, scale)
            perm.append(p); inv.append(i); o_r.append(o); lse_r.append(l)
        o_r, lse_r, inv = np.stack(o_r), np.stack(lse_r), np.stack(inv)
        out, lse = self.combine(o_r, lse_r, inv)
        g_lse = np.zeros(len(lse)) if g_lse is None else g_lse
        g_o, g_lse_r = self.combine_backward(o_r, lse_r, inv, out, lse, g_out, g_lse)
        dq = np.zeros_like(qk)
        dkhat = np.zeros_like(qk)
        dv = np.zeros_like(v)
        for r in range(n_rounds):
            a, b, c = self.attend_backward(qk, v, bucket[r], perm[r], chunk, causal, scale,
                                           o_r[r], lse_r[r], g_o[r], g_lse_r[r])
            dq += a; dkhat += b; dv += c
        return out, lse, dq + self.key_norm_backward(qk, dkhat), dv


def default() -> Oracle:
    """The oracle compiled from lsh_oracle.c (built on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def hash(x, R_r, n_buckets):
    return default().hash(x, R_r, n_buckets)


def hash_rounds(x, R, n_buckets):
    return default().hash_rounds(x, R, n_buckets)


def sort(bucket, n_buckets):
    return default().sort(bucket, n_buckets)


def inv_norm(qk):
    return default().inv_norm(qk)


def attend(qk, v, bucket, perm, chunk, causal, scale, rows=None):
    return default().attend(qk, v, bucket, perm, chunk, causal, scale, rows)


def combine(o_r, lse_r, inv, tokens=None):
    return default().combine(o_r, lse_r, inv, tokens)


def forward(qk, v, R, n_buckets, chunk, causal, scale, threads=None, intermediates=False):
    return default().forward(qk, v, R, n_buckets, chunk, causal, scale, threads, intermediates)


def backward(qk, v, R, n_buckets, chunk, causal, scale, g_out, g_lse):
    return default().backward(qk, v, R, n_buckets, chunk, causal, scale, g_out, g_lse)


def knn(x, bucket, perm, inv, chunk, k, tokens=None):
    return default().knn(x, bucket, perm, inv, chunk, k, tokens)


def exact_knn(x, k, tokens=None):
    return default().exact_knn(x, k, tokens)
