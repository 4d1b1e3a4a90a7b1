"""The oracle of the reversible residual block (fp64, numpy matmuls + the C attention oracle).

TEST INFRASTRUCTURE ONLY, like the rest of this package: only the test suite, the smoke
check and the benchmark's CPU-baseline leg use it.

The block, from the Reformer pages:
  * ai-scholar.tech Reformer article, sections "什么是可逆残余层？" and "RevNet 中的反向传播":
    the activations are split into two halves (x1, x2) and each half is updated by a
    function of the other, so a layer's inputs can be recomputed from its outputs
    instead of being stored;
  * "Reformer" glossary (ultralytics.com, es), section "Capas reversibles y división en
    fragmentos": the inputs come back as x2 = y2 - FeedForward(y1), then
    x1 = y1 - Attention(x2); the feed-forward layers run in chunks of positions because
    their hidden layer is several times wider than the model;
  * modulabs-hub Reformer notes, "Reversible Transformer" (F is the attention, G the
    feed-forward) and "Chunking".
Reading (the ai-scholar page prints the second update as y2 = x2 + g(x1), whose inverse
cannot be evaluated in the order it gives; the inverse on the ultralytics page fixes
the dependency):
    y1 = x1 + Attention(x2),        y2 = x2 + FeedForward(y1)
    x2 = y2 - FeedForward(y1),      x1 = y1 - Attention(x2)
Attention(x) = LSHAttention(x Wqk^T, x Wv^T) Wo^T, one shared query/key projection, the
heads split from and merged back into the model dimension (d_model = heads * d).
FeedForward(y) = relu(y W1^T + b1) W2^T + b2 (hidden width d_ff), applied to chunks of
positions.  The pages name no normalisation and no activation; none is added, and ReLU is
the activation.  Weight layout: W [out][in], as the GPU library takes it.

`q16`, when given, rounds the inputs of every matrix product and of the attention to
16-bit values at the points the GPU path does (the residual stream itself stays exact);
the pins run with q16 = None (pure fp64).  An optional "threads" entry of the parameters
sets the C attention oracle's thread count (all cores when absent).
"""
from __future__ import annotations

import numpy as np

from . import default as _default


def _q(a, q16):
    return a if q16 is None else q16(a)


def attention(x2, p, q16=None, orc=None):
    """Attention(x2) for x2 [B, L, d_model]: projections, LSH attention per head, head
    merge, output projection."""
    orc = orc or _default()
    B, L, dm = x2.shape
    H, d = p["heads"], dm // p["heads"]
    xq = _q(x2, q16)
    qk = _q((xq @ p["Wqk"].T).reshape(B, L, H, d).transpose(0, 2, 1, 3), q16)
    v = _q((xq @ p["Wv"].T).reshape(B, L, H, d).transpose(0, 2, 1, 3), q16)
    out, _ = orc.forward(qk, v, _q(p["R"], q16), p["n_buckets"], p["chunk"], p["causal"],
                         p["scale"], threads=p.get("threads"))
    merged = _q(out.transpose(0, 2, 1, 3).reshape(B, L, dm), q16)
    return merged @ p["Wo"].T


def feed_forward(y, p, q16=None, chunk=None):
    """FeedForward(y) for y [B, L, d_model], one chunk of positions at a time (all at once
    when chunk is None)."""
    B, L, dm = y.shape
    c = L if chunk is None else chunk
    out = np.zeros((B, L, dm))
    for i in range(0, L, c):
        yi = _q(y[:, i:i + c], q16)
        h = _q(np.maximum(yi @ p["W1"].T + p["b1"], 0.0), q16)
        out[:, i:i + c] = h @ p["W2"].T + p["b2"]
    return out


def forward(x1, x2, p, q16=None, orc=None):
    """(y1, y2) of the reversible block."""
    y1 = x1 + attention(x2, p, q16, orc)
    y2 = x2 + feed_forward(y1, p, q16, p.get("ff_chunk"))
    return y1, y2


def inverse(y1, y2, p, q16=None, orc=None):
    """(x1, x2) recomputed from the block's outputs."""
    x2 = y2 - feed_forward(y1, p, q16, p.get("ff_chunk"))
    x1 = y1 - attention(x2, p, q16, orc)
    return x1, x2


def random_params(rng, d_model, heads, d_ff, n_buckets, n_rounds, chunk, causal=True,
                  ff_chunk=None):
    """Random weights of one block (fan-in scaled normal), float64."""
    d = d_model // heads

    def lin(o, i):
        return rng.standard_normal((o, i)) / np.sqrt(i)

    return dict(heads=heads, n_buckets=n_buckets, chunk=chunk, causal=causal,
                scale=1.0 / np.sqrt(d), ff_chunk=ff_chunk,
                Wqk=lin(d_model, d_model), Wv=lin(d_model, d_model), Wo=lin(d_model, d_model),
                W1=lin(d_ff, d_model), b1=0.1 * rng.standard_normal(d_ff),
                W2=lin(d_model, d_ff), b2=0.1 * rng.standard_normal(d_model),
                R=rng.standard_normal((n_rounds, d, n_buckets // 2)))
