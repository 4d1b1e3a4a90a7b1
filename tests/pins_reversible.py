"""Pins of the reversible-block oracle (oracle/reversible.py): facts of the definition
that fix it without a second implementation of it.  Each pin takes the module under test
(`rv`) and the attention oracle (`orc`), so planted mistakes in a copy of the module can
be checked against them."""
from __future__ import annotations

import math

import numpy as np
import torch


def _rng(seed):
    return np.random.default_rng(4000 + seed)


def pin_inverse_recovers_the_inputs(rv, orc):
    """inverse(forward(x)) = x in fp64 (the RevNet identity), causal and not, with and
    without chunked feed-forward layers."""
    rng = _rng(1)
    for causal, ff_chunk in ((True, 16), (False, None)):
        p = rv.random_params(rng, 64, 2, 256, 8, 3, 16, causal, ff_chunk)
        x1 = rng.standard_normal((2, 64, 64))
        x2 = rng.standard_normal((2, 64, 64))
        y1, y2 = rv.forward(x1, x2, p, orc=orc)
        a1, a2 = rv.inverse(y1, y2, p, orc=orc)
        assert np.abs(a1 - x1).max() < 1e-10 and np.abs(a2 - x2).max() < 1e-10
        assert np.abs(y1 - x1).max() > 1e-2 and np.abs(y2 - x2).max() > 1e-2


def pin_chunked_feed_forward_equals_unchunked(rv, orc):
    """Chunks of positions give the position-wise layer's result (ultralytics glossary,
    "Capas reversibles y división en fragmentos")."""
    rng = _rng(2)
    p = rv.random_params(rng, 32, 2, 128, 8, 1, 16)
    y = rng.standard_normal((3, 96, 32))
    full = rv.feed_forward(y, p)
    for c in (1, 7, 32, 96):
        assert np.allclose(rv.feed_forward(y, p, chunk=c), full, rtol=0, atol=1e-12)


def pin_feed_forward_closed_forms(rv, orc):
    """With every hidden pre-activation negative the layer returns b2; with every one
    positive it is the affine map y W1^T W2^T + b1 W2^T + b2."""
    rng = _rng(3)
    p = rv.random_params(rng, 16, 2, 64, 8, 1, 16)
    y = np.abs(rng.standard_normal((2, 8, 16)))
    dead = dict(p, b1=np.full(64, -1e3))
    assert np.allclose(rv.feed_forward(y, dead), np.broadcast_to(p["b2"], y.shape), atol=0)
    live = dict(p, W1=np.abs(p["W1"]), b1=np.abs(p["b1"]) + 0.1)
    ref = y @ live["W1"].T @ live["W2"].T + live["b1"] @ live["W2"].T + live["b2"]
    assert np.allclose(rv.feed_forward(y, live), ref, rtol=1e-12, atol=1e-12)


def pin_attention_is_multi_head_softmax_at_one_bucket_and_chunk(rv, orc):
    """One bucket (R = 0) and one chunk: the attention sub-layer equals dense multi-head
    softmax attention with the self mask (torch SDPA) over the shared projection, keys
    normalised, heads merged back before the output projection."""
    rng = _rng(4)
    B, L, dm, H = 2, 32, 32, 4
    d = dm // H
    for causal in (False, True):
        p = rv.random_params(rng, dm, H, 64, 8, 2, L, causal)
        p["R"] = np.zeros_like(p["R"])
        x = rng.standard_normal((B, L, dm))
        got = rv.attention(x, p, orc=orc)
        qk = torch.from_numpy(x @ p["Wqk"].T).reshape(B, L, H, d).transpose(1, 2)
        v = torch.from_numpy(x @ p["Wv"].T).reshape(B, L, H, d).transpose(1, 2)
        k = qk / qk.norm(dim=-1, keepdim=True)
        allowed = ~torch.eye(L, dtype=torch.bool)
        if causal:
            allowed &= torch.tril(torch.ones(L, L, dtype=torch.bool))
        o = torch.nn.functional.scaled_dot_product_attention(qk, k, v, attn_mask=allowed,
                                                             scale=p["scale"])
        # causal position 0 has no key but itself: it copies its own value row
        if causal:
            o[:, :, 0] = v[:, :, 0]
        ref = o.transpose(1, 2).reshape(B, L, dm).numpy() @ p["Wo"].T
        assert np.allclose(got, ref, rtol=1e-10, atol=1e-10), causal


ALL = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
