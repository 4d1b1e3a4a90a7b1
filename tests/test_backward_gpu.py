"""Backward pass on the GPU against the oracle, through the C ABI (needs a B300).

Each case is compared on the GPU's own buckets, so hash near-ties do not enter:

* kernel parity -- lsh_attn_backward is given the oracle's out and lse (rounded to fp32),
  so only the kernel's arithmetic differs from the oracle's fp64 backward.  fp32 inputs
  (CUDA-core kernel): dot products of up to 128 terms carry relative errors near 1e-5, and
  g_out.v_j - D_i can cancel by about a factor 10: the bar is 1e-3 of the largest
  gradient.  bf16 inputs (tensor-core kernel): g_out, the weights pi and the score
  gradients are rounded to bf16 for the products (2^-9 relative each, at most two on any
  term's path), and the rounding of g_out enters ds through g_out.v_j - D_i, which the
  same factor 10 can amplify: about 2e-2 per term, so the bar is 3e-2 of the largest
  gradient.  Both are far below what a dropped or misplaced term gives (an error the size
  of the gradient itself);
* end to end -- lsh_attn_forward's own out and lse go into lsh_attn_backward.  With bf16
  inputs the forward keeps each round's rows in 16 bits (out off by up to ~1e-2), which
  moves D_i = g_out_i . out_i by a few 1e-2: the bar is 5e-2 of the largest gradient
  (1e-3 for fp32 inputs, whose rows stay in fp32).

Cases: several chunks with a ragged mix of bucket sizes, d = 64 and 128, chunk 32 and 64,
fp32 and bf16, causal and not, several rounds, a single chunk full of tokens with no key
left (the 1/n_rounds value path), and g_lse omitted.  All inputs are seeded.
"""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import lsh_attention_04_b300 as lsh
from lsh_attention_04_b300 import inputs as gen
from tests import parity as P

pytestmark = pytest.mark.gpu

W = gen.Workload
CASES = [
    W("bwd_bf16_B1_H2_L1344_d128_R3", 1, 2, 1344, 128, "bf16", 32, 3, 64, True, 16, 51),
    W("bwd_bf16_B2_H1_L1024_d64_R2_noncausal", 2, 1, 1024, 64, "bf16", 16, 2, 64, False, 8, 52),
    W("bwd_f32_B1_H2_L1088_d64_R2_chunk32", 1, 2, 1088, 64, "f32", 34, 2, 32, True, 0, 53),
    W("bwd_f32_B1_H1_L512_d128_R3_noncausal", 1, 1, 512, 128, "f32", 8, 3, 64, False, 0, 54),
    W("bwd_bf16_chunk32_L768_d128_R2", 1, 1, 768, 128, "bf16", 32, 2, 32, True, 8, 55),
    W("bwd_bf16_one_chunk_L64", 1, 1, 64, 64, "bf16", 16, 2, 64, True, 2, 56),
    W("bwd_f16_B1_H2_L1024_d128_R2", 1, 2, 1024, 128, "f16", 32, 2, 64, True, 16, 57),
    # the tcgen05 kernel non-causal, with a last 128-row tile of one chunk (L = 1088)
    W("bwd_bf16_B2_H1_L1088_d128_R2_noncausal", 2, 1, 1088, 128, "bf16", 32, 2, 64, False, 16, 59),
]
ids = [w.name for w in CASES]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lsh_attention_04_b300 import build
    build.build()
    lsh.load()


def _grads_in(w):
    rng = np.random.default_rng(w.seed + 1000)
    g_out = rng.standard_normal((w.B, w.H, w.L, w.d)).astype(np.float32)
    g_lse = rng.standard_normal((w.B, w.H, w.L)).astype(np.float32)
    return g_out, g_lse


def _oracle(w, qk, v, gb, g_out, g_lse):
    """Oracle forward + backward of every head on the GPU's buckets gb [heads, R, L]."""
    nh = w.B * w.H
    hq, hv = qk.reshape(nh, w.L, w.d), v.reshape(nh, w.L, w.d)
    go, gl = g_out.reshape(nh, w.L, w.d), None if g_lse is None else g_lse.reshape(nh, w.L)
    res = [oracle.default().backward_given_buckets(hq[h], hv[h], gb[h], w.n_buckets, w.chunk,
                                                   w.causal, w.scale, go[h],
                                                   None if gl is None else gl[h])
           for h in range(nh)]
    shape = (w.B, w.H, w.L, w.d)
    return (np.stack([r[0] for r in res]).reshape(shape),
            np.stack([r[1] for r in res]).reshape(shape[:-1]),
            np.stack([r[2] for r in res]).reshape(shape),
            np.stack([r[3] for r in res]).reshape(shape))


def _cuda_f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()


def _check(got, ref, frac, what):
    """Max abs error within frac of the largest gradient; returns that ratio."""
    scale = float(np.abs(ref).max())
    return P.check_close(got.cpu().numpy(), ref, frac * scale, what) / scale


@pytest.mark.parametrize("w", CASES, ids=ids)
def test_backward_parity(w):
    qk, v, R = gen.make_inputs(w)
    dq_, dv_, dR = P.to_device(qk, w.dtype), P.to_device(v, w.dtype), P.to_device(R, w.dtype)
    g_out, g_lse = _grads_in(w)
    use_glse = w.seed % 2 == 1           # every other case leaves g_lse out (zero)
    g_lse_in = g_lse if use_glse else None
    gb, _ = lsh.lsh_hash(dq_, dR, w.n_buckets)
    torch.cuda.synchronize()
    gb = gb.cpu().numpy().reshape(-1, w.n_rounds, w.L)
    out_o, lse_o, dqk_o, dv_o = _oracle(w, qk, v, gb, g_out, g_lse_in)
    g_out_d = _cuda_f32(g_out)
    g_lse_d = None if g_lse_in is None else _cuda_f32(g_lse)

    # kernel parity: the oracle's out and lse
    dqk, dv = lsh.lsh_attn_backward(dq_, dv_, dR, w.n_buckets, w.chunk, w.causal, w.scale,
                                    _cuda_f32(out_o), _cuda_f32(lse_o), g_out_d, g_lse_d)
    torch.cuda.synchronize()
    bar = 3e-2 if w.dtype == "bf16" else 1e-3           # fp16 runs the fp32 CUDA-core kernel
    e_q = _check(dqk, dqk_o, bar, f"{w.name} dqk (kernel)")
    e_v = _check(dv, dv_o, bar, f"{w.name} dv (kernel)")
    print(f"{w.name}: kernel errors / largest gradient: dqk {e_q:.2e}, dv {e_v:.2e}")

    # end to end: the GPU forward's out and lse
    out, lse = lsh.lsh_attn_forward(dq_, dv_, dR, w.n_buckets, w.chunk, w.causal, w.scale)
    dqk2, dv2 = lsh.lsh_attn_backward(dq_, dv_, dR, w.n_buckets, w.chunk, w.causal, w.scale,
                                      out, lse, g_out_d, g_lse_d)
    torch.cuda.synchronize()
    frac = 1e-3 if w.dtype == "f32" else 5e-2           # 16-bit inputs keep bf16 rows
    _check(dqk2, dqk_o, frac, f"{w.name} dqk (end to end)")
    _check(dv2, dv_o, frac, f"{w.name} dv (end to end)")
    assert torch.isfinite(dqk2).all() and torch.isfinite(dv2).all()


def test_backward_value_gradient_sums_to_output_gradient():
    """Each output row's weights sum to one, so with g_out = 1 the value gradients of a head
    sum to L in every column.  At the full 8-round, 1024-bucket shape of one long-sequence
    head (L = 65536, d = 128), with the forward's own out and lse: their rounding (lse off
    by up to ~2e-3) moves each row's weight sum by at most ~2e-3, so the bar is 5e-3 L; a
    value gradient counted twice, or weighted per round instead of by the combined lse,
    misses it by O(L)."""
    w = gen.WORKLOADS["long_B1_H8_L65536_d128_R8"].replace(H=1)
    qk, v, R = gen.make_inputs(w)
    dq_, dv_, dR = P.to_device(qk, w.dtype), P.to_device(v, w.dtype), P.to_device(R, w.dtype)
    g_out = torch.ones((w.B, w.H, w.L, w.d), dtype=torch.float32, device="cuda")
    out, lse = lsh.lsh_attn_forward(dq_, dv_, dR, w.n_buckets, w.chunk, w.causal, w.scale)
    dqk, dv = lsh.lsh_attn_backward(dq_, dv_, dR, w.n_buckets, w.chunk, w.causal, w.scale,
                                    out, lse, g_out)
    torch.cuda.synchronize()
    col = dv.double().sum(dim=(0, 1, 2))
    assert torch.allclose(col, torch.full_like(col, float(w.L)), rtol=0, atol=5e-3 * w.L)
    assert torch.isfinite(dqk).all() and torch.isfinite(dv).all()
