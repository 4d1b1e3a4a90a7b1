"""Zero rows of qk on the GPU, against the oracle (needs a B300).

A zero row has inverse norm 0 (it scores 0 as a key), projects to 0 in every round (bucket 0
by the first-index rule) and, as a query, weights its candidates uniformly.  The forward and
the backward pass are compared with the oracle on the GPU's own buckets, with the bars of the
other parity tests: 2e-2 (bf16) / 1e-4 (fp32) for out and lse, and 3e-2 (bf16, tensor-core
kernel) / 1e-3 (fp32) of the largest gradient for the backward fed the oracle's out and lse.
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
    W("zero_rows_bf16_B1_H2_L1344_d128_R2", 1, 2, 1344, 128, "bf16", 32, 2, 64, True, 16, 61),
    W("zero_rows_f32_B1_H1_L1024_d64_R2_noncausal", 1, 1, 1024, 64, "f32", 16, 2, 32, False, 0, 62),
    W("zero_rows_f16_B1_H1_L1024_d128_R2", 1, 1, 1024, 128, "f16", 32, 2, 64, True, 16, 63),
]
ZERO = [0, 1, 2, 63, 64, 500, 1023]       # first rows, a chunk boundary, a middle row


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lsh_attention_04_b300 import build
    build.build()
    lsh.load()


def zero_row_inputs(w):
    qk, v, R = gen.make_inputs(w)
    qk = qk.copy()
    qk[..., ZERO, :] = 0.0
    return qk, v, R


def oracle_on_buckets(w, qk, v, gb, g_out, g_lse):
    """Oracle forward and backward of every head on the buckets gb [heads, R, L]."""
    nh = w.B * w.H
    hq, hv = qk.reshape(nh, w.L, w.d), v.reshape(nh, w.L, w.d)
    go, gl = g_out.reshape(nh, w.L, w.d), g_lse.reshape(nh, w.L)
    res = [oracle.default().backward_given_buckets(hq[h], hv[h], gb[h], w.n_buckets, w.chunk,
                                                   w.causal, w.scale, go[h], gl[h])
           for h in range(nh)]
    shape = (w.B, w.H, w.L, w.d)
    return tuple(np.stack([r[k] for r in res]).reshape(shape if k != 1 else shape[:-1])
                 for k in range(4))


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_zero_rows(w):
    qk, v, R = zero_row_inputs(w)
    dq_, dv_, dR = P.to_device(qk, w.dtype), P.to_device(v, w.dtype), P.to_device(R, w.dtype)
    gb, inv_norm = lsh.lsh_hash(dq_, dR, w.n_buckets)
    torch.cuda.synchronize()
    gb = gb.cpu().numpy().reshape(-1, w.n_rounds, w.L)
    # a zero row projects to 0 in every round: bucket 0, inverse norm 0
    assert np.all(gb[:, :, ZERO] == 0)
    assert np.all(inv_norm.cpu().numpy()[..., ZERO] == 0)

    rng = np.random.default_rng(w.seed + 1000)
    g_out = rng.standard_normal(qk.shape).astype(np.float32)
    g_lse = rng.standard_normal(qk.shape[:-1]).astype(np.float32)
    out_o, lse_o, dqk_o, dv_o = oracle_on_buckets(w, qk, v, gb, g_out, g_lse)

    out, lse = lsh.lsh_attn_forward(dq_, dv_, dR, w.n_buckets, w.chunk, w.causal, w.scale)
    torch.cuda.synchronize()
    tol = P.TOL_OUT[w.dtype]
    P.check_close(out.cpu().numpy(), out_o, tol, f"{w.name} out")
    P.check_lse(lse.cpu().numpy(), lse_o, tol, f"{w.name} lse")

    as_dev = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()
    dqk, dv = lsh.lsh_attn_backward(dq_, dv_, dR, w.n_buckets, w.chunk, w.causal, w.scale,
                                    as_dev(out_o), as_dev(lse_o), as_dev(g_out), as_dev(g_lse))
    torch.cuda.synchronize()
    bar = 3e-2 if w.dtype == "bf16" else 1e-3     # the kernel-parity bars of test_backward_gpu
    P.check_close(dqk.cpu().numpy(), dqk_o, bar * float(np.abs(dqk_o).max()), f"{w.name} dqk")
    P.check_close(dv.cpu().numpy(), dv_o, bar * float(np.abs(dv_o).max()), f"{w.name} dv")
