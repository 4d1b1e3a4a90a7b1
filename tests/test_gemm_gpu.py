"""The tensor-core GEMM with its fused epilogue (lsh_gemm_bf16), through the C ABI, against
fp64 numpy products of the same bf16 values.

bf16 results must be a bf16 rounding of a value within the accumulation bound of the exact
result (tests/parity.py, bf16_interval); fp32 results within that bound plus the final
rounding (check_residual).  Shapes cover one row, fewer rows than a tile, ragged row
tails, several column tiles, more tiles than SMs (the persistent loop and both
accumulator buffers) and long K (many ring stages)."""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import lsh_attention_04_b300 as lsh
from lsh_attention_04_b300 import inputs as gen
from tests import parity as P

pytestmark = pytest.mark.gpu

SHAPES = [(1, 128, 64), (100, 128, 64), (300, 256, 192), (1000, 384, 1024), (4096, 1024, 256),
          (20000, 128, 128), (513, 640, 4096)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lsh_attention_04_b300 import build
    build.build()
    lsh.load()


def _operands(M, N, K, seed):
    rng = np.random.default_rng(seed)
    A = gen.round_bf16(rng.standard_normal((M, K), dtype=np.float32))
    W = gen.round_bf16(rng.standard_normal((N, K), dtype=np.float32) / np.float32(np.sqrt(K)))
    bias = (0.5 * rng.standard_normal(N)).astype(np.float32)
    res = rng.standard_normal((M, N), dtype=np.float32)
    dev = lambda a, dt: torch.from_numpy(a).cuda().to(dt)
    return ((A, W, bias, res),
            (dev(A, torch.bfloat16), dev(W, torch.bfloat16), dev(bias, torch.float32),
             dev(res, torch.float32)))


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemm_bias_relu_bf16(M, N, K):
    (A, W, b, _), (dA, dW, db, _) = _operands(M, N, K, M + N + K)
    _, o = lsh.lsh_gemm_bf16(dA, dW, bias=db, relu=True, f32=False, bf16=True)
    torch.cuda.synchronize()
    lo, hi = P.bf16_interval(A.astype(np.float64), W.astype(np.float64), b.astype(np.float64),
                             relu=True)
    amb = P.check_bf16_in(o.double().cpu().numpy(), lo, hi, "relu(A W^T + b)")
    assert amb < 0.5


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_gemm_residual_f32(M, N, K, sign):
    (A, W, b, r), (dA, dW, db, dr) = _operands(M, N, K, 7 * M + N + K)
    o, o16 = lsh.lsh_gemm_bf16(dA, dW, bias=db, res=dr, res_sign=sign, f32=True, bf16=True)
    torch.cuda.synchronize()
    o = o.double().cpu().numpy()
    # res + sign * (A W^T + b) == res + A (sign W)^T + sign b, negation being exact
    P.check_residual(o, r.astype(np.float64), A.astype(np.float64), sign * W.astype(np.float64),
                     sign * b.astype(np.float64), "res + s (A W^T + b)")
    # the bf16 copy is the rounding of the fp32 result itself
    assert np.array_equal(o16.double().cpu().numpy(), gen.round_bf16(o.astype(np.float32)))


@pytest.mark.parametrize("B,L,H,d,K", [(2, 1024, 2, 128, 256), (1, 300, 4, 64, 128),
                                       (3, 64, 8, 32, 64)])
def test_gemm_split_heads(B, L, H, d, K):
    """The bf16 result written as heads [B][H][L][d]: a permutation of the row-major one."""
    M, N = B * L, H * d
    (A, W, _, _), (dA, dW, _, _) = _operands(M, N, K, 11 * M + N)
    _, flat = lsh.lsh_gemm_bf16(dA, dW, f32=False, bf16=True)
    _, heads = lsh.lsh_gemm_bf16(dA, dW, f32=False, bf16=True, split=(L, d))
    torch.cuda.synchronize()
    want = flat.reshape(B, L, H, d).permute(0, 2, 1, 3)
    assert torch.equal(heads, want)
    lo, hi = P.bf16_interval(A.astype(np.float64), W.astype(np.float64))
    P.check_bf16_in(flat.double().cpu().numpy(), lo, hi, "A W^T")


def test_gemm_deterministic():
    """Repeated calls give identical bits (each output tile is one CTA's fixed K order)."""
    (_, _, _, _), (dA, dW, db, _) = _operands(4096, 1024, 1024, 3)
    a, _ = lsh.lsh_gemm_bf16(dA, dW, bias=db)
    b, _ = lsh.lsh_gemm_bf16(dA, dW, bias=db)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
