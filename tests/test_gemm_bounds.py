"""The GEMM checks of tests/parity.py (bf16_interval, check_bf16_in, check_residual) on the
CPU: an fp32 product passes, and plausible mistakes of a GEMM epilogue fail."""
from __future__ import annotations

import numpy as np
import pytest

from lsh_attention_04_b300.inputs import round_bf16
from tests import parity as P

M, N, K = 96, 64, 256


@pytest.fixture(scope="module")
def ops():
    rng = np.random.default_rng(17)
    A = round_bf16(rng.standard_normal((M, K), dtype=np.float32)).astype(np.float64)
    W = round_bf16(rng.standard_normal((N, K), dtype=np.float32) / 16).astype(np.float64)
    b = 0.5 * rng.standard_normal(N)
    r = rng.standard_normal((M, N))
    return A, W, b, r


def _f32(A, W, b=None):
    out = A.astype(np.float32) @ W.astype(np.float32).T
    return out if b is None else out + b.astype(np.float32)


def _trunc_bf16(x):
    u = np.ascontiguousarray(x, np.float32).view(np.uint32) & np.uint32(0xFFFF0000)
    return u.view(np.float32)


def test_fp32_product_passes(ops):
    A, W, b, r = ops
    lo, hi = P.bf16_interval(A, W, b, relu=True)
    P.check_bf16_in(round_bf16(np.maximum(_f32(A, W, b), 0)).astype(np.float64), lo, hi, "ok")
    P.check_residual((r.astype(np.float32) + _f32(A, W, b)).astype(np.float64),
                     r.astype(np.float32).astype(np.float64), A, W, b, "ok")


@pytest.mark.parametrize("mistake", ["truncate", "no_bias", "no_relu", "row_shift",
                                     "transposed_heads"])
def test_bf16_mistakes_fail(ops, mistake):
    A, W, b, _ = ops
    lo, hi = P.bf16_interval(A, W, b, relu=True)
    x = _f32(A, W, b)
    if mistake == "truncate":
        y = _trunc_bf16(np.maximum(x, 0))
    elif mistake == "no_bias":
        y = round_bf16(np.maximum(_f32(A, W), 0))
    elif mistake == "no_relu":
        y = round_bf16(x)
    elif mistake == "row_shift":
        y = round_bf16(np.maximum(np.roll(x, 1, axis=0), 0))
    else:       # two 32-column heads swapped
        y = round_bf16(np.maximum(np.concatenate([x[:, 32:], x[:, :32]], 1), 0))
    with pytest.raises(AssertionError):
        P.check_bf16_in(y.astype(np.float64), lo, hi, mistake)


@pytest.mark.parametrize("mistake", ["sign", "no_residual", "bias_twice", "k_tail_dropped"])
def test_residual_mistakes_fail(ops, mistake):
    A, W, b, r = ops
    r32 = r.astype(np.float32)
    if mistake == "sign":
        y = r32 - _f32(A, W, b)
    elif mistake == "no_residual":
        y = _f32(A, W, b)
    elif mistake == "bias_twice":
        y = r32 + _f32(A, W, b) + b.astype(np.float32)
    else:       # the last 64-wide K step left out
        y = r32 + _f32(A[:, :-64], W[:, :-64], b)
    with pytest.raises(AssertionError):
        P.check_residual(y.astype(np.float64), r32.astype(np.float64), A, W, b, mistake)
