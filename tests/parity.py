"""Helpers of the GPU-vs-oracle parity tests: tolerances and comparison rules.

Tolerances: the attention outputs must be within a max abs error of 2e-2 for bf16 and
fp16 inputs (fp32 accumulation; the per-round rows are bf16 for both) and 1e-4 for fp32
inputs; buckets and the sort must be
bit-exact, except buckets at near-ties, where the oracle's top-1/top-2 margin of the
concatenated projection is below 1e-5 * |x| * |R| (|R| = the largest column 2-norm of
R_r, which bounds every projection by Cauchy-Schwarz).  Self-only rows (every round
without a candidate) carry lse = -1e5 + ln(rounds), compared with relative error 1e-6.
"""
from __future__ import annotations

import numpy as np

from lsh_attention_04_b300.inputs import round_bf16

TOL_OUT = {"bf16": 2e-2, "f16": 2e-2, "f32": 1e-4}   # fp16 inputs keep bf16 per-round rows
NEAR_TIE = 1e-5
SELF_LOGIT = -1.0e5

#: Near-tie bucket mismatches per test case: {case: (mismatches, buckets compared)}.
#: Printed as a table at the end of the pytest run (tests/conftest.py).
NEAR_TIES: dict = {}


def record_near_ties(case, n_bad, n_total):
    """Count a case's near-tie bucket mismatches (all already checked to lie inside the
    near-tie band) for the end-of-run report."""
    bad, tot = NEAR_TIES.get(case, (0, 0))
    NEAR_TIES[case] = (bad + int(n_bad), tot + int(n_total))


def torch_dtype(name):
    import torch
    return {"bf16": torch.bfloat16, "f16": torch.float16}.get(name, torch.float32)


def dtype_code(name):
    """The library's dtype code of a workload dtype name."""
    import lsh_attention_04_b300 as lsh
    return {"bf16": lsh.LSH_BF16, "f16": lsh.LSH_F16}.get(name, lsh.LSH_F32)


def to_device(a, dtype_name, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device).to(
        torch_dtype(dtype_name)).contiguous()


def r_norm(R):
    """Largest column 2-norm of each round's R_r: [n_rounds]."""
    return np.linalg.norm(np.asarray(R, np.float64), axis=1).max(axis=1)


def check_buckets(gpu, ref, margin, x_norm, Rn):
    """gpu, ref, margin: [..., n_rounds, L]; x_norm [..., L]; Rn [n_rounds].

    Returns the number of mismatches (all of which must be near-ties)."""
    gpu = np.asarray(gpu)
    ref = np.asarray(ref)
    bad = gpu != ref
    if not bad.any():
        return 0
    band = NEAR_TIE * x_norm[..., None, :] * Rn[:, None]
    excused = margin < band
    wrong = bad & ~excused
    assert not wrong.any(), (
        f"{int(wrong.sum())} bucket mismatches outside the near-tie band; "
        f"first margins {margin[wrong][:5]} vs band {band[wrong][:5]}")
    return int(bad.sum())


def check_close(gpu, ref, tol, what):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(gpu - ref)
    m = float(err.max()) if err.size else 0.0
    assert m <= tol, f"{what}: max abs error {m:.3e} > {tol:.1e}"
    return m


def check_lse(gpu, ref, tol, what):
    """lse: self-only values (-1e5 + ln R) by relative error 1e-6, the rest by `tol`."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    selfish = ref < SELF_LOGIT / 2
    if selfish.any():
        rel = np.abs(gpu[selfish] - ref[selfish]) / np.abs(ref[selfish])
        assert rel.max() <= 1e-6, f"{what}: self-only lse relative error {rel.max():.2e}"
    return check_close(gpu[~selfish], ref[~selfish], tol, what)


# ---- products on the tensor cores ---------------------------------------------------

def acc_bound(K):
    """Relative error bound of an fp32-accumulated dot product of K bf16 pairs, as a
    multiple of the sum of the terms' magnitudes.  Products of bf16 values are exact in
    fp32; the tensor cores add them in K/16 steps of 16-term blocks into the fp32
    accumulator, so at most K/16 + 5 roundings touch any partial sum.  The unit 2^-23,
    twice round-to-nearest's, also covers adders that truncate."""
    return (K / 16 + 5) * 2.0 ** -23


def bf16_interval(A, W, bias=None, relu=False):
    """The bf16 values fp32-accumulated A W^T (+ bias, then ReLU) may round to: [lo, hi]."""
    ref = A @ W.T
    mag = np.abs(A) @ np.abs(W).T
    if bias is not None:
        ref = ref + bias
    e = acc_bound(A.shape[1]) * mag + 2.0 ** -23 * (np.abs(ref) + (0 if bias is None else np.abs(bias)))
    lo, hi = ref - e, ref + e
    if relu:
        lo, hi = np.maximum(lo, 0.0), np.maximum(hi, 0.0)
    return (round_bf16(lo.astype(np.float32)).astype(np.float64),
            round_bf16(hi.astype(np.float32)).astype(np.float64))


def check_bf16_in(gpu, lo, hi, what):
    bad = (gpu < lo) | (gpu > hi)
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} values outside their "
                           f"rounding interval; first {gpu[bad][:3]} not in "
                           f"[{lo[bad][:3]}, {hi[bad][:3]}]")
    return float(np.mean(lo != hi))


def check_residual(gpu, res, A, W, bias, what, extra=0.0):
    """gpu = res + A W^T (+ bias) in fp32, within ACC + the final rounding (+ extra)."""
    acc = A @ W.T + (0 if bias is None else bias)
    ref = res + acc
    mag = np.abs(A) @ np.abs(W).T + (0 if bias is None else np.abs(bias))
    tol = acc_bound(A.shape[1]) * mag + 2.0 ** -23 * (np.abs(ref) + np.abs(res) + np.abs(acc)) + extra
    err = np.abs(gpu - ref)
    assert (err <= tol).all(), (f"{what}: {int((err > tol).sum())} values outside the bound, "
                                f"worst excess {float((err - tol).max()):.3e}")
    return float(err.max())




def comparable_tokens(chunk, g_b, o_b, g_perm, o_perm, g_inv, o_inv):
    """[n_heads, L] mask of tokens whose every round saw the same window and buckets in two
    evaluations g and o of one attention (a bucket flip moves the sorted positions between
    its old and new place, and with them the chunk windows there).  Arrays [n_heads,
    n_rounds, L]."""
    nh, n_rounds, L = g_b.shape
    ok = np.ones((nh, L), bool)
    for h in range(nh):
        for r in range(n_rounds):
            if np.array_equal(g_b[h, r], o_b[h, r]):
                continue
            same_pos = g_perm[h, r] == o_perm[h, r]
            same_bucket = g_b[h, r][g_perm[h, r]] == o_b[h, r][o_perm[h, r]]
            good = (same_pos & same_bucket).astype(np.int64)
            cum = np.concatenate([[0], np.cumsum(good)])
            s = o_inv[h, r]
            k = s // chunk
            lo = np.maximum(0, (k - 1) * chunk)
            hi = np.minimum(L, (k + 1) * chunk)
            whole = (cum[hi] - cum[lo]) == (hi - lo)
            ok[h] &= whole & (g_inv[h, r] == s)
    return ok
