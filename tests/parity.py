"""Helpers of the GPU-vs-oracle parity tests: tolerances and comparison rules.

Tolerances: the attention outputs must be within a max abs error of 2e-2 for bf16
inputs (fp32 accumulation) and 1e-4 for fp32 inputs; buckets and the sort must be
bit-exact, except buckets at near-ties, where the oracle's top-1/top-2 margin of the
concatenated projection is below 1e-5 * |x| * |R| (|R| = the largest column 2-norm of
R_r, which bounds every projection by Cauchy-Schwarz).  Self-only rows (every round
without a candidate) carry lse = -1e5 + ln(rounds), compared with relative error 1e-6.
"""
from __future__ import annotations

import numpy as np

TOL_OUT = {"bf16": 2e-2, "f32": 1e-4}
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
    return torch.bfloat16 if name == "bf16" else torch.float32


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
