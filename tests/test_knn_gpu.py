"""LSH k-nearest-neighbour search on the GPU against the oracle, through the C ABI.

The GPU's buckets and sort (the same deterministic kernels lsh_knn runs) are handed to
the oracle, so both sides search the same candidate sets.  Checks per token:
  * similarities, in the order returned, within SIM_TOL of the oracle's;
  * indices equal to the oracle's wherever its ranking has no near-tie (neighbouring
    similarities further apart than 2 * SIM_TOL); elsewhere the returned index must be
    a candidate of the token with that similarity;
  * no index listed twice; padding (-1, -2) exactly where the oracle pads.
SIM_TOL: both sides take the cosine of the same input values; the GPU accumulates the
dot product in fp32 (bf16 products are exact in fp32) and uses fp32 inverse norms, an
error well below 1e-5 for unit-scale similarities.
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

SIM_TOL = 1e-5
W = gen.Workload

CASES = [
    (W("knn_bf16_B2_H2_L1024_d64_R4", 2, 2, 1024, 64, "bf16", 32, 4, 64, False, 16, 51), 8),
    (W("knn_bf16_B1_H2_L2048_d128_R8", 1, 2, 2048, 128, "bf16", 64, 8, 64, False, 32, 52), 16),
    (W("knn_bf16_chunk32_L1024_d64_R2", 1, 1, 1024, 64, "bf16", 32, 2, 32, False, 16, 53), 32),
    (W("knn_bf16_one_chunk_L64_R3", 1, 1, 64, 64, "bf16", 16, 3, 64, False, 2, 54), 5),
    (W("knn_bf16_few_candidates_nb512", 1, 1, 1024, 128, "bf16", 512, 2, 64, False, 0, 55), 8),
    (W("knn_bf16_k1_R8", 1, 1, 1024, 64, "bf16", 16, 8, 64, False, 16, 56), 1),
    (W("knn_f32_B1_H2_L1088_d128_R2", 1, 2, 1088, 128, "f32", 32, 2, 32, False, 0, 57), 8),
    (W("knn_f32_L512_d64_R4", 1, 1, 512, 64, "f32", 8, 4, 64, False, 8, 58), 12),
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lsh_attention_04_b300 import build
    build.build()
    lsh.load()


def _gpu_search(w, qk, R, k, zero_rows=(), dup_rows=()):
    qk = qk.copy()
    for r in zero_rows:
        qk[..., r, :] = 0.0
    for a, b in dup_rows:
        qk[..., b, :] = qk[..., a, :]
    dqk, dR = P.to_device(qk, w.dtype), P.to_device(R, w.dtype)
    idx, sim = lsh.lsh_knn(dqk, dR, w.n_buckets, w.chunk, k)
    b, _ = lsh.lsh_hash(dqk, dR, w.n_buckets)
    perm, inv, _ = lsh.lsh_bucket_sort(b, w.n_buckets)
    torch.cuda.synchronize()
    nh = w.B * w.H
    shape = (nh, w.n_rounds, w.L)
    return (qk, idx.cpu().numpy().reshape(nh, w.L, k), sim.cpu().numpy().reshape(nh, w.L, k),
            b.cpu().numpy().reshape(shape), perm.cpu().numpy().reshape(shape),
            inv.cpu().numpy().reshape(shape))


def _check_lists(x, g_idx, g_sim, o_idx, o_sim, full_idx, full_sim, k):
    """One head: GPU lists [n, k] against the oracle's [n, k]; full_* is the oracle's whole
    ranked candidate union of each token (for membership and similarity lookups)."""
    pad = o_idx < 0
    assert np.array_equal(g_idx < 0, pad), "padding differs"
    assert np.all(g_sim[pad] == -2.0)
    live = ~pad
    assert np.abs(g_sim[live] - o_sim[live]).max(initial=0.0) <= SIM_TOL
    assert np.array_equal(full_idx[:, :k], o_idx)      # the longer ranking extends the list
    for t in range(len(g_idx)):
        row = g_idx[t][g_idx[t] >= 0]
        assert len(set(row.tolist())) == len(row), "an index listed twice"
        cand = dict(zip(full_idx[t].tolist(), full_sim[t].tolist()))
        for a in range(k):
            if o_idx[t, a] < 0:
                break
            # gaps to the neighbouring candidates of the whole ranked union (the one after
            # the last listed position may be a near-tie of it too)
            gap_lo = full_sim[t, a - 1] - full_sim[t, a] if a > 0 else np.inf
            nxt = a + 1 < full_idx.shape[1] and full_idx[t, a + 1] >= 0
            gap_hi = full_sim[t, a] - full_sim[t, a + 1] if nxt else np.inf
            if min(gap_lo, gap_hi) > 2 * SIM_TOL:
                assert g_idx[t, a] == o_idx[t, a], (t, a)
            else:
                j = int(g_idx[t, a])
                assert j in cand and abs(cand[j] - g_sim[t, a]) <= SIM_TOL, (t, a)


@pytest.mark.parametrize("w,k", CASES, ids=[c[0].name for c in CASES])
def test_knn_parity(w, k):
    qk, v, R = gen.make_inputs(w)
    zero = (5, w.L // 2) if w.L > 64 else (5,)
    dup = ((7, 9), (100, 300)) if w.L > 300 else ((7, 9),)
    qk, g_idx, g_sim, b, perm, inv = _gpu_search(w, qk, R, k, zero, dup)
    heads = qk.reshape(-1, w.L, w.d)
    full_k = min(32 * 8, w.n_rounds * 2 * w.chunk)
    for h in range(len(heads)):
        for r in range(w.n_rounds):
            o_perm, o_inv, _ = oracle.sort(b[h, r], w.n_buckets)
            assert np.array_equal(perm[h, r], o_perm) and np.array_equal(inv[h, r], o_inv)
        o_idx, o_sim = oracle.knn(heads[h], b[h], perm[h], inv[h], w.chunk, k)
        f_idx, f_sim = oracle.knn(heads[h], b[h], perm[h], inv[h], w.chunk, full_k)
        _check_lists(heads[h], g_idx[h], g_sim[h], o_idx, o_sim, f_idx, f_sim, k)
    # the zero rows: similarity 0 with everything
    for zr in zero:
        live = g_idx[0, zr] >= 0
        assert np.all(g_sim[0, zr][live] == 0.0)


def test_knn_full_size_sampled():
    """The long-text shape (L = 65536, d = 128, 1024 buckets, 8 rounds, chunk 64) with
    k = 16, compared on 256 sampled tokens of two heads; recall@16 against the exhaustive
    search of the same tokens is recorded."""
    w = gen.WORKLOADS[gen.HEADLINE].replace(H=2, name="knn_long_B1_H2_L65536_d128_R8")
    k = 16
    qk, v, R = gen.make_inputs(w)
    qk, g_idx, g_sim, b, perm, inv = _gpu_search(w, qk, R, k)
    heads = qk.reshape(-1, w.L, w.d)
    rng = np.random.default_rng(5)
    recalls = []
    for h in range(2):
        toks = np.sort(rng.choice(w.L, 256, replace=False))
        o_idx, o_sim = oracle.knn(heads[h], b[h], perm[h], inv[h], w.chunk, k, toks)
        f_idx, f_sim = oracle.knn(heads[h], b[h], perm[h], inv[h], w.chunk, 256, toks)
        _check_lists(heads[h], g_idx[h][toks], g_sim[h][toks], o_idx, o_sim, f_idx, f_sim, k)
        e_idx, _ = oracle.exact_knn(heads[h], k, toks)
        recalls += [len(set(g_idx[h][t].tolist()) & set(e_idx[q].tolist())) / k
                    for q, t in enumerate(toks)]
    print(f"recall@{k} on the long-text shape: {np.mean(recalls):.3f}")
    assert np.mean(recalls) > 0.5


def test_knn_recall_vs_rounds_and_buckets():
    """Recall@16 of the GPU search against exhaustive cosine search on the long-text shape
    (L = 65536, d = 128, clustered, chunk 64), one head, 512 sampled queries, for rounds
    1, 2, 4, 8 and 256 / 1024 / 2048 buckets (the kernels' largest).  More rounds find
    more of the true neighbours, their candidate sets being unions over the rounds; the
    table is printed."""
    base = gen.WORKLOADS[gen.HEADLINE].replace(H=1, name="knn_recall_L65536_d128")
    k = 16
    qk, _, _ = gen.make_inputs(base)
    rng = np.random.default_rng(11)
    toks = np.sort(rng.choice(base.L, 512, replace=False))
    e_idx, _ = oracle.exact_knn(qk.reshape(base.L, base.d), k, toks)
    rows = []
    for nb in (256, 1024, 2048):
        rec = []
        for R_ in (1, 2, 4, 8):
            w = base.replace(n_buckets=nb, n_rounds=R_)
            _, _, R = gen.make_inputs(w)
            dqk, dR = P.to_device(qk, "bf16"), P.to_device(R, "bf16")
            idx, _ = lsh.lsh_knn(dqk, dR, nb, w.chunk, k)
            got = idx.cpu().numpy().reshape(base.L, k)[toks]
            rec.append(np.mean([len(set(got[q].tolist()) & set(e_idx[q].tolist())) / k
                                for q in range(len(toks))]))
        rows.append((nb, rec))
        # the inputs draw the rotations in order, so the first rounds of a larger count
        # are the rounds of a smaller one and the candidate sets are nested; a true
        # neighbour among the candidates is always kept (only true neighbours can rank
        # above it), so recall cannot fall as rounds are added
        assert all(b >= a for a, b in zip(rec, rec[1:])), rec
    print("recall@16 (rows: buckets; columns: rounds 1, 2, 4, 8)")
    for nb, rec in rows:
        print(f"  {nb:5d}: " + "  ".join(f"{r:.3f}" for r in rec))
