"""Pins: facts fixed by the Reformer pages or by mathematics that the oracle must meet.

Each ``pin_*`` takes an oracle front end (``oracle.Oracle``) and raises
AssertionError when the oracle disagrees.  The checks never re-type the
oracle's own formulas: they use printed values (``golden/``), closed forms,
invariants, special cases that reduce to a library routine (numpy argmax and
stable argsort, torch's scaled_dot_product_attention), and brute force on tiny
inputs.  ``test_oracle_pins.py`` runs them on the real oracle and
``test_oracle_mutants.py`` runs them on copies with planted mistakes.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


# --------------------------------------------------------------------------
# Hashing
# --------------------------------------------------------------------------

def pin_hash_is_first_argmax_of_concat(orc):
    """Bucket = first argmax of [xR, -xR] (glossary "Atencion LSH"); numpy's argmax returns
    the first maximal index, and the margin is top-1 minus top-2 of that vector."""
    rng = _rng(1)
    for d, nb in ((8, 2), (16, 8), (64, 32), (128, 96)):
        x = rng.standard_normal((200, d))
        R = rng.standard_normal((d, nb // 2))
        b, m = orc.hash(x, R, nb)
        p = x @ R
        cat = np.concatenate([p, -p], axis=1)
        assert np.array_equal(b, np.argmax(cat, axis=1)), (d, nb)
        srt = np.sort(cat, axis=1)
        assert np.allclose(m, srt[:, -1] - srt[:, -2], rtol=1e-12, atol=1e-12)


def pin_hash_simhash_closed_form(orc):
    """With 2 buckets the hash is the sign of one random projection (SimHash): two vectors at
    angle theta share a bucket with probability 1 - theta/pi.  Monte Carlo, 4 sigma."""
    rng = _rng(2)
    d, n = 16, 20000
    R = rng.standard_normal((n, d, 1))
    e0 = np.zeros(d); e0[0] = 1.0
    for theta in (math.pi / 6, math.pi / 3, math.pi / 2, 2 * math.pi / 3):
        e1 = np.zeros(d); e1[0] = math.cos(theta); e1[1] = math.sin(theta)
        b, _ = orc.hash_rounds(np.stack([e0, e1]), R, 2)
        same = float(np.mean(b[:, 0] == b[:, 1]))
        p = 1.0 - theta / math.pi
        sigma = math.sqrt(p * (1 - p) / n)
        assert abs(same - p) < 4 * sigma + 1e-9, (theta, same, p)


def pin_hash_pages_bucket_sharing_statistic(orc):
    """The glossary's worked example: dim 64, 16 buckets, 1000 rounds; a vector near the
    query (cos 0.96) shares its bucket in 72 % of rounds, an unrelated one (cos 0.04) in 9 %.
    Checked in distribution over our own seeds (tolerance band from the fixture)."""
    with open(os.path.join(GOLDEN, "bucket_sharing.json")) as f:
        g = json.load(f)
    s, band = g["setup"], g["band"]
    near_rates, far_rates = [], []
    for seed in range(band["seeds"]):
        rng = _rng(10_000 + seed)
        q = rng.standard_normal(s["dim"])
        near = q + 0.3 * rng.standard_normal(s["dim"])
        far = rng.standard_normal(s["dim"])
        R = rng.standard_normal((s["rounds"], s["dim"], s["n_buckets"] // 2))
        b, _ = orc.hash_rounds(np.stack([q, near, far]), R, s["n_buckets"])
        near_rates.append(np.mean(b[:, 1] == b[:, 0]))
        far_rates.append(np.mean(b[:, 2] == b[:, 0]))
        assert near_rates[-1] > far_rates[-1], seed
    pn, pf = g["printed"]["near"]["shared_fraction"], g["printed"]["far"]["shared_fraction"]
    assert abs(np.mean(near_rates) - pn) <= band["near_tolerance"], np.mean(near_rates)
    assert abs(np.mean(far_rates) - pf) <= band["far_tolerance"], np.mean(far_rates)


def pin_hash_positive_rescaling(orc):
    """hash(a x) = hash(x) for a > 0: exactly for powers of two (exact scaling in binary
    floating point), and outside a relative near-tie band for other factors."""
    rng = _rng(3)
    x = rng.standard_normal((300, 32))
    R = rng.standard_normal((32, 16))
    b0, m0 = orc.hash(x, R, 32)
    for k in (-6, -1, 1, 5):
        b, _ = orc.hash(x * 2.0 ** k, R, 32)
        assert np.array_equal(b, b0), k
    for a in (0.37, 3.3, 1234.5):
        b, _ = orc.hash(x * a, R, 32)
        safe = m0 > 1e-9 * np.linalg.norm(x, axis=1) * np.linalg.norm(R, axis=0).max()
        assert np.array_equal(b[safe], b0[safe]), a


def pin_hash_zero_rotation(orc):
    """R = 0 makes every entry of [xR, -xR] zero; the first index wins: bucket 0."""
    rng = _rng(4)
    b, m = orc.hash(rng.standard_normal((50, 16)), np.zeros((16, 8)), 16)
    assert np.all(b == 0) and np.all(m == 0)


def pin_hash_antipodal_and_relabel(orc):
    """hash(-x) = hash(x) + nb/2 (mod nb), and permuting R's columns by pi relabels the
    bucket j -> pi^-1(j) in each half (symmetry of the [p, -p] construction)."""
    rng = _rng(5)
    d, nb = 32, 24
    half = nb // 2
    x = rng.standard_normal((400, d))
    R = rng.standard_normal((d, half))
    b, m = orc.hash(x, R, nb)
    bn, _ = orc.hash(-x, R, nb)
    ok = m > 0
    assert np.array_equal(bn[ok], (b[ok] + half) % nb)
    pi = rng.permutation(half)
    bp, _ = orc.hash(x, R[:, pi], nb)
    inv_pi = np.argsort(pi)
    expect = np.where(b < half, inv_pi[b % half], half + inv_pi[b % half])
    assert np.array_equal(bp[ok], expect[ok])


# --------------------------------------------------------------------------
# Sorting
# --------------------------------------------------------------------------

def pin_sort_stable_by_bucket(orc):
    """perm orders positions by (bucket, position): it is a bijection, inv is its inverse,
    it equals numpy's stable argsort, and bstart is the running count of smaller buckets."""
    rng = _rng(6)
    for L, nb in ((1, 4), (17, 2), (1000, 32), (4096, 1024), (3000, 7)):
        bucket = rng.integers(0, nb, size=L).astype(np.int32)
        if L > 50:
            bucket[: L // 3] = rng.integers(0, 2, size=L // 3)   # heavy buckets
        perm, inv, bstart = orc.sort(bucket, nb)
        assert np.array_equal(np.sort(perm), np.arange(L))
        assert np.array_equal(inv[perm], np.arange(L))
        assert np.array_equal(perm, np.argsort(bucket, kind="stable"))
        sb = bucket[perm]
        assert np.all(np.diff(sb) >= 0)
        same = np.diff(sb) == 0
        assert np.all(np.diff(perm)[same] > 0)
        counts = np.bincount(bucket, minlength=nb)
        assert np.array_equal(bstart, np.concatenate([[0], np.cumsum(counts)]))


# --------------------------------------------------------------------------
# Attention
# --------------------------------------------------------------------------

def _sdpa(qk, v, allowed, scale):
    """Shared-QK softmax attention with unit-norm keys through torch's SDPA (fp64).

    Returns (out, lse) with lse from torch.logsumexp of the same masked scores."""
    q = torch.from_numpy(qk)
    k = q / q.norm(dim=-1, keepdim=True)
    m = torch.from_numpy(allowed)
    out = torch.nn.functional.scaled_dot_product_attention(
        q[None], k[None], torch.from_numpy(v)[None], attn_mask=m[None], scale=scale)[0]
    s = (q @ k.T) * scale
    s = s.masked_fill(~m, float("-inf"))
    return out.numpy(), torch.logsumexp(s, dim=-1).numpy()


def _self_masked(allowed_with_self):
    """Remove the diagonal except in rows where it is the only allowed entry."""
    a = allowed_with_self.copy()
    L = a.shape[0]
    diag = np.eye(L, dtype=bool)
    only_self = (a & ~diag).sum(1) == 0
    a &= ~diag
    a[only_self, np.arange(L)[only_self]] = True
    return a, only_self


def _check_rows(orc, out, lse, ref_out, ref_lse, only_self, n_rounds, v):
    assert np.allclose(out[~only_self], ref_out[~only_self], rtol=1e-10, atol=1e-10)
    assert np.allclose(lse[~only_self], ref_lse[~only_self], rtol=1e-10, atol=1e-10)
    if n_rounds == 1:
        assert np.array_equal(out[only_self], v[only_self])
    assert np.allclose(out[only_self], v[only_self], rtol=0, atol=1e-9)
    assert np.allclose(lse[only_self], orc.SELF_LOGIT + math.log(n_rounds), rtol=0, atol=1e-9)


def pin_attention_one_bucket_one_chunk_is_full_attention(orc):
    """With one bucket (R = 0) and one chunk covering the sequence, LSH attention is full
    shared-QK softmax attention with the self-mask, causal or not (library SDPA)."""
    rng = _rng(7)
    L, d = 24, 16
    qk = rng.standard_normal((L, d))
    v = rng.standard_normal((L, d))
    for causal in (False, True):
        for n_rounds, scale in ((1, 0.25), (2, 1.0)):
            R = np.zeros((n_rounds, d, 4))
            out, lse = orc.forward(qk[None], v[None], R, 8, L, causal, scale)
            allowed = np.tril(np.ones((L, L), bool)) if causal else np.ones((L, L), bool)
            allowed, only_self = _self_masked(allowed)
            ref_out, ref_lse = _sdpa(qk, v, allowed, scale)
            _check_rows(orc, out[0], lse[0], ref_out, ref_lse + math.log(n_rounds),
                        only_self, n_rounds, v)


def pin_attention_one_bucket_is_local_lookback_window(orc):
    """With one bucket, sorting is the identity and the method reduces to local attention
    over the own and previous chunk (glossary "Atencion LSH"), no look-ahead, no wrap."""
    rng = _rng(8)
    L, d, c = 40, 8, 8
    qk = rng.standard_normal((L, d))
    v = rng.standard_normal((L, d))
    idx = np.arange(L)
    kq, kk = (idx // c)[:, None], (idx // c)[None, :]
    window = (kk == kq) | (kk == kq - 1)
    for causal in (False, True):
        allowed = window & (idx[None, :] <= idx[:, None]) if causal else window
        allowed, only_self = _self_masked(allowed)
        out, lse = orc.forward(qk[None], v[None], np.zeros((1, d, 2)), 4, c, causal, 0.7)
        ref_out, ref_lse = _sdpa(qk, v, allowed, 0.7)
        _check_rows(orc, out[0], lse[0], ref_out, ref_lse, only_self, 1, v)


def pin_attention_single_candidate_rows(orc):
    """A row with one candidate copies that value exactly; the causal first token has no
    candidate and gets its own value with lse = self logit + ln(rounds)."""
    rng = _rng(9)
    L, d = 16, 8
    qk = rng.standard_normal((L, d))
    v = rng.standard_normal((L, d))
    for n_rounds in (1, 3):
        out, lse = orc.forward(qk[None], v[None], np.zeros((n_rounds, d, 1)), 2, 4, True, 0.5)
        if n_rounds == 1:
            assert np.array_equal(out[0, 0], v[0]) and np.array_equal(out[0, 1], v[0])
        assert np.allclose(out[0, 0], v[0], rtol=0, atol=1e-9)
        assert abs(lse[0, 0] - (orc.SELF_LOGIT + math.log(n_rounds))) < 1e-9
        assert np.allclose(out[0, 1], v[0], rtol=0, atol=1e-12)


def pin_attention_zero_scale_is_candidate_mean(orc):
    """scale = 0 gives equal weights: every row is the plain mean of its candidates'
    values, and lse_r = ln(count); the candidate sets are enumerated by brute force."""
    rng = _rng(10)
    L, d, nb, c = 48, 8, 6, 8
    qk = rng.standard_normal((L, d))
    v = rng.standard_normal((L, d))
    R = rng.standard_normal((1, d, nb // 2))
    for causal in (False, True):
        out, lse, it = orc.forward(qk[None], v[None], R, nb, c, causal, 0.0, intermediates=True)
        bucket = it["bucket"][0, 0]
        for i in range(L):
            cands = _brute_candidates(bucket, i, c, causal)
            if cands:
                assert np.allclose(out[0, i], v[cands].mean(0), rtol=1e-12, atol=1e-12)
                assert abs(lse[0, i] - math.log(len(cands))) < 1e-12
            else:
                assert np.array_equal(out[0, i], v[i])


def _brute_candidates(bucket, i, c, causal):
    """Candidates of token i straight from the definition: rank tokens by (bucket, pos)."""
    order = sorted(range(len(bucket)), key=lambda t: (bucket[t], t))
    s = order.index(i)
    k = s // c
    out = []
    for t in range(max(0, (k - 1) * c), min(len(bucket), (k + 1) * c)):
        j = order[t]
        if j == i or bucket[j] != bucket[i] or (causal and j >= i):
            continue
        out.append(j)
    return out


def pin_attention_brute_force_tiny(orc):
    """For L <= 16, several buckets and rounds: candidate sets enumerated from the definition,
    softmax and round combination evaluated directly with numpy, match the oracle."""
    rng = _rng(11)
    for L, d, nb, c, n_rounds in ((16, 4, 4, 4, 2), (12, 8, 2, 2, 3), (16, 4, 8, 8, 1)):
        for causal in (False, True):
            qk = rng.standard_normal((L, d))
            v = rng.standard_normal((L, d))
            R = rng.standard_normal((n_rounds, d, nb // 2))
            scale = 0.8
            out, lse, it = orc.forward(qk[None], v[None], R, nb, c, causal, scale,
                                       intermediates=True)
            kn = qk / np.linalg.norm(qk, axis=1, keepdims=True)
            for i in range(L):
                ls, os_ = [], []
                for r in range(n_rounds):
                    p = qk[i] @ R[r]
                    bucket = np.argmax(np.concatenate([qk @ R[r], -(qk @ R[r])], 1), 1)
                    assert bucket[i] == np.argmax(np.concatenate([p, -p]))
                    cands = _brute_candidates(bucket, i, c, causal)
                    if not cands:
                        ls.append(orc.SELF_LOGIT); os_.append(v[i]); continue
                    sc = scale * (kn[cands] @ qk[i])
                    w = np.exp(sc - sc.max())
                    ls.append(sc.max() + math.log(w.sum()))
                    os_.append((w[:, None] * v[cands]).sum(0) / w.sum())
                ls = np.array(ls)
                W = np.exp(ls - ls.max())
                ref_lse = ls.max() + math.log(W.sum())
                ref = (W[:, None] * np.array(os_)).sum(0) / W.sum()
                assert np.allclose(out[0, i], ref, rtol=1e-10, atol=1e-10), (L, i, causal)
                assert abs(lse[0, i] - ref_lse) < 1e-9


# --------------------------------------------------------------------------
# Round combination
# --------------------------------------------------------------------------

def pin_combine_identical_rounds(orc):
    """Equal rotations in every round give the single-round output, and the combined lse is
    the single-round lse plus ln(rounds)."""
    rng = _rng(12)
    L, d, nb, c = 64, 8, 8, 8
    qk = rng.standard_normal((2, L, d))
    v = rng.standard_normal((2, L, d))
    R1 = rng.standard_normal((1, d, nb // 2))
    o1, l1 = orc.forward(qk, v, R1, nb, c, True, 0.6)
    for n in (2, 5):
        on, ln = orc.forward(qk, v, np.repeat(R1, n, 0), nb, c, True, 0.6)
        assert np.allclose(on, o1, rtol=1e-9, atol=1e-9)
        assert np.allclose(ln, l1 + math.log(n), rtol=0, atol=1e-9)


def pin_combine_one_round_is_unsort(orc):
    """With one round the combination is the identity: out is the sorted-order output moved
    back to original order (numpy fancy indexing by inv)."""
    rng = _rng(13)
    L, d, nb, c = 64, 8, 8, 8
    qk = rng.standard_normal((1, L, d))
    v = rng.standard_normal((1, L, d))
    R = rng.standard_normal((1, d, nb // 2))
    out, lse, it = orc.forward(qk, v, R, nb, c, False, 0.9, intermediates=True)
    inv = it["inv"][0, 0]
    assert not np.array_equal(inv, np.arange(L))
    assert np.array_equal(out[0], it["o_r"][0, 0][inv])
    assert np.array_equal(lse[0], it["lse_r"][0, 0][inv])


def pin_combine_closed_form_two_rounds(orc):
    """Two rounds with given per-round (o, lse): out = (e^l1 o1 + e^l2 o2) / (e^l1 + e^l2),
    lse = ln(e^l1 + e^l2); includes a self-only round (lse = -1e5) that must get ~0 weight."""
    rng = _rng(14)
    L, d = 5, 3
    o = rng.standard_normal((2, L, d))
    l = np.array([[0.3, 2.0, -1.0, 5.0, 0.0], [1.1, -4.0, -1e5, 5.0, 0.0]])
    inv = np.stack([rng.permutation(L), rng.permutation(L)]).astype(np.int32)
    out, lse = orc.combine(o, l, inv)
    for i in range(L):
        l1, l2 = l[0, inv[0, i]], l[1, inv[1, i]]
        o1, o2 = o[0, inv[0, i]], o[1, inv[1, i]]
        e1, e2 = math.exp(l1), math.exp(l2)
        assert np.allclose(out[i], (e1 * o1 + e2 * o2) / (e1 + e2), rtol=1e-12, atol=1e-12)
        assert abs(lse[i] - math.log(e1 + e2)) < 1e-12


def pin_combine_self_only_round_has_no_weight(orc):
    """Self is attended only when nothing else is left (modulabs-hub notes, "LSH attention"):
    a round in which a token has no candidate must not dilute a round in which it has some.
    Round 1 puts every token in one bucket; in round 2 many tokens are alone in their
    bucket window (found by brute force).  Their output equals the round-1-only output."""
    rng = _rng(15)
    L, d, nb, c = 64, 8, 32, 8
    qk = rng.standard_normal((1, L, d))
    v = rng.standard_normal((1, L, d))
    R2 = rng.standard_normal((d, nb // 2))
    both, _ = orc.forward(qk, v, np.stack([np.zeros((d, nb // 2)), R2]), nb, c, True, 0.5)
    first, _ = orc.forward(qk, v, np.zeros((1, d, nb // 2)), nb, c, True, 0.5)
    p = qk[0] @ R2
    bucket2 = np.argmax(np.concatenate([p, -p], 1), 1)
    lonely = [i for i in range(1, L) if not _brute_candidates(bucket2, i, c, True)]
    assert len(lonely) >= 10
    assert np.allclose(both[0, lonely], first[0, lonely], rtol=0, atol=1e-12)


def pin_combine_is_softmax_over_the_rounds_multiset(orc):
    """Weighting each round by its share of the softmax mass, with no correction for keys
    found in several rounds, is one softmax over the multiset union of the rounds'
    candidate sets: key j carries weight count_ij * exp(s_ij), count_ij = the number of
    rounds in which j is a candidate of i.  Checked against library SDPA with the additive
    mask ln(count_ij), candidate sets enumerated by brute force from the oracle's buckets;
    the rows must include keys counted once and keys counted several times."""
    rng = _rng(16)
    L, d, nb, c, n_rounds, scale = 48, 8, 6, 8, 3, 0.6
    qk = rng.standard_normal((L, d))
    v = rng.standard_normal((L, d))
    R = rng.standard_normal((n_rounds, d, nb // 2))
    for causal in (False, True):
        out, lse, it = orc.forward(qk[None], v[None], R, nb, c, causal, scale,
                                   intermediates=True)
        count = np.zeros((L, L))
        for r in range(n_rounds):
            bucket = it["bucket"][0, r]
            for i in range(L):
                count[i, _brute_candidates(bucket, i, c, causal)] += 1
        rows = count.sum(1) > 0
        assert (count == 1).any() and (count >= 2).any() and rows.sum() >= L - 2
        logc = np.where(count > 0, np.log(np.maximum(count, 1)), -np.inf)
        logc[~rows, np.arange(L)[~rows]] = 0.0        # rows with no candidate: not compared
        q = torch.from_numpy(qk)
        k = q / q.norm(dim=-1, keepdim=True)
        mask = torch.from_numpy(logc)
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[None], k[None], torch.from_numpy(v)[None], attn_mask=mask[None], scale=scale)[0]
        ref_lse = torch.logsumexp((q @ k.T) * scale + mask, dim=-1)
        assert np.allclose(out[0][rows], ref.numpy()[rows], rtol=1e-10, atol=1e-10)
        assert np.allclose(lse[0][rows], ref_lse.numpy()[rows], rtol=1e-10, atol=1e-10)



# --------------------------------------------------------------------------
# Backward pass (gradients of the forward in qk and v, buckets held fixed)
# --------------------------------------------------------------------------

def _fixed_bucket_loss(orc, qk, v, it, c, causal, scale, g_out, g_lse, lse0):
    """sum(g_out * out) + sum(g_lse * (lse - lse0)) of one head, recomputed through the
    oracle's staged attention and combination with the given rounds' buckets and
    permutations.  lse0 (the unperturbed lse) is a constant offset that keeps the
    self-only tokens' lse (about -1e5) from swamping the differences in rounding."""
    o_r, lse_r = [], []
    for r in range(it["bucket"].shape[1]):
        o, l = orc.attend(qk, v, it["bucket"][0, r], it["perm"][0, r], c, causal, scale)
        o_r.append(o)
        lse_r.append(l)
    out, lse = orc.combine(np.stack(o_r), np.stack(lse_r), it["inv"][0])
    return float((g_out * out).sum() + (g_lse * (lse - lse0)).sum())


def pin_backward_matches_finite_differences(orc):
    """Central differences of the (pinned) forward, buckets held fixed, agree with the
    backward in every element of qk and v; the value gradients of each token sum to the
    token's output gradient summed over tokens (each output row's weights sum to one)."""
    rng = _rng(17)
    h = 1e-5
    for L, d, nb, c, n_rounds, causal in ((16, 4, 4, 4, 2, True), (16, 4, 2, 8, 3, False)):
        qk = rng.standard_normal((L, d))
        v = rng.standard_normal((L, d))
        R = rng.standard_normal((n_rounds, d, nb // 2))
        g_out = rng.standard_normal((L, d))
        g_lse = rng.standard_normal(L)
        scale = 0.8
        _, lse0, it = orc.forward(qk[None], v[None], R, nb, c, causal, scale,
                                  intermediates=True)
        lse0 = lse0[0]
        assert lse0[0] < -1e4 or not causal   # causal: token 0 is alone in every round
        dqk, dv = orc.backward(qk[None], v[None], R, nb, c, causal, scale, g_out[None],
                               g_lse[None])
        for name, x, grad in (("qk", qk, dqk[0]), ("v", v, dv[0])):
            fd = np.empty_like(x)
            for idx in np.ndindex(*x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                args_p = (xp, v) if name == "qk" else (qk, xp)
                args_m = (xm, v) if name == "qk" else (qk, xm)
                fd[idx] = (_fixed_bucket_loss(orc, *args_p, it, c, causal, scale, g_out, g_lse, lse0)
                           - _fixed_bucket_loss(orc, *args_m, it, c, causal, scale, g_out, g_lse,
                                                lse0)) / (2 * h)
            assert np.allclose(grad, fd, rtol=1e-7, atol=1e-8), (name, np.abs(grad - fd).max())
        # (a round weight exp(lse_r - LSE) of a token alone in every round subtracts two
        # numbers near -1e5, so it carries about 1e-11 of rounding)
        assert np.allclose(dv[0].sum(0), g_out.sum(0), rtol=0, atol=1e-9)


def pin_backward_matches_autograd_of_the_multiset_softmax(orc):
    """torch autograd of an independent dense formulation: one softmax over the multiset
    union of the rounds' brute-force candidate sets (additive mask ln count_ij), the rounds
    in which a token has no candidate entering as a constant diagonal logit
    self_logit + ln(their number) with value v_i.  Gradients in qk and v of
    sum(g_out * out) + sum(g_lse * lse) must match the oracle's backward."""
    rng = _rng(18)
    L, d, nb, c, n_rounds, scale = 48, 8, 6, 8, 3, 0.6
    qk = rng.standard_normal((L, d))
    v = rng.standard_normal((L, d))
    R = rng.standard_normal((n_rounds, d, nb // 2))
    g_out = rng.standard_normal((L, d))
    g_lse = rng.standard_normal(L)
    for causal in (False, True):
        _, _, it = orc.forward(qk[None], v[None], R, nb, c, causal, scale, intermediates=True)
        count = np.zeros((L, L))
        n_self = np.zeros(L)
        for r in range(n_rounds):
            bucket = it["bucket"][0, r]
            for i in range(L):
                cands = _brute_candidates(bucket, i, c, causal)
                count[i, cands] += 1
                n_self[i] += not cands
        assert n_self.max() >= 1 and (count >= 2).any()
        eye = torch.eye(L, dtype=torch.bool)
        logc = torch.from_numpy(np.where(count > 0, np.log(np.maximum(count, 1)), -np.inf))
        diag = torch.from_numpy(np.where(n_self > 0, orc.SELF_LOGIT + np.log(np.maximum(n_self, 1)),
                                         -np.inf))
        q = torch.tensor(qk, requires_grad=True)
        vv = torch.tensor(v, requires_grad=True)
        k = q / q.norm(dim=-1, keepdim=True)
        logits = torch.where(eye, diag[:, None].expand(L, L), (q @ k.T) * scale + logc)
        out = torch.softmax(logits, dim=-1) @ vv
        lse = torch.logsumexp(logits, dim=-1)
        ((torch.from_numpy(g_out) * out).sum() + (torch.from_numpy(g_lse) * lse).sum()).backward()
        dqk, dv = orc.backward(qk[None], v[None], R, nb, c, causal, scale, g_out[None],
                               g_lse[None])
        assert np.allclose(dqk[0], q.grad.numpy(), rtol=1e-9, atol=1e-10)
        assert np.allclose(dv[0], vv.grad.numpy(), rtol=1e-9, atol=1e-10)



def pin_backward_zero_key_gets_no_key_gradient(orc):
    """A zero row of qk has inverse norm 0 (reading R2): as a key it scores 0 whatever the
    query, so it gets no gradient through its key role, while its query and value roles
    still get theirs.  torch autograd of the dense multiset softmax, with the unit keys
    built from a guarded inverse norm (0 for the zero row), must match the oracle."""
    rng = _rng(19)
    L, d, nb, c, n_rounds, scale = 32, 8, 2, 8, 2, 0.7
    qk = rng.standard_normal((L, d))
    qk[5] = 0.0
    qk[20] = 0.0
    v = rng.standard_normal((L, d))
    R = rng.standard_normal((n_rounds, d, nb // 2))
    g_out = rng.standard_normal((L, d))
    g_lse = rng.standard_normal(L)
    _, _, it = orc.forward(qk[None], v[None], R, nb, c, False, scale, intermediates=True)
    count = np.zeros((L, L))
    n_self = np.zeros(L)
    for r in range(n_rounds):
        for i in range(L):
            cands = _brute_candidates(it["bucket"][0, r], i, c, False)
            count[i, cands] += 1
            n_self[i] += not cands
    assert count[:, 5].sum() > 0 and count[5].sum() > 0   # the zero row plays both roles
    eye = torch.eye(L, dtype=torch.bool)
    logc = torch.from_numpy(np.where(count > 0, np.log(np.maximum(count, 1)), -np.inf))
    diag = torch.from_numpy(np.where(n_self > 0, orc.SELF_LOGIT + np.log(np.maximum(n_self, 1)),
                                     -np.inf))
    q = torch.tensor(qk, requires_grad=True)
    vv = torch.tensor(v, requires_grad=True)
    norm = q.norm(dim=-1, keepdim=True)
    inv = torch.where(norm > 0, 1.0 / torch.where(norm > 0, norm, torch.ones_like(norm)),
                      torch.zeros_like(norm))
    logits = torch.where(eye, diag[:, None].expand(L, L), (q @ (q * inv).T) * scale + logc)
    out = torch.softmax(logits, dim=-1) @ vv
    lse = torch.logsumexp(logits, dim=-1)
    ((torch.from_numpy(g_out) * out).sum() + (torch.from_numpy(g_lse) * lse).sum()).backward()
    dqk, dv = orc.backward(qk[None], v[None], R, nb, c, False, scale, g_out[None], g_lse[None])
    assert np.all(np.isfinite(q.grad.numpy()))
    assert np.allclose(dqk[0], q.grad.numpy(), rtol=1e-9, atol=1e-10)
    assert np.allclose(dv[0], vv.grad.numpy(), rtol=1e-9, atol=1e-10)
    assert np.abs(dqk[0, 5]).max() > 0          # its query role still has a gradient


# --------------------------------------------------------------------------
# LSH bucketing as approximate nearest-neighbour search
# --------------------------------------------------------------------------

def _top_k_numpy(x, i, cands, k):
    """Top k of cands by cosine similarity to x_i (0 for a zero vector), ties to the
    smaller index, padded with (-1, -2)."""
    n = np.linalg.norm(x, axis=1)
    inv = np.where(n > 0, 1.0 / np.where(n > 0, n, 1.0), 0.0)
    cands = np.asarray(sorted(set(int(j) for j in cands)), dtype=np.int64)
    sim = (x[cands] @ x[i]) * inv[i] * inv[cands] if len(cands) else np.zeros(0)
    order = np.lexsort((cands, -sim))[:k]
    idx = np.full(k, -1, np.int64)
    val = np.full(k, -2.0)
    idx[:len(order)] = cands[order]
    val[:len(order)] = sim[order]
    return idx, val


def _knn_inputs(orc, x, R, nb):
    n_rounds = R.shape[0]
    L = len(x)
    b = np.empty((n_rounds, L), np.int32)
    p = np.empty_like(b)
    iv = np.empty_like(b)
    for r in range(n_rounds):
        b[r], _ = orc.hash(x, R[r], nb)
        p[r], iv[r], _ = orc.sort(b[r], nb)
    return b, p, iv


def pin_knn_one_bucket_one_chunk_is_exact_search(orc):
    """One bucket (R = 0) and one chunk: every other token is a candidate, so the LSH
    search equals the exhaustive one, which equals numpy's sort by (-cosine, index).
    Duplicate rows make exact ties; a zero row has similarity 0 with every token."""
    rng = _rng(31)
    L, d, k = 48, 6, 7
    x = rng.standard_normal((L, d))
    x[7] = x[3]
    x[20] = 2.0 * x[3]          # exact in floating point: the same cosine bit for bit
    x[11] = 0.0
    b, p, iv = _knn_inputs(orc, x, np.zeros((2, d, 1)), 2)
    idx, sim = orc.knn(x, b, p, iv, L, k)
    eidx, esim = orc.exact_knn(x, k)
    assert np.array_equal(idx, eidx) and np.array_equal(sim, esim)
    for i in range(L):
        ri, rv = _top_k_numpy(x, i, [j for j in range(L) if j != i], k)
        assert np.array_equal(eidx[i], ri), i
        assert np.allclose(esim[i], rv, rtol=0, atol=1e-12), i
    assert eidx[3][0] == 7 and eidx[3][1] == 20      # the tie goes to the smaller index


def pin_knn_brute_force_tiny(orc):
    """For L <= 16, several buckets and rounds: candidate sets enumerated from the
    definition (rank tokens by (bucket, position), own and previous chunk, no causality),
    united over the rounds and ranked with numpy, match the oracle's search."""
    rng = _rng(32)
    for L, d, nb, c, n_rounds, k in ((16, 4, 4, 4, 3, 5), (12, 8, 2, 2, 2, 3), (16, 4, 8, 8, 4, 9)):
        x = rng.standard_normal((L, d))
        R = rng.standard_normal((n_rounds, d, nb // 2))
        b, p, iv = _knn_inputs(orc, x, R, nb)
        idx, sim = orc.knn(x, b, p, iv, c, k)
        for i in range(L):
            cands = []
            for r in range(n_rounds):
                cands += _brute_candidates(b[r], i, c, False)
            ri, rv = _top_k_numpy(x, i, cands, k)
            assert np.array_equal(idx[i], ri), (L, i)
            assert np.allclose(sim[i], rv, rtol=0, atol=1e-12), (L, i)


def pin_knn_identical_rounds(orc):
    """Equal rotations in every round give the one-round search (a token found in several
    rounds is listed once)."""
    rng = _rng(33)
    L, d, nb, c, k = 256, 8, 16, 32, 6
    x = rng.standard_normal((L, d))
    R1 = rng.standard_normal((1, d, nb // 2))
    one = orc.knn(x, *_knn_inputs(orc, x, R1, nb), c, k)
    four = orc.knn(x, *_knn_inputs(orc, x, np.repeat(R1, 4, 0), nb), c, k)
    assert np.array_equal(one[0], four[0]) and np.array_equal(one[1], four[1])


def pin_knn_recall_rises_with_rounds(orc):
    """The glossary's claim in distribution: LSH finds most of a query's nearest
    neighbours, and more rounds find more.  On the clustered recipe (L = 4096, d = 64,
    64 centres, 64 buckets, chunk 64) recall@8 against the exhaustive search, averaged
    over three seeds, rises with the rounds (1, 2, 4, 8) and exceeds 0.8 at 8 rounds."""
    from lsh_attention_04_b300 import inputs as gen
    L, d, k = 4096, 64, 8
    toks = np.arange(0, L, 32)
    means = []
    for n_rounds in (1, 2, 4, 8):
        w = gen.Workload("knn_pin", 1, 1, L, d, "bf16", 64, n_rounds, 64, False, 64, 0)
        rec = []
        for seed in range(3):
            qk, _, R = gen.make_inputs(w, seed=100 + seed)
            x = qk[0, 0].astype(np.float64)
            idx, _ = orc.knn(x, *_knn_inputs(orc, x, R, 64), 64, k, toks)
            ex, _ = orc.exact_knn(x, k, toks)
            rec.append(np.mean([len(set(idx[t]) & set(ex[t])) / k for t in range(len(toks))]))
        means.append(np.mean(rec))
    assert all(a < b for a, b in zip(means, means[1:])), means
    assert means[-1] > 0.8, means


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
