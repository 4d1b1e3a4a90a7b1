"""The reversible residual block on the GPU, through the C ABI, against the oracle.

Forward, stage by stage, each stage fed the GPU's own input to it (read back from the
block's workspace), so every comparison has a derived bound:
  * the per-head projections qk = bf16(x2) Wqk^T and v (bf16 outputs of an fp32
    accumulation): each value must be a bf16 rounding of some number within the
    accumulation error bound ACC of the exact product;
  * the hash of the GPU's qk against the oracle's (near-tie rule), the sort bit-exact, and
    the attention output against the oracle's attention and combination on the GPU's
    buckets, within the attention's bf16 tolerance;
  * the merged heads equal to the bf16 rounding of the attention output, bit for bit;
  * y1 = x1 + merged Wo^T and y2 = x2 + FeedForward(y1) (fp32) within ACC plus the final
    rounding; the hidden layer is a bf16 rounding inside an interval (as the projections),
    and its width carries into y2's bound.
ACC: the accumulation error bound of tests/parity.py (acc_bound).

The whole block is also compared with the oracle's reversible block (fp64, rounding to
bf16 where the GPU does): outside the rare tokens that a rounding or near-tie difference
moves to another bucket, the outputs agree within the attention's tolerance.

Inverse: x2' = y2 - FeedForward(y1) and x1' = y1 - Attention(x2') bit for bit, where
FeedForward(y1) and Attention(x2') come from forward calls with the other half of the
stream zero; x2' = x2 up to the rounding of the two fp32 additions; and x1' = x1 within
the attention's tolerance wherever the attention saw the same buckets and windows in the
forward and the inverse (x2' and x2 can round to different bf16 values, and a near-tie
token can then land in another bucket).
"""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from oracle import reversible as orev
import lsh_attention_04_b300 as lsh
from lsh_attention_04_b300 import inputs as gen
from tests import parity as P

pytestmark = pytest.mark.gpu

BW = gen.BlockWorkload
CASES = [
    BW("block_B2_L1024_dm256_H2_ff512_R4_ffc300", 2, 1024, 256, 2, 512, 32, 4, 64, True, 300, 61),
    BW("block_B2_L2048_dm256_H4_ff1024_R2_noncausal", 2, 2048, 256, 4, 1024, 64, 2, 64, False,
       4096, 62),
    BW("block_B1_L512_dm128_H1_ff384_R8_c32_ffc100", 1, 512, 128, 1, 384, 16, 8, 32, True, 100, 63),
    BW("block_B1_L1088_dm512_H4_ff640_R3_ragged", 1, 1088, 512, 4, 640, 32, 3, 32, True, 1088, 64),
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lsh_attention_04_b300 import build
    build.build()
    lsh.load()


def _device(inp):
    out = {}
    for k, a in inp.items():
        t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
        out[k] = t.to(torch.bfloat16) if k in ("Wqk", "Wv", "Wo", "W1", "W2", "R") else t
    return out


def _forward(w, d, x1, x2, ws=None):
    return lsh.lsh_revblock_forward(x1, x2, d, w.heads, w.n_buckets, w.chunk, w.causal, w.scale,
                                    w.ff_chunk, ws=ws)


def _inverse(w, d, y1, y2, ws=None):
    return lsh.lsh_revblock_inverse(y1, y2, d, w.heads, w.n_buckets, w.chunk, w.causal, w.scale,
                                    w.ff_chunk, ws=ws)


def _workspace(w):
    return lsh.revblock_workspace(w.B, w.L, w.d_model, w.heads, w.d_ff, w.n_buckets, w.n_rounds,
                                  w.chunk, w.ff_chunk)


def _intermediates(w, ws):
    """The block's intermediates of the last call, as numpy arrays (fp64)."""
    lay = lsh.lsh_revblock_workspace_layout(w.B, w.L, w.d_model, w.heads, w.d_ff, w.n_buckets,
                                            w.n_rounds, w.chunk, w.ff_chunk)
    n = w.B * w.L * w.d_model

    def view(off, nbytes, dt):
        return ws[off: off + nbytes].view(dt).double().cpu().numpy()

    shp = (w.B, w.heads, w.L, w.d)
    out = dict(qk=view(lay["qk"], 2 * n, torch.bfloat16).reshape(shp),
               v=view(lay["v"], 2 * n, torch.bfloat16).reshape(shp),
               attn_out=view(lay["attn_out"], 4 * n, torch.float32).reshape(shp),
               merged=view(lay["merged"], 2 * n, torch.bfloat16).reshape(w.B * w.L, w.d_model))
    alay = lsh.lsh_attn_workspace_layout(w.B, w.heads, w.L, w.d, w.n_buckets, w.n_rounds, w.chunk,
                                         lsh.LSH_BF16)
    nr = w.B * w.heads * w.n_rounds * w.L
    for k in ("buckets", "perm", "inv"):
        o = lay["attn_ws"] + alay[k]
        out[k] = ws[o: o + 4 * nr].view(torch.int32).cpu().numpy().reshape(
            w.B * w.heads, w.n_rounds, w.L)
    return out


def check_attention(w, g, case):
    """The hash, sort and attention of the block's attention step on the GPU's qk, v."""
    nh = w.B * w.heads
    qk = g["qk"].reshape(nh, w.L, w.d)
    v = g["v"].reshape(nh, w.L, w.d)
    R = gen.make_block_inputs(w)["R"]
    xn = np.linalg.norm(qk, axis=2)
    Rn = P.r_norm(R)
    n_bad = 0
    out = g["attn_out"].reshape(nh, w.L, w.d)
    worst = 0.0
    for h in range(nh):
        ob, om = oracle.hash_rounds(qk[h].astype(np.float32), R, w.n_buckets)
        n_bad += P.check_buckets(g["buckets"][h], ob, om, xn[h], Rn)
        o_r = np.zeros((w.n_rounds, w.L, w.d))
        l_r = np.zeros((w.n_rounds, w.L))
        for r in range(w.n_rounds):
            perm, inv, _ = oracle.sort(g["buckets"][h, r], w.n_buckets)
            assert np.array_equal(g["perm"][h, r], perm) and np.array_equal(g["inv"][h, r], inv)
            o_r[r], l_r[r] = oracle.attend(qk[h].astype(np.float32), v[h].astype(np.float32),
                                           g["buckets"][h, r], perm, w.chunk, w.causal, w.scale)
        co, _ = oracle.combine(o_r, l_r, g["inv"][h])
        worst = max(worst, P.check_close(out[h], co, P.TOL_OUT["bf16"], "attention output"))
    P.record_near_ties(case, n_bad, nh * w.n_rounds * w.L)
    return worst


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_revblock_forward_stages(w):
    inp = gen.make_block_inputs(w)
    d = _device(inp)
    ws = _workspace(w)
    y1, y2 = _forward(w, d, d["x1"], d["x2"], ws)
    torch.cuda.synchronize()
    assert lsh.lsh_workspace_status(ws) == (lsh.LSH_OK, 0)
    y1, y2 = y1.double().cpu().numpy(), y2.double().cpu().numpy()
    assert np.isfinite(y1).all() and np.isfinite(y2).all()
    g = _intermediates(w, ws)
    f64 = {k: a.astype(np.float64) for k, a in inp.items()}
    M, dm = w.B * w.L, w.d_model

    def heads_to_rows(a):          # [B][H][L][d] -> [B*L][d_model]
        return a.transpose(0, 2, 1, 3).reshape(M, dm)

    # projections
    X = gen.round_bf16(inp["x2"]).astype(np.float64).reshape(M, dm)
    amb = []
    for name, W in (("qk", f64["Wqk"]), ("v", f64["Wv"])):
        lo, hi = P.bf16_interval(X, W)
        amb.append(P.check_bf16_in(heads_to_rows(g[name]), lo, hi, name))
    # attention on the GPU's projections and buckets
    att = check_attention(w, g, w.name)
    # head merge: the bf16 rounding of the attention output, bit for bit
    want = gen.round_bf16(heads_to_rows(g["attn_out"]).astype(np.float32))
    assert np.array_equal(g["merged"], want)
    # y1 = x1 + merged Wo^T
    e1 = P.check_residual(y1.reshape(M, dm), f64["x1"].reshape(M, dm), g["merged"], f64["Wo"],
                        None, "y1")
    # y2 = x2 + relu(bf16(y1) W1^T + b1) W2^T + b2, the hidden layer in bf16
    Y = gen.round_bf16(y1.astype(np.float32)).astype(np.float64).reshape(M, dm)
    lo, hi = P.bf16_interval(Y, f64["W1"], f64["b1"], relu=True)
    mid = 0.5 * (lo + hi)
    extra = 0.5 * (hi - lo) @ np.abs(f64["W2"]).T
    e2 = P.check_residual(y2.reshape(M, dm), f64["x2"].reshape(M, dm), mid, f64["W2"], f64["b2"],
                        "y2", extra + P.acc_bound(w.d_ff) * (0.5 * (hi - lo)) @ np.abs(f64["W2"]).T)
    print(f"{w.name}: ambiguous projection roundings {max(amb):.3%}, attention err {att:.2e}, "
          f"y1 err {e1:.2e}, y2 err {e2:.2e}")


def _oracle_params(w, inp):
    p = {k: inp[k].astype(np.float64) for k in ("Wqk", "Wv", "Wo", "W1", "b1", "W2", "b2", "R")}
    p.update(heads=w.heads, n_buckets=w.n_buckets, chunk=w.chunk, causal=w.causal,
             scale=w.scale, ff_chunk=w.ff_chunk)
    return p


def _q16(a):
    return gen.round_bf16(np.asarray(a, np.float32)).astype(np.float64)


@pytest.mark.parametrize("w", CASES[:3], ids=[c.name for c in CASES[:3]])
def test_revblock_forward_vs_oracle_block(w):
    """The whole block against the oracle's (which hashes its own fp64 projections)."""
    inp = gen.make_block_inputs(w)
    d = _device(inp)
    y1, y2 = _forward(w, d, d["x1"], d["x2"])
    torch.cuda.synchronize()
    o1, o2 = orev.forward(inp["x1"].astype(np.float64), inp["x2"].astype(np.float64),
                          _oracle_params(w, inp), q16=_q16)
    M = w.B * w.L
    tol = P.TOL_OUT["bf16"]
    rows_bad = 0
    for g_, o_ in ((y1, o1), (y2, o2)):
        err = np.abs(g_.double().cpu().numpy() - o_).reshape(M, -1).max(axis=1)
        rows_bad = max(rows_bad, int((err > tol).sum()))
    print(f"{w.name}: {rows_bad} of {M} positions beyond {tol} of the oracle's block")
    # a token moved to another bucket changes the attention of its bucket's neighbours;
    # the rounding differences that can move one are rare
    assert rows_bad <= max(4, M // 200)


def check_x1_recovered(w, x1, x1r, ws_f, ws_i):
    """x1' - x1 = Attention(x2) - Attention(x2'), two evaluations of the bf16 attention on
    inputs equal up to fp32 rounding: within the attention's tolerance at every position
    whose windows and buckets were the same in both evaluations (every head and round);
    the positions beyond it must all be ones where a rounding moved a token to another
    bucket.  Returns (positions beyond the tolerance, positions not comparable)."""
    g_f, g_i = _intermediates(w, ws_f), _intermediates(w, ws_i)
    ok = P.comparable_tokens(w.chunk, g_i["buckets"], g_f["buckets"], g_i["perm"], g_f["perm"],
                             g_i["inv"], g_f["inv"])
    pos_ok = ok.reshape(w.B, w.heads, w.L).all(axis=1)
    err = (x1r.double() - x1.double()).abs().amax(dim=2).cpu().numpy()
    beyond = err > P.TOL_OUT["bf16"]
    assert not (beyond & pos_ok).any(), (
        f"x1 off by {err[pos_ok].max():.3e} at a position with unchanged attention windows")
    return int(beyond.sum()), int((~pos_ok).sum())


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_revblock_inverse(w):
    inp = gen.make_block_inputs(w)
    d = _device(inp)
    ws_f, ws_i = _workspace(w), _workspace(w)
    y1, y2 = _forward(w, d, d["x1"], d["x2"], ws_f)
    x1r, x2r = _inverse(w, d, y1, y2, ws_i)
    zeros = torch.zeros_like(y1)
    y1_again, F = _forward(w, d, y1, zeros)          # = (y1, FeedForward(y1))
    A, _ = _forward(w, d, zeros, x2r)                # = (Attention(x2'), ...)
    torch.cuda.synchronize()
    assert lsh.lsh_workspace_status(ws_i) == (lsh.LSH_OK, 0)
    assert torch.equal(y1_again, y1), "Attention(0) must add exactly zero"
    assert torch.equal(x2r, y2 - F), "x2' = y2 - FeedForward(y1)"
    assert torch.equal(x1r, y1 - A), "x1' = y1 - Attention(x2')"
    bound2 = 2.0 ** -23 * (y2.double().abs() + d["x2"].double().abs())
    assert ((x2r.double() - d["x2"].double()).abs() <= bound2).all()
    n_beyond, n_moved = check_x1_recovered(w, d["x1"], x1r, ws_f, ws_i)
    flips = int((x2r.to(torch.bfloat16) != d["x2"].to(torch.bfloat16)).sum())
    print(f"{w.name}: {flips} entries of x2' round to another bf16 value than x2's; "
          f"{n_moved} positions with moved windows, {n_beyond} beyond tolerance")


def test_revblock_ff_chunk_invariance():
    """Chunking the feed-forward over positions changes nothing: ff_chunk = 1 (every
    product one row), 37 and all positions give identical outputs."""
    base = BW("block_B1_L128_dm128_H2_ff256_R1", 1, 128, 128, 2, 256, 16, 1, 64, True, 128, 65)
    inp = gen.make_block_inputs(base)
    d = _device(inp)
    outs = []
    for c in (1, 37, 128):
        w = dataclasses.replace(base, ff_chunk=c)
        outs.append(_forward(w, d, d["x1"], d["x2"]))
    torch.cuda.synchronize()
    for y1, y2 in outs[1:]:
        assert torch.equal(y1, outs[0][0]) and torch.equal(y2, outs[0][1])


def test_revblock_full_size_sampled():
    """The long-text block (L = 65536, d_model 1024, 8 heads of 128, d_ff 4096, 8 rounds,
    1024 buckets, feed-forward chunks of 8192 positions) as the benchmark runs it: forward
    and inverse, the stages checked on 256 sampled positions (the attention on one head)."""
    w = gen.BLOCK_LONG
    inp = gen.make_block_inputs(w)
    d = _device(inp)
    ws = _workspace(w)
    y1, y2 = _forward(w, d, d["x1"], d["x2"], ws)
    torch.cuda.synchronize()
    assert lsh.lsh_workspace_status(ws) == (lsh.LSH_OK, 0)
    assert torch.isfinite(y1).all() and torch.isfinite(y2).all()
    g = _intermediates(w, ws)
    f64 = {k: a.astype(np.float64) for k, a in inp.items() if k not in ("x1", "x2")}
    M, dm = w.B * w.L, w.d_model
    rng = np.random.default_rng(7)
    rows = np.sort(rng.choice(M, 256, replace=False))
    X = gen.round_bf16(inp["x2"].reshape(M, dm)[rows]).astype(np.float64)
    qk_rows = g["qk"].transpose(0, 2, 1, 3).reshape(M, dm)[rows]
    lo, hi = P.bf16_interval(X, f64["Wqk"])
    P.check_bf16_in(qk_rows, lo, hi, "qk")
    merged = g["merged"][rows]
    assert np.array_equal(merged, gen.round_bf16(
        g["attn_out"].transpose(0, 2, 1, 3).reshape(M, dm)[rows].astype(np.float32)))
    y1n = y1.double().cpu().numpy().reshape(M, dm)
    P.check_residual(y1n[rows], inp["x1"].reshape(M, dm)[rows].astype(np.float64), merged,
                   f64["Wo"], None, "y1")
    Y = gen.round_bf16(y1n[rows].astype(np.float32)).astype(np.float64)
    lo, hi = P.bf16_interval(Y, f64["W1"], f64["b1"], relu=True)
    mid = 0.5 * (lo + hi)
    extra = (1 + P.acc_bound(w.d_ff)) * (0.5 * (hi - lo)) @ np.abs(f64["W2"]).T
    P.check_residual(y2.double().cpu().numpy().reshape(M, dm)[rows],
                   inp["x2"].reshape(M, dm)[rows].astype(np.float64), mid, f64["W2"], f64["b2"],
                   "y2", extra)
    # attention of one head on sampled tokens, on the GPU's buckets
    h = 3
    qk = g["qk"][0, h].astype(np.float32)
    v = g["v"][0, h].astype(np.float32)
    toks = np.sort(rng.choice(w.L, 256, replace=False))
    o_r = np.zeros((w.n_rounds, w.L, w.d))
    l_r = np.zeros((w.n_rounds, w.L))
    for r in range(w.n_rounds):
        perm, inv, _ = oracle.sort(g["buckets"][h, r], w.n_buckets)
        assert np.array_equal(g["perm"][h, r], perm)
        sel = np.unique(inv[toks])
        ro, rl = oracle.attend(qk, v, g["buckets"][h, r], perm, w.chunk, w.causal, w.scale,
                               rows=sel)
        o_r[r][sel], l_r[r][sel] = ro, rl
    co, _ = oracle.combine(o_r, l_r, g["inv"][h], tokens=toks)
    P.check_close(g["attn_out"][0, h][toks], co, P.TOL_OUT["bf16"], "attention output")
    # the inverse at full size, in its own workspace
    del g
    ws_i = _workspace(w)
    x1r, x2r = _inverse(w, d, y1, y2, ws_i)
    torch.cuda.synchronize()
    assert lsh.lsh_workspace_status(ws_i) == (lsh.LSH_OK, 0)
    bound2 = 2.0 ** -23 * (y2.abs() + d["x2"].abs())
    assert ((x2r - d["x2"]).abs() <= bound2).all()
    n_beyond, n_moved = check_x1_recovered(w, d["x1"], x1r, ws, ws_i)
    print(f"long block inverse: {n_moved} of {M} positions with moved windows, "
          f"{n_beyond} beyond tolerance")
    # at this length the roundings of x2' move a few tokens to other buckets in almost
    # every head and round, which shifts the sorted order and so nearly every window by
    # a position; the recovery is then statistical
    assert n_beyond <= M // 100
    # the inverse's own arithmetic, bit for bit
    zeros = torch.zeros_like(y1)
    y1_again, F = _forward(w, d, y1, zeros, ws)
    assert torch.equal(y1_again, y1) and torch.equal(x2r, y2 - F)
    del y1_again, F
    A, _ = _forward(w, d, zeros, x2r, ws)
    assert torch.equal(x1r, y1 - A)
