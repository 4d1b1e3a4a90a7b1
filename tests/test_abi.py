"""The C-ABI library loads, exports every symbol its header declares, and validates
arguments on the host (no GPU needed: every call here fails validation or only
computes sizes, so no kernel is launched)."""
import ctypes
import os
import re
import subprocess

import pytest

import lsh_attention_04_b300 as lsh
from lsh_attention_04_b300 import build as lbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    lbuild.build()
    return lsh.load()


def header_functions():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(lsh_\w+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = header_functions()
    for n in ("lsh_attn_forward", "lsh_hash", "lsh_bucket_sort", "lsh_chunk_attn",
              "lsh_unsort_combine", "lsh_attn_workspace_bytes", "lsh_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in header_functions():
        assert hasattr(lib, n), n
    nm = subprocess.run(["nm", "-D", "--defined-only", lsh.LIB_PATH], capture_output=True,
                        text=True, check=True).stdout
    exported = set(re.findall(r"\bT (lsh_\w+)", nm))
    assert set(header_functions()) <= exported
    assert set(lsh.EXPORTS) == set(header_functions())


def test_library_is_built_for_sm103a_only(lib):
    # the build compiles every source for sm_103a and nothing else (no other arch,
    # no PTX for a JIT fallback)
    from lsh_attention_04_b300 import build as b
    assert b.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert not any("gencode" in f or "arch" in f for f in b.FLAGS)
    assert all(not any("gencode" in f or "arch" in f for f in fl) for fl in b.EXTRA.values())


def test_status_strings(lib):
    assert lsh.lsh_status_string(0) == "LSH_OK"
    assert lsh.lsh_status_string(5) == "LSH_ERR_DEVICE_CHECK"
    assert lsh.lsh_status_string(77) == "LSH_ERR_UNKNOWN"


def test_workspace_sizing(lib):
    f = lib.lsh_attn_workspace_bytes
    n = f(1, 8, 65536, 128, 1024, 8, 64, lsh.LSH_BF16)
    # o_r alone is B*H*R*L*d*2 bytes
    assert n > 1 * 8 * 8 * 65536 * 128 * 2
    assert n % 256 == 0
    assert f(1, 8, 65536, 128, 1024, 8, 64, lsh.LSH_F32) > n
    # invalid or unsupported -> 0
    assert f(1, 1, 100, 64, 32, 1, 64, lsh.LSH_F32) == 0      # L % chunk
    assert f(1, 1, 1024, 64, 31, 1, 32, lsh.LSH_F32) == 0     # odd n_buckets
    assert f(1, 1, 1024, 96, 32, 1, 32, lsh.LSH_F32) == 0     # d
    assert f(1, 1, 1024, 64, 4096, 1, 32, lsh.LSH_F32) == 0   # n_buckets > 2048
    assert f(0, 1, 1024, 64, 32, 1, 32, lsh.LSH_F32) == 0
    assert lib.lsh_chunk_attn_workspace_bytes() >= 256
    assert lib.lsh_bucket_sort_workspace_bytes(1, 1, 1024, 32, 1) >= 256


def test_workspace_layout_is_disjoint(lib):
    args = (8, 8, 4096, 64, 64, 4, 64, lsh.LSH_BF16)
    lay = lsh.lsh_attn_workspace_layout(*args)
    total = lsh.lsh_attn_workspace_bytes(*args)
    SL = 8 * 8 * 4 * 4096
    sizes = dict(buckets=4 * SL, inv_norm=4 * 8 * 8 * 4096, perm=4 * SL, inv=4 * SL,
                 bstart=4 * 8 * 8 * 4 * 65, o_r=2 * SL * 64, lse_r=4 * SL)
    spans = sorted((lay[k], lay[k] + sizes[k]) for k in sizes)
    assert spans[0][0] >= 256
    for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
        assert a1 <= b0
    assert spans[-1][1] <= total
    assert all(lay[k] % 256 == 0 for k in lay)


# The validation tests below pass made-up pointer values.  They are meant to be
# rejected before any CUDA call; on a machine with a GPU a validation bug would hand
# such a pointer to the device, so these tests only run where no GPU exists.
no_device = pytest.mark.skipif(__import__("torch").cuda.is_available(),
                               reason="fake pointers are only passed where no GPU exists")


def _fwd(lib, **kw):
    a = dict(qk=1, v=1, R=1, dtype=lsh.LSH_BF16, B=1, H=1, L=1024, d=64, nb=32, R_=1,
             chunk=64, causal=1, scale=0.125, out=1, lse=1, ws=256, wsb=1 << 30, st=None)
    a.update(kw)
    P = ctypes.c_void_p
    return lib.lsh_attn_forward(P(a["qk"]), P(a["v"]), P(a["R"]), a["dtype"], a["B"], a["H"],
                                a["L"], a["d"], a["nb"], a["R_"], a["chunk"], a["causal"],
                                a["scale"], P(a["out"]), P(a["lse"]), P(a["ws"]), a["wsb"],
                                a["st"])


@pytest.mark.parametrize("kw,expect", [
    (dict(qk=0), lsh.LSH_ERR_INVALID_ARGUMENT),
    (dict(out=0), lsh.LSH_ERR_INVALID_ARGUMENT),
    (dict(ws=0), lsh.LSH_ERR_INVALID_ARGUMENT),
    (dict(ws=4), lsh.LSH_ERR_INVALID_ARGUMENT),          # misaligned workspace
    (dict(L=1000), lsh.LSH_ERR_INVALID_ARGUMENT),        # not a multiple of chunk
    (dict(nb=33), lsh.LSH_ERR_INVALID_ARGUMENT),
    (dict(B=0), lsh.LSH_ERR_INVALID_ARGUMENT),
    (dict(R_=-1), lsh.LSH_ERR_INVALID_ARGUMENT),
    (dict(causal=2), lsh.LSH_ERR_INVALID_ARGUMENT),
    (dict(dtype=7), lsh.LSH_ERR_INVALID_ARGUMENT),
    (dict(d=96), lsh.LSH_ERR_UNSUPPORTED),
    (dict(chunk=256, L=1024), lsh.LSH_ERR_UNSUPPORTED),
    (dict(chunk=128, d=128, dtype=lsh.LSH_F32), lsh.LSH_ERR_UNSUPPORTED),
    (dict(chunk=128, wsb=1024), lsh.LSH_ERR_WORKSPACE_TOO_SMALL),   # chunk 128 passes validation
    (dict(nb=4096), lsh.LSH_ERR_UNSUPPORTED),
    (dict(nb=40), lsh.LSH_ERR_UNSUPPORTED),              # bf16 needs n_buckets % 16 == 0
    (dict(B=1 << 12, H=1 << 12, L=1 << 10, R_=1 << 2), lsh.LSH_ERR_UNSUPPORTED),
    (dict(wsb=1024), lsh.LSH_ERR_WORKSPACE_TOO_SMALL),
])
@no_device
def test_forward_validation(lib, kw, expect):
    assert _fwd(lib, **kw) == expect


@no_device
def test_stage_validation(lib):
    P = ctypes.c_void_p
    # null outputs
    assert lib.lsh_hash(P(1), P(1), lsh.LSH_F32, 1, 1, 64, 64, 32, 1, None, P(1), P(256), 1 << 20,
                        None) == lsh.LSH_ERR_INVALID_ARGUMENT
    assert lib.lsh_bucket_sort(P(1), 1, 1, 64, 32, 1, None, P(1), P(1), P(256), 1 << 20,
                               None) == lsh.LSH_ERR_INVALID_ARGUMENT
    assert lib.lsh_bucket_sort(P(1), 1, 1, 64, 4096, 1, P(1), P(1), P(1), P(256), 1 << 20,
                               None) == lsh.LSH_ERR_UNSUPPORTED
    assert lib.lsh_bucket_sort(P(1), 1, 1, 64, 32, 1, P(1), P(1), P(1), P(256), 8,
                               None) == lsh.LSH_ERR_WORKSPACE_TOO_SMALL
    assert lib.lsh_unsort_combine(P(1), P(1), None, lsh.LSH_F32, 1, 1, 64, 64, 1, P(1), P(1),
                                  None) == lsh.LSH_ERR_INVALID_ARGUMENT
    assert lib.lsh_unsort_combine(P(1), P(1), P(1), lsh.LSH_F32, 1, 1, 64, 32, 1, P(1), P(1),
                                  None) == lsh.LSH_ERR_UNSUPPORTED
    assert lib.lsh_chunk_attn(P(1), P(1), lsh.LSH_F32, P(1), P(1), P(1), P(1), 1, 1, 100, 64, 32,
                              1, 32, 1, ctypes.c_float(1.0), P(1), P(1), P(256), 1 << 20,
                              None) == lsh.LSH_ERR_INVALID_ARGUMENT   # L % chunk
    assert lib.lsh_workspace_status(None, None, None) == lsh.LSH_ERR_INVALID_ARGUMENT
    # bounded-wait self test: needs a 256-byte aligned status block
    assert lib.lsh_selftest_wait_timeout(None, 256, None) == lsh.LSH_ERR_INVALID_ARGUMENT
    assert lib.lsh_selftest_wait_timeout(P(256), 128, None) == lsh.LSH_ERR_INVALID_ARGUMENT
    assert lib.lsh_selftest_wait_timeout(P(260), 256, None) == lsh.LSH_ERR_INVALID_ARGUMENT


def test_backward_workspace_sizing(lib):
    args = (1, 8, 65536, 128, 1024, 8, 64, lsh.LSH_BF16)
    fwd = lib.lsh_attn_workspace_bytes(*args)
    bwd = lib.lsh_attn_backward_workspace_bytes(*args)
    # no per-round outputs (o_r alone is B*H*R*L*d*2 bytes), but buckets, perm, inv, and
    # for bf16 the tensor-core kernel's g_out in bf16 plus one fp32 per token
    n_tok = 8 * 65536
    assert 0 < bwd < fwd - 1 * 8 * 8 * 65536 * 128 * 2 + n_tok * (2 * 128 + 4)
    assert bwd > 3 * 4 * 8 * 8 * 65536 + n_tok * (2 * 128 + 4) and bwd % 256 == 0
    f32 = lib.lsh_attn_backward_workspace_bytes(*args[:-1], lsh.LSH_F32)
    assert f32 < bwd
    assert lib.lsh_attn_backward_workspace_bytes(1, 1, 100, 64, 32, 1, 64, lsh.LSH_F32) == 0


def _bwd(lib, **kw):
    a = dict(qk=0x100, v=0x200, R=0x300, dtype=lsh.LSH_BF16, B=1, H=1, L=1024, d=64, nb=32,
             R_=1, chunk=64, causal=1, scale=0.125, out=0x400, lse=0x500, g_out=0x600, g_lse=0,
             dqk=0x700, dv=0x800, ws=0x1000, wsb=1 << 30, st=None)
    a.update(kw)
    P = ctypes.c_void_p
    return lib.lsh_attn_backward(P(a["qk"]), P(a["v"]), P(a["R"]), a["dtype"], a["B"], a["H"],
                                 a["L"], a["d"], a["nb"], a["R_"], a["chunk"], a["causal"],
                                 a["scale"], P(a["out"]), P(a["lse"]), P(a["g_out"]),
                                 P(a["g_lse"]), P(a["dqk"]), P(a["dv"]), P(a["ws"]), a["wsb"],
                                 a["st"])


@pytest.mark.parametrize("kw,expect", [
    (dict(qk=0), lsh.LSH_ERR_INVALID_ARGUMENT),
    (dict(out=0), lsh.LSH_ERR_INVALID_ARGUMENT),
    (dict(lse=0), lsh.LSH_ERR_INVALID_ARGUMENT),
    (dict(g_out=0), lsh.LSH_ERR_INVALID_ARGUMENT),
    (dict(dqk=0), lsh.LSH_ERR_INVALID_ARGUMENT),
    (dict(dv=0), lsh.LSH_ERR_INVALID_ARGUMENT),
    (dict(ws=0), lsh.LSH_ERR_INVALID_ARGUMENT),
    (dict(ws=4), lsh.LSH_ERR_INVALID_ARGUMENT),          # misaligned workspace
    (dict(L=1000), lsh.LSH_ERR_INVALID_ARGUMENT),        # not a multiple of chunk
    (dict(causal=2), lsh.LSH_ERR_INVALID_ARGUMENT),
    (dict(d=96), lsh.LSH_ERR_UNSUPPORTED),
    (dict(chunk=128, L=1024), lsh.LSH_ERR_UNSUPPORTED),
    (dict(nb=40), lsh.LSH_ERR_UNSUPPORTED),
    (dict(wsb=1024), lsh.LSH_ERR_WORKSPACE_TOO_SMALL),
    (dict(g_out=0x604), lsh.LSH_ERR_INVALID_ARGUMENT),   # bf16: 16-byte aligned gradients
    (dict(dv=0x804), lsh.LSH_ERR_INVALID_ARGUMENT),
    (dict(g_out=0x604, dtype=lsh.LSH_F32, wsb=1024), lsh.LSH_ERR_WORKSPACE_TOO_SMALL),
    (dict(chunk=128), lsh.LSH_ERR_UNSUPPORTED),
])
@no_device
def test_backward_validation(lib, kw, expect):
    assert _bwd(lib, **kw) == expect


@no_device
def test_backward_timed_needs_four_events(lib):
    P = ctypes.c_void_p
    ev = (ctypes.c_void_p * 4)(1, 1, 0, 1)
    args = [P(1), P(1), P(1), lsh.LSH_BF16, 1, 1, 1024, 64, 32, 1, 64, 1, ctypes.c_float(0.125),
            P(1), P(1), P(1), None, P(1), P(1), P(256), 1 << 30, None]
    assert lib.lsh_attn_backward_timed(*args, None) == lsh.LSH_ERR_INVALID_ARGUMENT
    assert lib.lsh_attn_backward_timed(*args, ev) == lsh.LSH_ERR_INVALID_ARGUMENT


def test_knn_workspace_sizing(lib):
    f = lib.lsh_knn_workspace_bytes
    n = f(1, 8, 65536, 128, 1024, 8, 64, 16, lsh.LSH_BF16)
    # the per-round candidate lists alone are B*H*R*L*k*(4 + 4) bytes
    assert n > 1 * 8 * 8 * 65536 * 16 * 8 and n % 256 == 0
    assert f(1, 1, 1024, 64, 32, 2, 64, 0, lsh.LSH_BF16) == 0      # k < 1
    assert f(1, 1, 1024, 64, 32, 2, 64, 33, lsh.LSH_BF16) == 0     # k > 32
    assert f(1, 1, 1024, 64, 32, 16, 64, 32, lsh.LSH_BF16) == 0    # rounds * k > 256
    assert f(1, 1, 1000, 64, 32, 2, 64, 8, lsh.LSH_BF16) == 0      # L % chunk
    assert f(1, 1, 1024, 64, 32, 2, 64, 8, lsh.LSH_F16) == 0       # fp16: not taken


@no_device
@pytest.mark.parametrize("kw,expect", [
    (dict(qk=0), lsh.LSH_ERR_INVALID_ARGUMENT),
    (dict(idx=0), lsh.LSH_ERR_INVALID_ARGUMENT),
    (dict(ws=4), lsh.LSH_ERR_INVALID_ARGUMENT),
    (dict(k=0), lsh.LSH_ERR_INVALID_ARGUMENT),
    (dict(k=40), lsh.LSH_ERR_INVALID_ARGUMENT),
    (dict(d=96), lsh.LSH_ERR_UNSUPPORTED),
    (dict(dtype=lsh.LSH_F16), lsh.LSH_ERR_UNSUPPORTED),
    (dict(dtype=3), lsh.LSH_ERR_INVALID_ARGUMENT),
    (dict(chunk=128), lsh.LSH_ERR_UNSUPPORTED),
    (dict(wsb=256), lsh.LSH_ERR_WORKSPACE_TOO_SMALL),
])
def test_knn_argument_checks(lib, kw, expect):
    a = dict(qk=1, R=1, dtype=lsh.LSH_BF16, B=1, H=1, L=1024, d=64, nb=32, R_=2, chunk=64, k=8,
             idx=1, sim=1, ws=256, wsb=1 << 30)
    a.update(kw)
    P = ctypes.c_void_p
    st = lib.lsh_knn(P(a["qk"]), P(a["R"]), a["dtype"], a["B"], a["H"], a["L"], a["d"], a["nb"],
                     a["R_"], a["chunk"], a["k"], P(a["idx"]), P(a["sim"]), P(a["ws"]), a["wsb"],
                     None)
    assert st == expect


def test_revblock_workspace_sizing(lib):
    f = lib.lsh_revblock_workspace_bytes
    n = f(1, 65536, 1024, 8, 4096, 1024, 8, 64, 4096)
    # the attention's own workspace plus qk, v (bf16), the attention output (fp32), two
    # bf16 copies of the stream and one chunk of the hidden layer
    M = 65536
    assert n > lib.lsh_attn_workspace_bytes(1, 8, M, 128, 1024, 8, 64, lsh.LSH_BF16) + \
        M * 1024 * (2 + 2 + 4 + 2 + 2) + 4096 * 4096 * 2
    assert n % 256 == 0
    assert f(1, 1024, 192, 2, 512, 32, 2, 64, 256) == 0     # d_model % 128
    assert f(1, 1024, 256, 2, 500, 32, 2, 64, 256) == 0     # d_ff % 128
    assert f(1, 1024, 256, 3, 512, 32, 2, 64, 256) == 0     # d_model % heads
    assert f(1, 1024, 256, 2, 512, 32, 2, 64, 0) == 0       # ff_chunk
    assert f(1, 1024, 384, 4, 512, 32, 2, 64, 256) == 0     # head size 96
    assert f(1, 1000, 256, 2, 512, 32, 2, 64, 256) == 0     # L % chunk


def test_revblock_layout(lib):
    lay = lsh.lsh_revblock_workspace_layout(2, 1024, 256, 2, 512, 32, 4, 64, 300)
    n = lib.lsh_revblock_workspace_bytes(2, 1024, 256, 2, 512, 32, 4, 64, 300)
    assert lay["attn_ws"] >= 256 and all(v % 256 == 0 for v in lay.values())
    assert lay["attn_ws"] < lay["qk"] < lay["v"] < lay["attn_out"] < lay["merged"] < n


@no_device
@pytest.mark.parametrize("fn", ["lsh_revblock_forward", "lsh_revblock_inverse"])
@pytest.mark.parametrize("kw,expect", [
    (dict(x1=0), lsh.LSH_ERR_INVALID_ARGUMENT),
    (dict(W1=0), lsh.LSH_ERR_INVALID_ARGUMENT),
    (dict(b2=0x104), lsh.LSH_ERR_INVALID_ARGUMENT),       # misaligned
    (dict(y2=0x100), lsh.LSH_ERR_INVALID_ARGUMENT),       # the same array as x1
    (dict(ws=0x110), lsh.LSH_ERR_INVALID_ARGUMENT),
    (dict(dm=192), lsh.LSH_ERR_INVALID_ARGUMENT),
    (dict(causal=2), lsh.LSH_ERR_INVALID_ARGUMENT),
    (dict(wsb=256), lsh.LSH_ERR_WORKSPACE_TOO_SMALL),
])
def test_revblock_argument_checks(lib, fn, kw, expect):
    a = dict(x1=0x100, x2=0x200, Wqk=0x300, Wv=0x400, Wo=0x500, W1=0x600, b1=0x700, W2=0x800,
             b2=0x900, R=0xa00, B=1, L=1024, dm=256, H=2, dff=512, nb=32, R_=2, chunk=64,
             causal=1, ff_chunk=256, y1=0xb00, y2=0xc00, ws=0x1000, wsb=1 << 30)
    a.update(kw)
    P = ctypes.c_void_p
    st = getattr(lib, fn)(
        *[P(a[k]) for k in ("x1", "x2", "Wqk", "Wv", "Wo", "W1", "b1", "W2", "b2", "R")],
        a["B"], a["L"], a["dm"], a["H"], a["dff"], a["nb"], a["R_"], a["chunk"], a["causal"],
        ctypes.c_float(0.125), a["ff_chunk"], P(a["y1"]), P(a["y2"]), P(a["ws"]), a["wsb"], None)
    assert st == expect


@no_device
@pytest.mark.parametrize("kw,expect", [
    (dict(A=0), lsh.LSH_ERR_INVALID_ARGUMENT),
    (dict(A=0x108), lsh.LSH_ERR_INVALID_ARGUMENT),            # misaligned
    (dict(of=0, ob=0), lsh.LSH_ERR_INVALID_ARGUMENT),         # no output
    (dict(relu=2), lsh.LSH_ERR_INVALID_ARGUMENT),
    (dict(M=0), lsh.LSH_ERR_INVALID_ARGUMENT),
    (dict(sL=64, sd=0), lsh.LSH_ERR_INVALID_ARGUMENT),
    (dict(sL=100, sd=64), lsh.LSH_ERR_INVALID_ARGUMENT),      # M % split_L
    (dict(sL=64, sd=48), lsh.LSH_ERR_INVALID_ARGUMENT),       # split_d % 32
    (dict(sL=64, sd=64, ob=0), lsh.LSH_ERR_INVALID_ARGUMENT),  # split needs the bf16 output
    (dict(ws=0x180), lsh.LSH_ERR_INVALID_ARGUMENT),
    (dict(N=200), lsh.LSH_ERR_UNSUPPORTED),
    (dict(K=96), lsh.LSH_ERR_UNSUPPORTED),
    (dict(wsb=128), lsh.LSH_ERR_WORKSPACE_TOO_SMALL),
])
def test_gemm_argument_checks(lib, kw, expect):
    a = dict(A=0x100, W=0x200, M=256, N=256, K=128, bias=0x300, relu=0, res=0, of=0x400,
             ob=0x500, sL=0, sd=0, ws=0x1000, wsb=256)
    a.update(kw)
    P = ctypes.c_void_p
    st = lib.lsh_gemm_bf16(P(a["A"]), P(a["W"]), a["M"], a["N"], a["K"], P(a["bias"]), a["relu"],
                           P(a["res"]), ctypes.c_float(1.0), P(a["of"]), P(a["ob"]), a["sL"],
                           a["sd"], P(a["ws"]), a["wsb"], None)
    assert st == expect


def test_f16_workspace_matches_bf16(lib):
    """fp16 inputs keep bf16 per-round rows: the same workspace as bf16."""
    args = (1, 8, 65536, 128, 1024, 8, 64)
    assert lib.lsh_attn_workspace_bytes(*args, lsh.LSH_F16) == \
        lib.lsh_attn_workspace_bytes(*args, lsh.LSH_BF16)
    assert lib.lsh_attn_workspace_bytes(1, 1, 1024, 64, 40, 1, 64, lsh.LSH_F16) == 0   # nb % 16
    assert lib.lsh_attn_workspace_bytes(1, 1, 1024, 64, 32, 1, 64, 3) == 0


def test_chunk128_scope(lib):
    """Chunk 128: the forward pass only, and not fp32 rows at d = 128."""
    f = lib.lsh_attn_workspace_bytes
    assert f(1, 1, 1024, 64, 16, 2, 128, lsh.LSH_F32) > 0
    assert f(1, 1, 1024, 128, 16, 2, 128, lsh.LSH_BF16) > 0
    assert f(1, 1, 1024, 128, 16, 2, 128, lsh.LSH_F32) == 0
    assert f(1, 1, 1024, 64, 16, 2, 256, lsh.LSH_BF16) == 0
    assert lib.lsh_attn_backward_workspace_bytes(1, 1, 1024, 64, 16, 2, 128, lsh.LSH_BF16) == 0
    assert lib.lsh_knn_workspace_bytes(1, 1, 1024, 64, 16, 2, 128, 8, lsh.LSH_BF16) == 0
