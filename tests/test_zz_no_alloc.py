"""lsh_bucket_sort_noalloc: the bucket sort for callers that cannot allocate.

Callers inside frameworks with their own allocator, runtimes that forbid allocation
after start-up, or code that must not call cudaMalloc get a sort that takes its scratch
from a fixed array inside the library.  This test calls it through the C ABI twice in a
row, on different problems, and checks each result against lsh_bucket_sort (which uses
a caller workspace).  Sort outputs are integers: they must be identical.  It also checks
that a problem larger than the array is rejected before anything runs.

The file name sorts last so that a run stopping at the first failure has already run
every other test.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import lsh_attention_04_b300 as lsh
from lsh_attention_04_b300 import inputs as gen

pytestmark = pytest.mark.gpu


def _noalloc(lib):
    f = lib.lsh_bucket_sort_noalloc
    P, I = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [P, I, I, I, I, I, P, P, P, P]
    f.restype = I
    return f


def _run_noalloc(f, keys, nb):
    B, H, R, L = keys.shape
    perm = torch.empty_like(keys)
    inv = torch.empty_like(keys)
    bstart = torch.empty((B, H, R, nb + 1), dtype=torch.int32, device=keys.device)
    st = f(ctypes.c_void_p(keys.data_ptr()), B, H, L, nb, R, ctypes.c_void_p(perm.data_ptr()),
           ctypes.c_void_p(inv.data_ptr()), ctypes.c_void_p(bstart.data_ptr()),
           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == lsh.LSH_OK, lsh.lsh_status_string(st)
    return perm, inv, bstart


def test_noalloc_sort_matches_workspace_sort_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lsh_attention_04_b300 import build
    build.build()
    lib = lsh.load()
    f = _noalloc(lib)
    rng = np.random.default_rng(2024)
    cases = [(2, 4, 2, 8256, 128), (1, 8, 8, 65536, 1024)]
    results = []
    for B, H, R, L, nb in cases:
        keys = torch.from_numpy(
            gen.synthetic_buckets(rng, B * H * R, L, nb).reshape(B, H, R, L)).cuda()
        got = _run_noalloc(f, keys, nb)
        ref = lsh.lsh_bucket_sort(keys, nb)
        results.append((got, ref))
    torch.cuda.synchronize()
    for got, ref in results:
        for g, r in zip(got, ref):
            assert torch.equal(g, r)
    # too large for the 8 MiB array: rejected, nothing launched
    keys = torch.zeros((4, 8, 8, 65536), dtype=torch.int32, device="cuda")
    st = f(ctypes.c_void_p(keys.data_ptr()), 4, 8, 65536, 2048, 8, ctypes.c_void_p(keys.data_ptr()),
           ctypes.c_void_p(keys.data_ptr()), ctypes.c_void_p(keys.data_ptr()), None)
    assert st == lsh.LSH_ERR_WORKSPACE_TOO_SMALL
