"""Failure reporting on the GPU: a bounded wait that runs out reports, it does not hang.

Every wait in the tensor-core kernels goes through one bounded wait.  The library's self
test makes one wait on an mbarrier that nothing arrives on; after the limit (1 s) it must
record its code in the workspace status block and return, leaving the context usable.
The failure is made without any fault: no trap, no bad address, no endless loop.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import lsh_attention_04_b300 as lsh
from lsh_attention_04_b300 import inputs as gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lsh_attention_04_b300 import build
    build.build()
    lsh.load()


def test_bounded_wait_gives_up_and_reports():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    t0 = time.time()
    lsh.lsh_selftest_wait_timeout(ws)
    st, detail = lsh.lsh_workspace_status(ws)
    dt = time.time() - t0
    assert st == lsh.LSH_ERR_DEVICE_CHECK, lsh.lsh_status_string(st)
    assert detail == lsh.SELFTEST_WAIT_CODE
    assert 0.5 < dt < 60, dt          # it waited out its limit, then returned

    # the context stays usable: a small forward still matches the oracle
    w = gen.Workload("after_timeout_bf16_B1_H1_L1024_d64_R2", 1, 1, 1024, 64, "bf16", 32, 2, 64,
                     True, 16, 21)
    qk, v, R = gen.make_inputs(w)
    dev = lambda a: torch.from_numpy(a).cuda().to(torch.bfloat16)
    out, lse = lsh.lsh_attn_forward(dev(qk), dev(v), dev(R), w.n_buckets, w.chunk, w.causal,
                                    w.scale)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.forward(qk, v, R, w.n_buckets, w.chunk, w.causal, w.scale)
    assert float(np.abs(out.cpu().numpy() - ref_out).max()) <= 2e-2
    assert float(np.abs(lse.cpu().numpy() - ref_lse).max()) <= 2e-2
