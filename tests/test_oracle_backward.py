"""The oracle's staged backward (given buckets, as the GPU comparisons use it) agrees with
its whole backward pass when given the oracle's own buckets (CPU only)."""
import numpy as np
import pytest

import oracle


@pytest.mark.parametrize("causal", [False, True])
def test_staged_backward_matches_whole_backward(causal):
    orc = oracle.default()
    rng = np.random.default_rng(40 + causal)
    n_heads, L, d, nb, c, n_rounds, scale = 2, 96, 16, 6, 16, 3, 0.5
    qk = rng.standard_normal((n_heads, L, d))
    v = rng.standard_normal((n_heads, L, d))
    R = rng.standard_normal((n_rounds, d, nb // 2))
    g_out = rng.standard_normal((n_heads, L, d))
    g_lse = rng.standard_normal((n_heads, L))
    out, lse, it = orc.forward(qk, v, R, nb, c, causal, scale, intermediates=True)
    dqk, dv = orc.backward(qk, v, R, nb, c, causal, scale, g_out, g_lse)
    for h in range(n_heads):
        o2, l2, dq2, dv2 = orc.backward_given_buckets(qk[h], v[h], it["bucket"][h], nb, c,
                                                      causal, scale, g_out[h], g_lse[h])
        assert np.allclose(o2, out[h], rtol=0, atol=1e-12)
        assert np.allclose(l2, lse[h], rtol=0, atol=1e-12)
        assert np.allclose(dq2, dqk[h], rtol=0, atol=1e-12)
        assert np.allclose(dv2, dv[h], rtol=0, atol=1e-12)
    # g_lse = None means zero
    _, _, dq0, dv0 = orc.backward_given_buckets(qk[0], v[0], it["bucket"][0], nb, c, causal,
                                                scale, g_out[0], None)
    dqz, dvz = orc.backward(qk[:1], v[:1], R, nb, c, causal, scale, g_out[:1],
                            np.zeros((1, L)))
    assert np.allclose(dq0, dqz[0], rtol=0, atol=1e-12)
    assert np.allclose(dv0, dvz[0], rtol=0, atol=1e-12)
