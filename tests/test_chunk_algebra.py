"""The chunked algebra the kernels implement equals the sequential oracle (fp64).

Pins the forms derived from the Q-Delta notes' sec. 3.3.2 (WY / UT transform,
with the notes' corrections) and the QED notes' Eq. 6 / GDN-2 update, including
ragged final chunks and a carried initial state.
"""
import numpy as np
import pytest

import oracle
from chunk_model import qdelta_chunked, qdelta_chunked_bwd, qed_chunked

rng = np.random.default_rng(7)


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


@pytest.mark.parametrize("T,C", [(1, 16), (16, 16), (37, 16), (64, 16), (100, 32), (130, 64)])
@pytest.mark.parametrize("mode", ["qdelta", "gdn", "deltanet"])
def test_qdelta_chunked_equals_sequential(T, C, mode):
    dk, dv = 8, 6
    q = _unit(rng.standard_normal((1, T, 1, dk)))
    k = _unit(rng.standard_normal((1, T, 1, dk)))
    v = rng.standard_normal((1, T, 1, dv))
    beta = rng.uniform(0.05, 1.0, (1, T, 1))
    alpha = rng.uniform(0.7, 1.0, (1, T, 1)) if mode != "deltanet" else None
    lam = rng.uniform(0, 1, (1, T, 1)) if mode == "qdelta" else None
    S0 = rng.standard_normal((1, 1, dv, dk)) * 0.5
    o_ref, S_ref = oracle.qdelta_fwd(q, k, v, alpha, beta, lam, S0)
    o, S = qdelta_chunked(q[0, :, 0], k[0, :, 0], v[0, :, 0],
                          None if alpha is None else alpha[0, :, 0], beta[0, :, 0],
                          None if lam is None else lam[0, :, 0], S0[0, 0], C)
    scale = max(1.0, np.abs(o_ref).max())
    assert np.abs(o - o_ref[0, :, 0]).max() <= 1e-12 * scale
    assert np.abs(S - S_ref[0, 0]).max() <= 1e-12 * max(1.0, np.abs(S_ref).max())


@pytest.mark.parametrize("T,C", [(1, 16), (37, 16), (100, 32), (130, 64)])
def test_qed_chunked_equals_sequential(T, C):
    K, V = 8, 6
    q = _unit(rng.standard_normal((1, T, 1, K)))
    k = _unit(rng.standard_normal((1, T, 1, K)))
    v = rng.standard_normal((1, T, 1, V))
    g = -rng.uniform(0.0, 0.1, (1, T, 1, K))
    b = rng.uniform(0.05, 0.95, (1, T, 1, K))
    w = rng.uniform(0.05, 0.95, (1, T, 1, V))
    lam_h = np.array([0.6])
    S0 = rng.standard_normal((1, 1, V, K)) * 0.5
    o_ref, S_ref = oracle.qed_fwd(q, k, v, g, b, w, lam_h, S0)
    o, S = qed_chunked(q[0, :, 0], k[0, :, 0], v[0, :, 0], g[0, :, 0], b[0, :, 0], w[0, :, 0],
                       0.6, S0[0, 0], C)
    assert np.abs(o - o_ref[0, :, 0]).max() <= 1e-12 * max(1.0, np.abs(o_ref).max())
    assert np.abs(S - S_ref[0, 0]).max() <= 1e-12 * max(1.0, np.abs(S_ref).max())


@pytest.mark.parametrize("T,C", [(1, 16), (16, 16), (37, 16), (100, 32), (130, 64)])
@pytest.mark.parametrize("mode", ["qdelta", "gdn", "deltanet"])
def test_qdelta_chunked_backward_equals_sequential_adjoint(T, C, mode):
    """The chunked backward (per-chunk adjoint of the WY form, reverse chunk order)
    equals the oracle's step-by-step adjoint in fp64."""
    dk, dv = 8, 6
    q = _unit(rng.standard_normal((1, T, 1, dk)))
    k = _unit(rng.standard_normal((1, T, 1, dk)))
    v = rng.standard_normal((1, T, 1, dv))
    beta = rng.uniform(0.05, 1.0, (1, T, 1))
    alpha = rng.uniform(0.7, 1.0, (1, T, 1)) if mode != "deltanet" else None
    lam = rng.uniform(0, 1, (1, T, 1)) if mode == "qdelta" else None
    S0 = rng.standard_normal((1, 1, dv, dk)) * 0.5
    dO = rng.standard_normal((1, T, 1, dv))
    dS = rng.standard_normal((1, 1, dv, dk))
    ref = oracle.qdelta_bwd(q, k, v, alpha, beta, lam, S0, dO, dS)
    sq = lambda a: None if a is None else a[0, :, 0]
    g = qdelta_chunked_bwd(sq(q), sq(k), sq(v), sq(alpha), sq(beta), sq(lam), S0[0, 0], sq(dO), dS[0, 0], C)
    for name, r in ref.items():
        if r is None:
            assert g[name] is None
            continue
        r = r[0, 0] if name == "dS0" else r[0, :, 0]
        np.testing.assert_allclose(g[name], r, atol=1e-11 * max(1.0, np.abs(r).max()), err_msg=name)
