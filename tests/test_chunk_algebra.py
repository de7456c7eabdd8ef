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


def eda_subtokens(q, k, v, e, beta):
    """The sub-token sequence of the tensor-core EDA path ([T, d] arrays of one stream,
    beta None = 1): keys, values, strengths and queries of 2T+1 Delta-rule sub-tokens
    (a leading no-op carrying r_0, then per token the erase e_t (value 0, strength 1,
    query 0) and the write k_t (v_t, beta_t, query r_{t+1})), and c_t = beta_t k_t.q_t."""
    T, dk = q.shape
    b = np.ones(T) if beta is None else beta
    c = b * np.einsum("td,td->t", k, q)
    y = q - c[:, None] * k
    r = y - np.einsum("td,td->t", e, y)[:, None] * e
    n = 2 * T + 1
    K = np.zeros((n, dk)); V = np.zeros((n, v.shape[1])); Bs = np.zeros(n); Q = np.zeros((n, dk))
    K[1::2], Bs[1::2] = e, 1.0
    K[2::2], V[2::2], Bs[2::2] = k, v, b
    Q[0:2 * T:2] = r
    return K, V, Bs, Q, c


@pytest.mark.parametrize("T", [1, 2, 33, 100])
@pytest.mark.parametrize("erase", ["random", "query", "scaled"])
@pytest.mark.parametrize("unit_step", [False, True])
def test_eda_is_a_delta_rule_over_subtokens(T, erase, unit_step):
    """EDA ("Erase-then-Delta Attention": erase along e, then the Delta write) equals the
    Delta rule over 2T+1 sub-tokens read one sub-token before each erase with
    r_t = (I - e e^T)(q - c k), plus c_t v_t: the oracle's EDA against the oracle's
    Q-Delta forward (alpha 1, lambda 0) over that sequence, both fp64."""
    dk, dv = 8, 6
    q = _unit(rng.standard_normal((1, T, 1, dk)))
    k = _unit(rng.standard_normal((1, T, 1, dk)))
    e = q.copy() if erase == "query" else _unit(rng.standard_normal((1, T, 1, dk)))
    if erase == "scaled":               # |e| != 1: the identity needs only (I - e e^T) symmetric
        e = e * rng.uniform(0.5, 1.5, (1, T, 1, 1))
    v = rng.standard_normal((1, T, 1, dv))
    beta = None if unit_step else rng.uniform(0.05, 1.0, (1, T, 1))
    S0 = rng.standard_normal((1, 1, dv, dk)) * 0.5
    o_ref, S_ref = oracle.eda_fwd(q, k, v, e, beta, S0)
    K, V, Bs, Q, c = eda_subtokens(q[0, :, 0], k[0, :, 0], v[0, :, 0], e[0, :, 0],
                                   None if beta is None else beta[0, :, 0])
    o_sub, S = oracle.qdelta_fwd(Q[None, :, None], K[None, :, None], V[None, :, None], None, Bs[None, :, None],
                                 None, S0)
    o = o_sub[0, 0:2 * T:2, 0] + c[:, None] * v[0, :, 0]
    assert np.abs(o - o_ref[0, :, 0]).max() <= 1e-12 * max(1.0, np.abs(o_ref).max())
    assert np.abs(S - S_ref).max() <= 1e-12 * max(1.0, np.abs(S_ref).max())


def pair_map_box(compact, j0, C=64):
    """A pair-map box as the tensor-core EDA path reads it: 64 sub-token rows whose row
    2i + p is compact row j0 + i for p = 0 and zero for p = 1 (the size-1 dimension), zero
    too where j0 + i falls outside [0, len(compact))."""
    out = np.zeros((C, compact.shape[1]))
    for i in range(C // 2):
        j = j0 + i
        if 0 <= j < len(compact):
            out[2 * i] = compact[j]
    return out


@pytest.mark.parametrize("T", [1, 31, 32, 33, 100])
def test_eda_pair_maps_give_the_subtoken_rows(T):
    """The compact queries r_t and values v_t, read chunk by chunk through pair-map boxes
    at row j0 = 32 c (queries) and 32 c - 1 (values), give exactly the sub-token query
    and value rows; the even rows of the sub-token outputs are what a pair-map store at
    row 32 c keeps (and a chunk starting at row T, holding only sub-token 2T, keeps none)."""
    dk, dv = 8, 6
    q = _unit(rng.standard_normal((T, dk)))
    k = _unit(rng.standard_normal((T, dk)))
    e = _unit(rng.standard_normal((T, dk)))
    v = rng.standard_normal((T, dv))
    beta = rng.uniform(0.05, 1.0, T)
    K, V, Bs, Q, c = eda_subtokens(q, k, v, e, beta)
    r = Q[0:2 * T:2]                                   # the compact queries
    n = 2 * T + 1
    nch = (n + 63) // 64
    Qm = np.concatenate([pair_map_box(r, 32 * ch) for ch in range(nch)])[:n]
    Vm = np.concatenate([pair_map_box(v, 32 * ch - 1) for ch in range(nch)])[:n]
    np.testing.assert_array_equal(Qm, Q)
    np.testing.assert_array_equal(Vm, V)
    O = rng.standard_normal((nch * 64, dv))            # any sub-token outputs
    kept = np.zeros((T, dv))
    for ch in range(nch):
        if 32 * ch >= T:                               # the kernel skips this store
            continue
        for i in range(32):
            if 32 * ch + i < T:
                kept[32 * ch + i] = O[64 * ch + 2 * i]
    np.testing.assert_array_equal(kept, O[0:2 * T:2])
