"""Pins for the fp64 oracle: facts the KDA pages and plain mathematics fix.

Each pin takes a loaded oracle library (``oracle.load(path)``) so the same
checks also run against deliberately broken copies of the oracle
(``test_oracle_mutants.py``): every planted mistake must trip at least one pin.

Sources of the facts:
* Bounded gate, g = g_min Sigmoid(e^A z) in (g_min, 0) with g_min = -5, A_h a
  per-head scalar: "Kimi K3 technical report review" (devpress/CSDN), section
  3.2, Eq. 5.
* Recurrence, S_t = (I - b k k^T) Diag(alpha) S_{t-1} + b k v^T, o_t = S_t^T q_t,
  and its delta form: same review, section 3.1, Eq. 1; "Kimi K3: architecture,
  training and inference systems" (weigao.cc), section 3.1.
* Decay is applied before the erase ("forgetting gate placed before the
  Householder-like transform"): "Kimi K3 notes" (s1mplewind blog), section
  "Kimi Delta Attention".
* Chunkwise WY/UT form: "Kimi K3 notes", section "Chunkwise form".
* KCP segment composition S = S~ + M S_in: "Kimi K3 technical report review",
  section 8.1, Eq. 17.
"""

from __future__ import annotations

import numpy as np
import scipy.special

import oracle

TOL = 1e-11


def _rng(seed):
    return np.random.default_rng(seed)


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def random_case(seed, T=40, H=2, dk=8, dv=6, g_lo=-5.0, h0=True, N=1):
    r = _rng(seed)
    q = _unit(r.standard_normal((T, H, dk)))
    k = _unit(r.standard_normal((T, H, dk)))
    v = r.standard_normal((T, H, dv))
    g = r.uniform(g_lo, 0.0, (T, H, dk))
    beta = r.uniform(0.0, 1.0, (T, H))
    S0 = r.standard_normal((N, H, dv, dk)) * 0.5 if h0 else None
    return q, k, v, g, beta, S0


# ----------------------------------------------------------------------------- gate
def pin_gate_midpoint(lib):
    """z = 0 gives Sigmoid(0) = 1/2, so g = g_min / 2 for every A."""
    z = np.zeros((3, 4, 5))
    A = np.array([-2.0, 0.0, 0.7, 3.0])
    g = oracle.gate(z, A, -5.0, lib=lib)
    assert np.allclose(g, -2.5, atol=0, rtol=1e-15), g


def pin_gate_A0_is_scaled_logistic(lib):
    """With A = 0 the gate is g_min times the logistic function (scipy.expit)."""
    r = _rng(1)
    z = r.standard_normal((7, 3, 16)) * 4
    g = oracle.gate(z, np.zeros(3), -5.0, lib=lib)
    assert np.allclose(g, -5.0 * scipy.special.expit(z), rtol=1e-14, atol=1e-15)


def pin_gate_scale_equivariance(lib):
    """A enters only as the scale e^A on z: g(z, A) = g(e^A z, 0)."""
    r = _rng(2)
    z = r.standard_normal((5, 4, 8))
    A = np.array([-1.0, -0.3, 0.4, 1.0])
    g = oracle.gate(z, A, -5.0, lib=lib)
    g0 = oracle.gate(z * np.exp(A)[None, :, None], np.zeros(4), -5.0, lib=lib)
    assert np.allclose(g, g0, rtol=1e-14, atol=1e-15)


def pin_gate_range_and_monotone(lib):
    """g lies in [g_min, 0], decreases in z, and tends to g_min / 0 at +/- inf."""
    z = np.linspace(-40, 40, 801).reshape(-1, 1, 1)
    g = oracle.gate(z, np.array([0.3]), -5.0, lib=lib).ravel()
    assert np.all(g <= 0) and np.all(g >= -5.0)
    assert np.all(np.diff(g) <= 0)
    assert abs(g[0]) < 1e-15 and abs(g[-1] + 5.0) < 1e-15


def pin_tile_log_decay_bound(lib):
    """Sixteen gate values sum to more than -80, the tile bound of the K3 report
    (cumulative log-decay of a 16-token tile in (-80, 0))."""
    r = _rng(3)
    z = r.standard_normal((16, 2, 128)) * 10
    g = oracle.gate(z, np.array([2.0, -2.0]), -5.0, lib=lib)
    tile = g.sum(axis=0)
    assert np.all(tile >= -80.0) and np.all(tile <= 0.0)


# ------------------------------------------------------------------------ recurrence
def pin_identity_without_decay_or_write(lib):
    """alpha = 1 (g = 0) and beta = 0 leave S unchanged: hT = h0, o_t = h0^T q_t."""
    q, k, v, g, beta, S0 = random_case(10)
    g[:] = 0.0
    beta[:] = 0.0
    o, hT = oracle.recurrence(q, k, v, g, beta, S0, lib=lib)
    assert np.allclose(hT, S0, atol=TOL, rtol=0)
    want = np.einsum("hjc,thc->thj", S0[0], q)
    assert np.allclose(o, want, atol=TOL, rtol=0)


def pin_pure_decay_closed_form(lib):
    """beta = 0: S_t = Diag(exp(sum_{j<=t} g_j)) S_0 and o_t = S_t^T q_t."""
    q, k, v, g, beta, S0 = random_case(11, g_lo=-0.5)
    beta[:] = 0.0
    o, hT = oracle.recurrence(q, k, v, g, beta, S0, lib=lib)
    G = np.cumsum(g, axis=0)  # [T, H, dk]
    St = np.exp(G)[:, :, None, :] * S0[0][None]  # stored transposed [T, H, dv, dk]
    assert np.allclose(hT[0], St[-1], atol=TOL, rtol=1e-12)
    assert np.allclose(o, np.einsum("thjc,thc->thj", St, q), atol=TOL, rtol=1e-12)


def pin_delta_overwrite_any_decay(lib):
    """beta = 1 and |k| = 1: S_t^T k_t = v_t exactly, for any per-channel decay.

    With the decay applied first, k^T S_t = k^T D S - (k^T k) k^T D S + v^T = v^T.
    Queries equal to the keys therefore read back the values."""
    q, k, v, g, beta, S0 = random_case(12)
    beta[:] = 1.0
    o, _ = oracle.recurrence(k, k, v, g, beta, S0, lib=lib)
    assert np.allclose(o, v, atol=1e-12, rtol=0)


def pin_orthonormal_retrieval(lib):
    """Orthonormal keys, no decay, beta = 1, S_0 = 0: after writing (k_i, v_i),
    a query k_i (with beta = 0 so it writes nothing) returns v_i."""
    dk, dv, H = 8, 5, 1
    r = _rng(13)
    basis = np.linalg.qr(r.standard_normal((dk, dk)))[0]
    keys = basis[r.permutation(dk)]
    vals = r.standard_normal((dk, dv))
    T = 2 * dk
    k = np.zeros((T, H, dk))
    k[:dk, 0] = keys
    k[dk:, 0] = keys[::-1]
    q = k.copy()
    v = np.zeros((T, H, dv))
    v[:dk, 0] = vals
    g = np.zeros((T, H, dk))
    beta = np.zeros((T, H))
    beta[:dk] = 1.0
    o, _ = oracle.recurrence(q, k, v, g, beta, None, lib=lib)
    assert np.allclose(o[dk:, 0], vals[::-1], atol=1e-12)


def pin_scalar_affine_closed_form(lib):
    """dk = dv = 1 with constant inputs: s_t = a s_{t-1} + c with
    a = alpha (1 - beta k^2), c = beta k v, so s_t = s* + a^t (s_0 - s*)."""
    T = 30
    kk, vv, bb, gg, s0 = 0.8, -1.3, 0.6, -0.2, 0.9
    k = np.full((T, 1, 1), kk)
    v = np.full((T, 1, 1), vv)
    g = np.full((T, 1, 1), gg)
    beta = np.full((T, 1), bb)
    q = np.ones((T, 1, 1))
    o, hT = oracle.recurrence(q, k, v, g, beta, np.full((1, 1, 1, 1), s0), lib=lib)
    a = np.exp(gg) * (1 - bb * kk * kk)
    c = bb * kk * vv
    star = c / (1 - a)
    want = star + a ** np.arange(1, T + 1) * (s0 - star)
    assert np.allclose(o[:, 0, 0], want, atol=1e-13, rtol=1e-13)


def pin_scalar_gate_is_gated_deltanet(lib):
    """A decay equal on every channel turns KDA into Gated DeltaNet,
    S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T ("Kimi K3 notes",
    section "Kimi Delta Attention", the GDN line it is compared with).  For a
    constant unit key the read-out y_t = k^T S_t then obeys the scalar map
    y_t = alpha (1 - beta) y_{t-1} + beta v, iterated here on its own."""
    T = 400
    dk, dv = 4, 3
    r = _rng(14)
    kk = _unit(r.standard_normal(dk))
    vv = r.standard_normal(dv)
    a, b = np.exp(-0.05), 0.7
    k = np.tile(kk, (T, 1, 1))
    v = np.tile(vv, (T, 1, 1))
    g = np.full((T, 1, dk), np.log(a))
    beta = np.full((T, 1), b)
    q = k.copy()
    o, _ = oracle.recurrence(q, k, v, g, beta, None, lib=lib)
    y = np.zeros(dv)
    ys = []
    for _ in range(T):
        y = a * (1 - b) * y + b * vv
        ys.append(y.copy())
    assert np.allclose(o[:, 0], np.array(ys), atol=1e-12)


def pin_explicit_matrix_form(lib):
    """The oracle's operator form equals the explicit transition-matrix product."""
    q, k, v, g, beta, S0 = random_case(15, T=25, dk=6, dv=5)
    o, hT = oracle.recurrence(q, k, v, g, beta, S0, lib=lib)
    oe, hTe = oracle.explicit_product_form(q, k, v, g, beta, S0[0])
    assert np.allclose(o, oe, atol=TOL, rtol=1e-11)
    assert np.allclose(hT[0], hTe, atol=TOL, rtol=1e-11)


def pin_delta_form_agrees(lib):
    """Product form and delta form of the same step agree to rounding."""
    q, k, v, g, beta, S0 = random_case(16, T=60, dk=16, dv=12)
    o0, h0 = oracle.recurrence(q, k, v, g, beta, S0, form=0, lib=lib)
    o1, h1 = oracle.recurrence(q, k, v, g, beta, S0, form=1, lib=lib)
    assert np.allclose(o0, o1, atol=1e-12) and np.allclose(h0, h1, atol=1e-12)


def pin_chunked_equals_recurrence(lib):
    """The chunkwise WY/UT form, for chunk sizes 1, 16 and 64, equals the
    token recurrence (varlen, ragged tails, nonzero h0)."""
    lens = [70, 1, 64, 129]
    cu = np.concatenate([[0], np.cumsum(lens)])
    q, k, v, g, beta, S0 = random_case(17, T=int(cu[-1]), dk=16, dv=8, N=len(lens))
    o, hT = oracle.recurrence(q, k, v, g, beta, S0, cu_seqlens=cu, lib=lib)
    for C in (1, 16, 64):
        oc, hc = oracle.chunked(q, k, v, g, beta, S0, cu_seqlens=cu, C=C)
        assert np.allclose(o, oc, atol=1e-9, rtol=1e-9), C
        assert np.allclose(hT, hc, atol=1e-9, rtol=1e-9), C


def pin_linearity(lib):
    """(o, hT) is linear in (S_0, V) for fixed q, k, g, beta."""
    q, k, v, g, beta, S0 = random_case(18)
    r = _rng(19)
    v2 = r.standard_normal(v.shape)
    S2 = r.standard_normal(S0.shape)
    oa, ha = oracle.recurrence(q, k, v, g, beta, S0, lib=lib)
    ob, hb = oracle.recurrence(q, k, v2, g, beta, S2, lib=lib)
    oc, hc = oracle.recurrence(q, k, 2.0 * v - 3.0 * v2, g, beta, 2.0 * S0 - 3.0 * S2, lib=lib)
    assert np.allclose(oc, 2 * oa - 3 * ob, atol=1e-10)
    assert np.allclose(hc, 2 * ha - 3 * hb, atol=1e-10)


def pin_resumption(lib):
    """Running tokens [0, s) and then [s, T) from the handed-over state equals
    one run over [0, T) (the prefill -> decode state hand-off)."""
    q, k, v, g, beta, S0 = random_case(20, T=50)
    o, hT = oracle.recurrence(q, k, v, g, beta, S0, lib=lib)
    for s in (1, 17, 49):
        o1, h1 = oracle.recurrence(q[:s], k[:s], v[:s], g[:s], beta[:s], S0, lib=lib)
        o2, h2 = oracle.recurrence(q[s:], k[s:], v[s:], g[s:], beta[s:], h1, lib=lib)
        assert np.allclose(np.concatenate([o1, o2]), o, atol=1e-12)
        assert np.allclose(h2, hT, atol=1e-12)


def pin_varlen_equals_separate(lib):
    """Packed sequences with cu_seqlens equal separate runs, each from its own h0."""
    lens = [5, 0, 13, 1]
    cu = np.concatenate([[0], np.cumsum(lens)])
    q, k, v, g, beta, S0 = random_case(21, T=int(cu[-1]), N=len(lens))
    o, hT = oracle.recurrence(q, k, v, g, beta, S0, cu_seqlens=cu, lib=lib)
    for n in range(len(lens)):
        a, b = cu[n], cu[n + 1]
        on, hn = oracle.recurrence(q[a:b], k[a:b], v[a:b], g[a:b], beta[a:b], S0[n:n + 1],
                                   lib=lib)
        assert np.allclose(o[a:b], on, atol=1e-13)
        assert np.allclose(hT[n], hn[0], atol=1e-13)


def pin_non_expansive(lib):
    """For |k| = 1, beta in [0, 1], alpha in (0, 1]: |(I - b k k^T) D|_2 <= 1, so
    |S_t|_2 <= |S_{t-1}|_2 + beta_t |v_t|."""
    q, k, v, g, beta, S0 = random_case(22, T=30, H=1)
    prev = np.linalg.norm(S0[0, 0], 2)
    for t in range(30):
        _, h = oracle.recurrence(q[:t + 1], k[:t + 1], v[:t + 1], g[:t + 1], beta[:t + 1], S0,
                                 lib=lib)
        cur = np.linalg.norm(h[0, 0], 2)
        assert cur <= prev + beta[t, 0] * np.linalg.norm(v[t, 0]) + 1e-12
        prev = cur


def pin_segment_composition(lib):
    """KCP algebra: a segment maps S_in to S~ + M S_in, where S~ is the segment
    run from zero and M is the product of the transitions (I - b k k^T) Diag(alpha)."""
    q, k, v, g, beta, S0 = random_case(23, T=20, H=1, dk=6, dv=4)
    _, h_full = oracle.recurrence(q, k, v, g, beta, S0, lib=lib)
    _, h_zero = oracle.recurrence(q, k, v, g, beta, None, lib=lib)
    M = np.eye(6)
    for t in range(20):
        kt = k[t, 0]
        M = (np.eye(6) - beta[t, 0] * np.outer(kt, kt)) @ np.diag(np.exp(g[t, 0])) @ M
    S_end = h_zero[0, 0].T + M @ S0[0, 0].T
    assert np.allclose(h_full[0, 0].T, S_end, atol=1e-12)


def pin_decode_step_is_one_token(lib):
    """The decode form (N one-token sequences) equals one recurrence step each."""
    r = _rng(24)
    N, H, dk, dv = 3, 2, 8, 4
    q = _unit(r.standard_normal((N, H, dk)))
    k = _unit(r.standard_normal((N, H, dk)))
    v = r.standard_normal((N, H, dv))
    g = r.uniform(-5, 0, (N, H, dk))
    beta = r.uniform(0, 1, (N, H))
    S = r.standard_normal((N, H, dv, dk))
    o, S1 = oracle.decode_step(q, k, v, g, beta, S, lib=lib)
    for n in range(N):
        on, hn = oracle.recurrence(q[n:n + 1], k[n:n + 1], v[n:n + 1], g[n:n + 1],
                                   beta[n:n + 1], S[n:n + 1], lib=lib)
        assert np.allclose(o[n], on[0], atol=1e-13) and np.allclose(S1[n], hn[0], atol=1e-13)


def pin_chunk_cumsum(lib):
    """The in-chunk running sum: C = 1 returns g, one chunk covering a sequence
    is a plain cumulative sum, and the chunks of a sequence add up to its total."""
    r = _rng(25)
    g = r.uniform(-5, 0, (70, 2, 3))
    cu = [0, 70]
    assert np.array_equal(oracle.chunk_cumsum(g, cu, C=1), g)
    assert np.allclose(oracle.chunk_cumsum(g, cu, C=128), np.cumsum(g, axis=0), atol=1e-13)
    c64 = oracle.chunk_cumsum(g, cu, C=64)
    assert np.allclose(c64[63] + c64[69], g.sum(axis=0), atol=1e-12)
    assert np.allclose(c64[64], g[64], atol=0)  # a new chunk starts at token 64
    cu2 = [0, 10, 70]
    c2 = oracle.chunk_cumsum(g, cu2, C=64)
    assert np.allclose(c2[10], g[10], atol=0)  # a new sequence starts a new chunk


ALL_PINS = [
    pin_gate_midpoint,
    pin_gate_A0_is_scaled_logistic,
    pin_gate_scale_equivariance,
    pin_gate_range_and_monotone,
    pin_tile_log_decay_bound,
    pin_identity_without_decay_or_write,
    pin_pure_decay_closed_form,
    pin_delta_overwrite_any_decay,
    pin_orthonormal_retrieval,
    pin_scalar_affine_closed_form,
    pin_scalar_gate_is_gated_deltanet,
    pin_explicit_matrix_form,
    pin_delta_form_agrees,
    pin_chunked_equals_recurrence,
    pin_linearity,
    pin_resumption,
    pin_varlen_equals_separate,
    pin_non_expansive,
    pin_segment_composition,
    pin_decode_step_is_one_token,
    pin_chunk_cumsum,
]
