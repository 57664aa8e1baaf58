"""Pins for the oracle's fused prologue / epilogue pieces and the unbounded gate
(CPU only).

* ``oracle.l2_normalize`` -- the L2Norm on the q and k branches ("Kimi K3:
  architecture, training and inference systems", section 3.2), with the
  caller's epsilon inside the square root.
* ``oracle.output_gate`` -- head-wise RMSNorm of the KDA output times the
  Sigmoid gate ("Kimi K3 technical report review", section 3.3, Eq. 6).
* ``oracle.gate_softplus`` -- the unbounded gate -exp(A) Softplus(z) the bounded
  one replaced (same review, section 3.2), and the recurrence under it.

Every expected value below is worked out by hand from those definitions.  Each
pin takes the implementation as an argument so that the planted mistakes at the
end (a sum for the mean, a dropped square root, the gate's sign flipped, the
wrong axis, ...) can be shown to trip at least one pin.
"""

import math

import numpy as np
import pytest

import oracle

TOL = 1e-12


# ------------------------------------------------------------------ L2 norm pins
def l2_pin_345(f):
    """|(3, 4)| = 5: (0.6, 0.8) with eps = 0."""
    np.testing.assert_allclose(f(np.array([3.0, 4.0]), 0.0), [0.6, 0.8], atol=TOL)


def l2_pin_eps_inside_root(f):
    """eps = 11: 1 / sqrt(25 + 11) = 1/6, so (0.5, 2/3)."""
    np.testing.assert_allclose(f(np.array([3.0, 4.0]), 11.0), [0.5, 2.0 / 3.0], atol=TOL)


def l2_pin_last_axis_only(f):
    """[T=1, H=2, d=2]: each head's channels are normalised on their own."""
    x = np.array([[[3.0, 4.0], [0.0, -2.0]]])
    np.testing.assert_allclose(f(x, 0.0), [[[0.6, 0.8], [0.0, -1.0]]], atol=TOL)


L2_PINS = [l2_pin_345, l2_pin_eps_inside_root, l2_pin_last_axis_only]


# -------------------------------------------------------------- output gate pins
def og_pin_constant_row(f):
    """o = c * ones: rms = |c|, so with x = 0 every entry is Sigmoid(0) sign(c) = +-1/2."""
    o = np.array([[-3.0] * 4, [0.25] * 4])
    np.testing.assert_allclose(f(o, np.zeros_like(o), None, 0.0),
                               [[-0.5] * 4, [0.5] * 4], atol=TOL)


def og_pin_gate_values(f):
    """o = 2 (1, -1, 1, -1): rms = 2; x = (0, ln 3, -ln 3, 40) gives gates
    (1/2, 3/4, 1/4, ~1), so y = (1/2, -3/4, 1/4, -1)."""
    o = np.array([2.0, -2.0, 2.0, -2.0])
    x = np.array([0.0, math.log(3.0), -math.log(3.0), 40.0])
    np.testing.assert_allclose(f(o, x, None, 0.0), [0.5, -0.75, 0.25, -1.0], atol=1e-12)


def og_pin_eps_and_weight(f):
    """o = (3, 4): mean(o^2) = 12.5; eps = 3.5 gives rms 4, o / rms = (3/4, 1);
    w = (2, -1) and x = 0 give (3/4, -1/2)."""
    np.testing.assert_allclose(f(np.array([3.0, 4.0]), np.zeros(2), np.array([2.0, -1.0]), 3.5),
                               [0.75, -0.5], atol=TOL)


def og_pin_headwise(f):
    """[T=1, H=2, d=2]: heads scaled by 10 and 0.1 give the same normalised rows."""
    o = np.array([[[30.0, 40.0], [0.3, 0.4]]])
    r = 1.0 / math.sqrt(12.5)
    np.testing.assert_allclose(f(o, np.zeros_like(o), None, 0.0),
                               [[[1.5 * r, 2.0 * r], [1.5 * r, 2.0 * r]]], atol=1e-12)


OG_PINS = [og_pin_constant_row, og_pin_gate_values, og_pin_eps_and_weight, og_pin_headwise]


@pytest.mark.parametrize("pin", L2_PINS, ids=lambda p: p.__name__)
def test_l2_normalize_pin(pin):
    pin(oracle.l2_normalize)


@pytest.mark.parametrize("pin", OG_PINS, ids=lambda p: p.__name__)
def test_output_gate_pin(pin):
    pin(lambda o, x, w, eps: oracle.output_gate(o, x, w, eps))


# ---------------------------------------------------------------- planted mistakes
def _l2_eps_outside(x, eps):
    return x / (np.sqrt(np.sum(x * x, axis=-1, keepdims=True)) + eps)


def _l2_no_root(x, eps):
    return x / (np.sum(x * x, axis=-1, keepdims=True) + eps)


def _l2_first_axis(x, eps):
    # (an all-zero column over the wrong axis gives 0 / 0 here: expected of the mutant)
    with np.errstate(invalid="ignore", divide="ignore"):
        return x / np.sqrt(np.sum(x * x, axis=0, keepdims=True) + eps)


def _og_sum_for_mean(o, x, w, eps):
    y = o / np.sqrt(np.sum(o * o, axis=-1, keepdims=True) + eps) / (1 + np.exp(-x))
    return y if w is None else y * w


def _og_gate_sign(o, x, w, eps):
    y = o / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps) / (1 + np.exp(x))
    return y if w is None else y * w


def _og_no_weight(o, x, w, eps):
    return o / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps) / (1 + np.exp(-x))


def _og_eps_outside(o, x, w, eps):
    y = o / (np.sqrt(np.mean(o * o, axis=-1, keepdims=True)) + eps) / (1 + np.exp(-x))
    return y if w is None else y * w


def _og_whole_token(o, x, w, eps):  # normalised over all heads of a token
    ax = (-2, -1) if o.ndim >= 2 else -1
    y = o / np.sqrt(np.mean(o * o, axis=ax, keepdims=True) + eps) / (1 + np.exp(-x))
    return y if w is None else y * w


@pytest.mark.parametrize("mutant", [_l2_eps_outside, _l2_no_root, _l2_first_axis],
                         ids=lambda m: m.__name__)
def test_l2_mutant_trips_a_pin(mutant):
    tripped = 0
    for pin in L2_PINS:
        try:
            pin(mutant)
        except AssertionError:
            tripped += 1
    assert tripped > 0


@pytest.mark.parametrize("mutant", [_og_sum_for_mean, _og_gate_sign, _og_no_weight,
                                    _og_eps_outside, _og_whole_token],
                         ids=lambda m: m.__name__)
def test_output_gate_mutant_trips_a_pin(mutant):
    tripped = 0
    for pin in OG_PINS:
        try:
            pin(mutant)
        except AssertionError:
            tripped += 1
    assert tripped > 0


# ------------------------------------------------------------ unbounded gate pins
def sp_pin_zero(f):
    """Softplus(0) = ln 2: g = -ln 2 for A = 0 and -2 ln 2 for A = ln 2."""
    z = np.zeros((1, 2, 1))
    np.testing.assert_allclose(f(z, np.array([0.0, math.log(2.0)])),
                               [[[-math.log(2.0)], [-2 * math.log(2.0)]]], rtol=1e-14)


def sp_pin_tails(f):
    """Softplus(x) = x + log(1 + e^-x) -> x for large x (no overflow at 1000) and
    log(1 + e^x) = e^x (1 - e^x / 2 + ...) for very negative x."""
    z = np.array([[[1000.0, 30.0, -30.0]]])
    want = [[[-1000.0, -(30.0 + math.log1p(math.exp(-30.0))), -math.log1p(math.exp(-30.0))]]]
    np.testing.assert_allclose(f(z, np.array([0.0])), want, rtol=1e-14)


def sp_pin_unbounded_monotone(f):
    """g is below any bound for large z and decreasing in z."""
    z = np.linspace(-5, 200, 50).reshape(50, 1, 1)
    g = f(z, np.array([0.5]))[:, 0, 0]
    assert g[-1] < -300 and np.all(np.diff(g) < 0)


SP_PINS = [sp_pin_zero, sp_pin_tails, sp_pin_unbounded_monotone]


@pytest.mark.parametrize("pin", SP_PINS, ids=lambda p: p.__name__)
def test_gate_softplus_pin(pin):
    pin(oracle.gate_softplus)


@pytest.mark.parametrize("mutant", [
    lambda z, A: -np.exp(A)[None, :, None] * np.log1p(np.maximum(z, -0.999)),  # log(1 + z)
    lambda z, A: -A[None, :, None] * np.logaddexp(0.0, z),                   # A without exp
    lambda z, A: -np.exp(A)[None, :, None] * np.logaddexp(0.0, -z),          # sign of z
], ids=["log1p_of_z", "A_without_exp", "z_sign"])
def test_gate_softplus_mutant_trips_a_pin(mutant):
    tripped = 0
    for pin in SP_PINS:
        try:
            pin(mutant)
        except (AssertionError, FloatingPointError):
            tripped += 1
    assert tripped > 0


def test_recurrence_full_forgetting_closed_form(oracle_lib):
    """g = -10^4 (alpha = e^-10000 = 0 in fp64): the state carries nothing between
    tokens, so S_t = b_t k_t v_t^T and o_t = b_t (q_t . k_t) v_t."""
    rng = np.random.default_rng(5)
    T, H, dk, dv = 7, 2, 8, 5
    q, k = rng.standard_normal((T, H, dk)), rng.standard_normal((T, H, dk))
    v, b = rng.standard_normal((T, H, dv)), rng.uniform(0, 1, (T, H))
    g = np.full((T, H, dk), -1e4)
    h0 = rng.standard_normal((1, H, dv, dk))
    o, hT = oracle.recurrence(q, k, v, g, b, h0, lib=oracle_lib)
    want = b[..., None] * np.sum(q * k, axis=-1)[..., None] * v
    np.testing.assert_allclose(o, want, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(hT[0], b[-1][:, None, None] * v[-1][:, :, None] * k[-1][:, None, :],
                               rtol=1e-12, atol=1e-14)
