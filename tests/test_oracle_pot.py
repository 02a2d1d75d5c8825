"""Pins of the oracle's Rowmax-PoT weights ("Approximating Softmax in Pretrained LLMs:
Model Sensitivity and Kernel Acceleration", AI Summary and Abstract: powers of two
anchored at each row maximum).

Hand-worked examples use D = 1 and scale = 1, so a logit is q * k; logits are
chosen as multiples of ln 2 so that exponents in log2 units are read off directly.
Special cases reduce to a library routine (torch SDPA); a bound holds for any input.
"""

import math

import numpy as np
import pytest

import oracle
from oracle import skipsm_oracle as so
from pins import causal_allowed, sdpa

LN2 = math.log(2.0)


def _one(logits, values, *, tile_k, lam=0.0, causal=False):
    """One row (q = 1) against keys k = logits: (o, lse, mask, ambiguous fraction)."""
    n = len(logits)
    q = np.ones((1, 1, 1, 1))
    k = np.asarray(logits, dtype=np.float64).reshape(1, 1, n, 1)
    v = np.asarray(values, dtype=np.float64).reshape(1, 1, n, 1)
    r = oracle.prefill(q, k, v, causal=causal, lam=lam, tile_q=1, tile_k=tile_k, scale=1.0,
                       pot=True)
    return r.o[0, 0, 0, 0], r.lse[0, 0, 0], r.mask[0, 0, 0], r.pot_ambiguous[0, 0, 0]


def test_worked_single_tile_rounding():
    # exponents (log2 units) relative to the max: 0, -1.4, -2.6  ->  weights 1, 1/2, 1/8
    o, lse, _, amb = _one([0.0, -1.4 * LN2, -2.6 * LN2], [1.0, 2.0, 3.0], tile_k=4)
    want = (1.0 * 1 + 0.5 * 2 + 0.125 * 3) / 1.625
    assert abs(o - want) < 1e-14
    assert abs(lse - math.log(1.625)) < 1e-14
    assert amb == 0.0


def test_worked_online_anchor_moves_with_the_running_max():
    # tile 0: exponents 0, -1.4 (max 0)         -> 1, 1/2 relative to 0
    # tile 1: exponents 2.3, 0.9 (new max 2.3)  -> 1, 2^round(-1.4) = 1/2 relative to 2.3
    # tile 0 is rescaled exactly by 2^(0 - 2.3); a global anchor would instead give
    # 2^round(-2.3) = 1/4 and 2^round(-3.7) = 1/16 to the first two keys.
    vals = [1.0, 2.0, 3.0, 4.0]
    o, lse, mask, _ = _one([0.0, -1.4 * LN2, 2.3 * LN2, 0.9 * LN2], vals, tile_k=2)
    assert mask.tolist() == [0, 0]
    a = 2.0 ** -2.3
    w = [a, a * 0.5, 1.0, 0.5]
    want = sum(wi * vi for wi, vi in zip(w, vals)) / sum(w)
    assert abs(o - want) < 1e-13
    assert abs(lse - (2.3 * LN2 + math.log(sum(w)))) < 1e-13


def test_worked_underflow_and_masked_keys_weigh_zero():
    # exponent -130 is below 2^-126.5 -> weight 0; -126.4 rounds to -126 -> 2^-126
    o, _, _, _ = _one([0.0, -130.0 * LN2], [5.0, -7.0], tile_k=2)
    assert o == 5.0
    o, _, _, _ = _one([0.0, -126.4 * LN2], [0.0, 1.0], tile_k=2)
    assert abs(o - 2.0 ** -126 / (1.0 + 2.0 ** -126)) < 1e-300
    # causal, Sq = Skv = 2: the first row sees only key 0
    q = np.ones((1, 1, 2, 1))
    k = np.array([0.0, 3.0]).reshape(1, 1, 2, 1)
    v = np.array([1.0, 9.0]).reshape(1, 1, 2, 1)
    r = oracle.prefill(q, k, v, causal=True, lam=0.0, tile_q=2, tile_k=2, scale=1.0, pot=True)
    assert r.o[0, 0, 0, 0] == 1.0


def test_worked_skip_rule_unchanged_and_ambiguity_flagged():
    # the vote uses exact maxima: tile 1 (max exponent -3 below the running max 0) is
    # skipped for lambda = 2^-2 and kept for lambda = 2^-4, exactly as without PoT
    logits = [0.0, -0.2 * LN2, -3.0 * LN2, -5.0 * LN2]
    _, _, mask, _ = _one(logits, [1, 2, 3, 4], tile_k=2, lam=0.25)
    assert mask.tolist() == [0, 1]
    _, _, mask, _ = _one(logits, [1, 2, 3, 4], tile_k=2, lam=2.0 ** -4)
    assert mask.tolist() == [0, 0]
    # an exponent within the band of a rounding boundary is reported as ambiguous
    _, _, _, amb = _one([0.0, -(1.5 - 0.3 * so.POT_AMBIGUOUS_BAND) * LN2], [1, 2], tile_k=2)
    assert 0.0 < amb < 1.0
    _, _, _, amb = _one([0.0, -1.3 * LN2], [1, 2], tile_k=2)
    assert amb == 0.0


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("tile_k", [2, 3, 16])
def test_integer_exponents_reduce_to_exact_softmax(causal, tile_k):
    # logits a * b_c * ln 2 with integer a, b_c: every exponent is an integer, so the
    # powers of two are the exact exponentials and the result is dense softmax (SDPA)
    rng = np.random.default_rng(3)
    Sq, Skv, D = 5, 11, 1
    qi = rng.integers(-2, 3, size=(Sq, 1)).astype(np.float64)
    ki = rng.integers(-6, 7, size=(Skv, 1)).astype(np.float64)
    v = rng.standard_normal((Skv, D))
    q, k = qi * LN2, ki
    r = oracle.prefill(q[None, None], k[None, None], v[None, None], causal=causal, lam=0.0,
                       tile_q=2, tile_k=tile_k, scale=1.0, pot=True)
    want = sdpa(q, k, v, causal_allowed(Sq, Skv, causal), 1.0)
    assert np.max(np.abs(r.o[0, 0] - want)) < 1e-12


@pytest.mark.parametrize("seed", range(4))
def test_bound_against_dense_softmax(seed):
    # each PoT weight is within a factor 2^(1/2) of exp(s - m'), so the normalised
    # weights are within total variation (2-1)/(2+1) = 1/3 of the softmax, and each
    # output component is within range(v)/3 of dense attention
    rng = np.random.default_rng(seed)
    Sq, Skv, D = 6, 13, 8
    q, k, v = (rng.standard_normal((n, D)) * 2 for n in (Sq, Skv, Skv))
    r = oracle.prefill(q[None, None], k[None, None], v[None, None], causal=True, lam=0.0,
                       tile_q=3, tile_k=4, scale=None, pot=True)
    want = sdpa(q, k, v, causal_allowed(Sq, Skv, True), 1.0 / math.sqrt(D))
    rng_v = v.max(axis=0) - v.min(axis=0)
    assert np.all(np.abs(r.o[0, 0] - want) <= rng_v[None, :] / 3 + 1e-12)
    # and the outputs are convex combinations of the values
    assert np.all(r.o[0, 0] <= v.max(axis=0) + 1e-12)
    assert np.all(r.o[0, 0] >= v.min(axis=0) - 1e-12)


def test_pot_off_is_unchanged():
    rng = np.random.default_rng(7)
    q, k, v = (rng.standard_normal((1, 2, 9, 4)) for _ in range(3))
    a = oracle.prefill(q, k[:, :1], v[:, :1], causal=True, lam=0.3, tile_q=3, tile_k=2)
    b = oracle.prefill(q, k[:, :1], v[:, :1], causal=True, lam=0.3, tile_q=3, tile_k=2,
                       pot=False)
    assert np.array_equal(a.o, b.o) and a.pot_ambiguous is None


# ---------------------------------------------------------------------------
# plausible mistakes planted in the oracle's PoT steps must fail a pin above
# ---------------------------------------------------------------------------
def _w_floor(s, m_new):
    w, amb = _W_ORIG(s, m_new)
    with np.errstate(invalid="ignore"):
        x = np.maximum((s - m_new[:, None]) * so.LOG2E, -127.0)
    n = np.floor(x)
    return np.where(n < -126.0, 0.0, np.exp2(n)), amb


def _w_unrounded(s, m_new):
    w, amb = _W_ORIG(s, m_new)
    with np.errstate(invalid="ignore"):
        x = (s - m_new[:, None]) * so.LOG2E
    return np.where(np.isfinite(x), np.exp2(x), 0.0), amb


def _w_natural_base(s, m_new):
    w, amb = _W_ORIG(s, m_new)
    with np.errstate(invalid="ignore"):
        x = np.maximum(s - m_new[:, None], -127.0)
    n = np.rint(x)
    return np.where(n < -126.0, 0.0, np.exp2(n)), amb


def _upd_no_rescale(m, l, o, a, s, vt):
    m_new = np.maximum(m, np.max(s, axis=1))
    w, amb = so._pot_weights(s, m_new)
    return m_new, l + w.sum(axis=1), o + w @ vt, a + (w * amb).sum(axis=1)


def _upd_global_anchor_first_tile(m, l, o, a, s, vt):
    # anchors every tile at the first tile's maximum (never moves the anchor)
    m_anchor = np.where(m == -np.inf, np.max(s, axis=1), m)
    w, amb = so._pot_weights(s, m_anchor)
    return m_anchor, l + w.sum(axis=1), o + w @ vt, a + (w * amb).sum(axis=1)


_W_ORIG = so._pot_weights
_PINS = [test_worked_single_tile_rounding, test_worked_online_anchor_moves_with_the_running_max,
         test_worked_underflow_and_masked_keys_weigh_zero]


@pytest.mark.parametrize("name,target,fn", [
    ("floor_not_round", "_pot_weights", _w_floor),
    ("no_quantisation", "_pot_weights", _w_unrounded),
    ("natural_log_units", "_pot_weights", _w_natural_base),
    ("earlier_tiles_not_rescaled", "_online_update_pot", _upd_no_rescale),
    ("anchor_never_moves", "_online_update_pot", _upd_global_anchor_first_tile),
])
def test_pot_mutants_are_caught(monkeypatch, name, target, fn):
    monkeypatch.setattr(so, target, fn)
    caught = 0
    for pin in _PINS:
        try:
            pin()
        except AssertionError:
            caught += 1
    assert caught > 0, f"mutant {name} passed every PoT pin"
