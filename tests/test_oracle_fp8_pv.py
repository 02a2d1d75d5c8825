"""The oracle's FP8 P.V reading against what the definition and mathematics fix (CPU).

Reading ("Approximating Softmax in Pretrained LLMs ...", AI Summary: FP8/BF16 mixed
precision): on a kept tile each weight p = exp(s - m') (m' the running row maximum after
the tile) enters P.V as e4m3(2^8 p) 2^-8, rounded to nearest with ties to even; the row
sum keeps the exact p; the skip vote is unchanged.

Pins: e4m3 rounding against worked values and torch's float8_e4m3fn cast; a worked
example with a growing maximum; reduction to the exact oracle when every scaled weight
is an e4m3 value; the bound |o_fp8 - o| <= (2^-4 + n 2^-18 / l) max|v| per row against
the exact oracle with the same skip mask; the ambiguity report at a rounding midpoint;
and planted mistakes (no 2^8 scale, the row sum from quantised weights, truncation,
the pre-tile maximum as anchor), each caught by one of these pins.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import skipsm_oracle as so

E, L2, L3 = math.exp, math.log(2.0), math.log(3.0)


def test_e4m3_round_worked_values():
    cases = [
        (85.3333, 88.0),            # [64, 128): step 8, 10.67 steps -> 11
        (17.0, 16.0),               # [16, 32): step 2, 8.5 steps -> tie -> 8 (even)
        (19.0, 20.0),               # 9.5 steps -> tie -> 10 (even)
        (1.0625, 1.0),              # [1, 2): step 1/8, 8.5 -> 8
        (1.3, 1.25),                # 10.4 steps -> 10
        (2.0 ** -10, 0.0),          # half the subnormal step 2^-9: tie -> 0
        (3 * 2.0 ** -10, 2 * 2.0 ** -9),   # 1.5 subnormal steps -> 2
        (2.0 ** -6 * 1.05, 2.0 ** -6),     # smallest normal binade, step 2^-9: 8.4 -> 8
        (2.0 ** -6 * 1.07, 9 * 2.0 ** -9),  # 8.56 steps -> 9
        (448.0, 448.0), (460.0, 448.0), (1e6, 448.0),   # saturating
        (-19.0, -20.0), (0.0, 0.0),
    ]
    for x, want in cases:
        assert oracle.e4m3_round(np.array([x]))[0] == want, x


def test_e4m3_round_matches_torch_cast():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.uniform(-448, 448, 20000),
                        rng.uniform(-1, 1, 20000) * 2.0 ** rng.integers(-12, 8, 20000),
                        np.arange(-2000, 2001) * 2.0 ** -11])    # every tie of small values
    mine = oracle.e4m3_round(x)
    theirs = torch.from_numpy(x).float().to(torch.float8_e4m3fn).double().numpy()
    xs = torch.from_numpy(x).float().double().numpy()           # torch rounds the fp32 value
    mine32 = oracle.e4m3_round(xs)
    assert np.array_equal(mine32, theirs)
    assert np.mean(mine == theirs) > 0.999


def _worked():
    # one query row (q = 1, D = 1, scale 1), key tiles of 2, lambda = 0 (nothing skipped)
    q = np.array([[[[1.0]]]])
    k = np.array([0.0, -L3, L2, L2 + math.log(1.3 * 2.0 ** -8)]).reshape(1, 1, 4, 1)
    v = np.array([1.0, 2.0, 3.0, 4.0]).reshape(1, 1, 4, 1)
    return q, k, v


def _worked_expected():
    # tile 0 (m' = 0): p = 1, 1/3 -> 2^8 p = 256, 85.33 -> e4m3 256, 88 -> w = 1, 0.34375
    # tile 1 (m' = ln 2): alpha = 1/2; p = 1, 1.3 * 2^-8 -> 2^8 p = 256, 1.3 -> 256, 1.25
    #                     -> w = 1, 1.25 / 256
    l = 0.5 * (1 + 1 / 3) + (1 + 1.3 * 2.0 ** -8)
    o = 0.5 * (1 * 1 + 0.34375 * 2) + (1 * 3 + (1.25 / 256) * 4)
    return o / l, math.log(2.0) + math.log(l)


def test_worked_example_with_a_growing_maximum():
    q, k, v = _worked()
    r = oracle.prefill(q, k, v, causal=False, lam=0.0, tile_q=1, tile_k=2, scale=1.0,
                       fp8_pv=True)
    o_want, lse_want = _worked_expected()
    assert abs(r.o[0, 0, 0, 0] - o_want) < 1e-14
    assert abs(r.lse[0, 0, 0] - lse_want) < 1e-14
    assert r.pot_ambiguous[0, 0, 0] == 0.0
    # and the exact oracle differs (the quantisation is visible at this size)
    e = oracle.prefill(q, k, v, causal=False, lam=0.0, tile_q=1, tile_k=2, scale=1.0)
    assert abs(e.o[0, 0, 0, 0] - o_want) > 1e-3


def test_ambiguous_rounding_is_reported():
    # 2^8 p = 17 lies on the midpoint between the e4m3 values 16 and 18
    q = np.array([[[[1.0]]]])
    k = np.array([0.0, math.log(17 / 256)]).reshape(1, 1, 2, 1)
    v = np.array([1.0, -1.0]).reshape(1, 1, 2, 1)
    r = oracle.prefill(q, k, v, causal=False, lam=0.0, tile_q=1, tile_k=2, scale=1.0,
                       fp8_pv=True)
    share = (17 / 256) / (1 + 17 / 256)
    assert abs(r.pot_ambiguous[0, 0, 0] - share) < 1e-12


def test_reduces_to_exact_when_weights_are_e4m3_values():
    # logits -n ln 2 below a first-tile maximum of 0: every 2^8 p = 2^(8-n) is an e4m3 value
    rng = np.random.default_rng(7)
    for trial in range(5):
        Skv, D = 24, 4
        n = rng.integers(0, 17, Skv)
        n[0] = 0
        q = np.ones((1, 1, 3, 1))
        k = (-n * L2).reshape(1, 1, Skv, 1)
        v = rng.standard_normal((1, 1, Skv, 1))
        a = oracle.prefill(q, k, v, causal=False, lam=0.0, tile_q=4, tile_k=8, scale=1.0,
                           fp8_pv=True)
        b = oracle.prefill(q, k, v, causal=False, lam=0.0, tile_q=4, tile_k=8, scale=1.0)
        assert np.allclose(a.o, b.o, rtol=0, atol=1e-12)
        assert np.allclose(a.lse, b.lse, rtol=0, atol=1e-12)


@pytest.mark.parametrize("lam", [0.0, 1e-3, 0.05])
@pytest.mark.parametrize("causal", [True, False])
def test_bound_against_the_exact_oracle_and_same_mask(lam, causal):
    rng = np.random.default_rng(11)
    B, Hq, Hkv, Sq, Skv, D = 1, 2, 1, 37, 53 if not causal else 37, 8
    q = rng.standard_normal((B, Hq, Sq, D)) * 1.5
    k = rng.standard_normal((B, Hkv, Skv, D)) * 1.5
    v = rng.standard_normal((B, Hkv, Skv, D))
    a = oracle.prefill(q, k, v, causal=causal, lam=lam, tile_q=8, tile_k=16, fp8_pv=True)
    b = oracle.prefill(q, k, v, causal=causal, lam=lam, tile_q=8, tile_k=16)
    assert np.array_equal(a.mask, b.mask)
    assert np.allclose(a.lse, b.lse, rtol=0, atol=1e-12)      # same exact row sums
    vmax = np.abs(v).max()
    # per key |w - p| <= 2^-4 p (half an e4m3 step of 2^8 p, normal range) or 2^-18 (subnormal
    # range, 2^8 p < 2^-6); the row sum l >= 1 (the key holding the final maximum has p = 1)
    bound = (2.0 ** -4 + Skv * 2.0 ** -18) * vmax
    err = np.abs(a.o - b.o)
    assert np.all(err <= bound + 1e-12), err.max()
    assert err.max() > 0                                      # the quantisation is visible


# ---------------------------------------------------------------------------
# planted mistakes: each must break the worked example
# ---------------------------------------------------------------------------
def _w_no_scale(p):
    return oracle.e4m3_round(p), np.zeros_like(p, dtype=bool)


def _w_truncate(p):
    y = p * 256.0
    q = so.e4m3_step(y)
    return np.floor(y / q) * q / 256.0, np.zeros_like(p, dtype=bool)


def _upd_l_quantised(m, l, o, a, s, vtile):
    m_new = np.maximum(m, np.max(s, axis=1))
    with np.errstate(invalid="ignore"):
        alpha = np.where(m == so.NEG_INF, 0.0, np.exp(m - m_new))
        p = np.where(s == so.NEG_INF, 0.0, np.exp(s - m_new[:, None]))
    w, amb = so._fp8_pv_weights(p)
    return m_new, alpha * l + w.sum(axis=1), alpha[:, None] * o + w @ vtile, a


def _upd_old_anchor(m, l, o, a, s, vtile):
    m_new = np.maximum(m, np.max(s, axis=1))
    anchor = np.where(m == so.NEG_INF, m_new, m)
    with np.errstate(invalid="ignore"):
        alpha = np.where(m == so.NEG_INF, 0.0, np.exp(m - m_new))
        p = np.where(s == so.NEG_INF, 0.0, np.exp(s - anchor[:, None]))
        p_new = np.where(s == so.NEG_INF, 0.0, np.exp(s - m_new[:, None]))
    w, _ = so._fp8_pv_weights(p)
    w = w * np.exp(anchor - m_new)[:, None]
    return m_new, alpha * l + p_new.sum(axis=1), alpha[:, None] * o + w @ vtile, a


@pytest.mark.parametrize("mutant", ["no_scale", "truncate", "l_quantised", "old_anchor"])
def test_planted_mistakes_are_caught(monkeypatch, mutant):
    if mutant == "no_scale":
        monkeypatch.setattr(so, "_fp8_pv_weights", _w_no_scale)
    elif mutant == "truncate":
        monkeypatch.setattr(so, "_fp8_pv_weights", _w_truncate)
    elif mutant == "l_quantised":
        monkeypatch.setattr(so, "_online_update_fp8_pv", _upd_l_quantised)
    else:
        monkeypatch.setattr(so, "_online_update_fp8_pv", _upd_old_anchor)
    q, k, v = _worked()
    r = oracle.prefill(q, k, v, causal=False, lam=0.0, tile_q=1, tile_k=2, scale=1.0,
                       fp8_pv=True)
    o_want, lse_want = _worked_expected()
    assert abs(r.o[0, 0, 0, 0] - o_want) > 1e-6 or abs(r.lse[0, 0, 0] - lse_want) > 1e-6
