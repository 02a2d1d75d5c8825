"""Plant plausible mistakes in the oracle (on the CPU) and check a pin catches each.

Each mutant replaces one step of the oracle's tile loop with a wrong variant;
the pins of ``pins.py`` must then fail on a small planted problem.
"""

import math

import numpy as np
import pytest

import oracle
import synth
from oracle import skipsm_oracle as so
from pins import check_decode, check_prefill

NEG_INF = -np.inf


def _vote_any(d, lam):
    if lam <= 0:
        return False, math.inf
    return bool(np.any(d < math.log(lam))), 1.0


def _gap_sign(m_loc, m_run):
    d = so.__dict__["_row_gap_orig"](m_loc, m_run)
    return np.where(np.isfinite(d), -d, d)


def _gap_no_first(m_loc, m_run):
    with np.errstate(invalid="ignore"):
        d = m_loc - np.where(m_run == NEG_INF, 0.0, m_run)
    return np.where(m_loc == NEG_INF, NEG_INF, d)


def _update_no_o_rescale(m, l, o, s, vt):
    m_new, l_new, _ = so.__dict__["_online_update_orig"](m, l, o, s, vt)
    with np.errstate(invalid="ignore"):
        p = np.where(s == NEG_INF, 0.0, np.exp(s - m_new[:, None]))
    return m_new, l_new, o + p @ vt


def _update_no_l_rescale(m, l, o, s, vt):
    m_new, _, o_new = so.__dict__["_online_update_orig"](m, l, o, s, vt)
    with np.errstate(invalid="ignore"):
        p = np.where(s == NEG_INF, 0.0, np.exp(s - m_new[:, None]))
    return m_new, l + p.sum(axis=1), o_new


def _logits_causal_off_by_one(qrows, ktile, scale, qpos, kidx, causal):
    s = (qrows @ ktile.T) * scale
    if causal:
        s = np.where(kidx[None, :] >= qpos[:, None], NEG_INF, s)
    return s


def _logits_no_scale(qrows, ktile, scale, qpos, kidx, causal):
    return so.__dict__["_tile_logits_orig"](qrows, ktile, 1.0, qpos, kidx, causal)


def _finish_no_log(m, l, o):
    return o / l[:, None], m + l


MUTANTS = {
    "vote_any_row": ("_vote", _vote_any),
    "gap_sign_flipped": ("_row_gap", _gap_sign),
    "first_tile_not_forced": ("_row_gap", _gap_no_first),
    "output_not_rescaled": ("_online_update", _update_no_o_rescale),
    "rowsum_not_rescaled": ("_online_update", _update_no_l_rescale),
    "causal_off_by_one": ("_tile_logits", _logits_causal_off_by_one),
    "scale_dropped": ("_tile_logits", _logits_no_scale),
    "lse_without_log": ("_finish", _finish_no_log),
}


@pytest.fixture(scope="module")
def planted():
    w = synth.WORKLOADS["prefill_1k_d64"].with_(Sq=256, Skv=256, window=64)
    _, qb, kb, vb = synth.gen_all(w)
    return tuple(synth.bf16_bits_to_f64(x) for x in (qb, kb, vb))


@pytest.fixture(scope="module")
def planted_decode():
    w = synth.WORKLOADS["decode_32k_gqa8"].with_(B=1, Hq=8, Hkv=1, Skv=1024, window=128)
    _, qb, kb, vb = synth.gen_all(w)
    return tuple(synth.bf16_bits_to_f64(x) for x in (qb, kb, vb))


def _run_all_pins(q, k, v, qd, kd, vd):
    for lam in (0.0, 1e-3, 3e-2):
        check_prefill(q, k, v, causal=True, lam=lam, tile_q=32, tile_k=32)
        check_decode(qd, kd, vd, lam=lam, num_splits=3, tile_k=64)
    # every logit of the first tile far below zero: only the forced first visit keeps it
    qn = np.array([[[[1.0], [0.5]]]])
    kn = np.array([[[[-5.0], [-6.0], [1.0], [-9.0]]]])
    vn = np.array([[[[1.0], [2.0], [3.0], [4.0]]]])
    check_prefill(qn, kn, vn, causal=False, lam=0.5, tile_q=2, tile_k=2, scale=1.0)


def test_unmutated_oracle_passes(planted, planted_decode):
    _run_all_pins(*planted, *planted_decode)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, planted, planted_decode, monkeypatch):
    attr, fn = MUTANTS[name]
    so.__dict__.setdefault(attr + "_orig", getattr(so, attr))
    monkeypatch.setattr(so, attr, fn)
    with pytest.raises(AssertionError):
        _run_all_pins(*planted, *planted_decode)


def test_mutant_split_combine_unnormalised(planted_decode, monkeypatch):
    """A combine that forgets to renormalise the split weights must be caught."""
    orig = so.decode_group

    def bad(qg, kh, vh, **kw):
        o, lse, mask, margin, parts = orig(qg, kh, vh, **kw)
        o2 = sum(p[0] for p in parts) / len(parts)
        return o2, lse, mask, margin, parts

    monkeypatch.setattr(so, "decode_group", bad)
    qd, kd, vd = planted_decode
    with pytest.raises(AssertionError):
        check_decode(qd, kd, vd, lam=0.0, num_splits=3, tile_k=64)
