"""The fp64 oracle against what the mathematics fixes (CPU only).

The Skip Softmax pages print no worked example, so the pins are: dense
attention from a library routine at lambda = 0, the closed-form mask and
kept-key output, monotonicity in lambda, the analytic error bound, and small
examples worked out by hand below.
"""

import math

import numpy as np
import pytest

import oracle
import synth
from pins import check_decode, check_prefill, sdpa, causal_allowed

E = math.exp


def _rand(rng, *shape, scale=1.0):
    return rng.standard_normal(shape) * scale


# ---------------------------------------------------------------------------
# hand-worked examples (D = 1, scale = 1, so logit = q * k)
# ---------------------------------------------------------------------------
def test_worked_prefill_noncausal():
    # logits of both rows: [3, 0 | -10, 2]; tiles of 2 keys, one query tile of 2 rows.
    q = np.array([[[[1.0], [1.0]]]])
    k = np.array([[[[3.0], [0.0], [-10.0], [2.0]]]])
    v = np.array([[[[1.0], [2.0], [3.0], [4.0]]]])
    # tile 1: local max 2, running max 3 -> gap -1.  lambda = e^-0.5: -1 < -0.5 -> skipped.
    r = oracle.prefill(q, k, v, causal=False, lam=E(-0.5), tile_q=2, tile_k=2, scale=1.0)
    assert r.mask[0, 0, 0].tolist() == [0, 1]
    want = (E(3) * 1 + E(0) * 2) / (E(3) + E(0))
    assert abs(r.o[0, 0, 0, 0] - want) < 1e-14 and abs(r.o[0, 0, 1, 0] - want) < 1e-14
    assert abs(r.lse[0, 0, 0] - math.log(E(3) + 1)) < 1e-14
    assert abs(r.margin[0, 0, 0, 1] - 0.5) < 1e-14
    # lambda = e^-2: -1 < -2 is false -> kept, output is the full softmax.
    r = oracle.prefill(q, k, v, causal=False, lam=E(-2), tile_q=2, tile_k=2, scale=1.0)
    assert r.mask[0, 0, 0].tolist() == [0, 0]
    z = E(3) + E(0) + E(-10) + E(2)
    want = (E(3) * 1 + 2 + E(-10) * 3 + E(2) * 4) / z
    assert abs(r.o[0, 0, 0, 0] - want) < 1e-14


def test_worked_skipped_mass():
    # the non-causal example above at lambda = e^-0.5: key tile 1 (logits -10, 2) is skipped
    # for both rows.  Dense probabilities are e^s / z with z = e^3 + e^0 + e^-10 + e^2, so the
    # skipped mass is eps = (e^-10 + e^2) / z (about 0.2595) -- not 1 (all keys), not the kept
    # mass, not a single key's probability.
    q = np.array([[1.0], [1.0]])
    k = np.array([[3.0], [0.0], [-10.0], [2.0]])
    v = np.array([[1.0], [2.0], [3.0], [4.0]])
    o_dense, lse, p = oracle.dense_attention(q, k, v, causal=False, scale=1.0)
    skipped = np.array([[False, False, True, True]] * 2)
    eps = oracle.skipped_mass(p, skipped)
    z = E(3) + E(0) + E(-10) + E(2)
    want = (E(-10) + E(2)) / z
    assert np.allclose(eps, want, rtol=0, atol=1e-15)
    assert abs(want - 0.25949) < 1e-4
    assert abs(lse[0] - math.log(z)) < 1e-14
    # the output moves by exactly eps times (skipped keys' mean value - kept output):
    # o_dense = (1 - eps) o_kept + eps vbar_skipped
    o_kept = (E(3) * 1 + E(0) * 2) / (E(3) + E(0))
    vbar = (E(-10) * 3 + E(2) * 4) / (E(-10) + E(2))
    assert abs(o_dense[0, 0] - ((1 - want) * o_kept + want * vbar)) < 1e-14
    r = oracle.prefill(q[None, None], k[None, None], v[None, None], causal=False, lam=E(-0.5),
                       tile_q=2, tile_k=2, scale=1.0)
    assert abs(r.o[0, 0, 0, 0] - o_kept) < 1e-14
    assert np.all(np.abs(o_dense[:, 0] - r.o[0, 0, :, 0]) <= eps * (4.0 - 1.0))


def test_worked_prefill_causal():
    # Sq = Skv = 4, tiles 2x2; row i sees keys <= i.
    q = np.ones((1, 1, 4, 1))
    k = np.array([3.0, 0.0, -10.0, 2.0]).reshape(1, 1, 4, 1)
    v = np.array([1.0, 2.0, 3.0, 4.0]).reshape(1, 1, 4, 1)
    r = oracle.prefill(q, k, v, causal=True, lam=E(-0.5), tile_q=2, tile_k=2, scale=1.0)
    # query tile 0 visits key tile 0 only; query tile 1: row 2 gap -13, row 3 gap -1 -> skip
    assert r.mask[0, 0].tolist() == [[0, -1], [0, 1]]
    o = r.o[0, 0, :, 0]
    assert abs(o[0] - 1.0) < 1e-15
    assert abs(o[1] - (E(3) + 2) / (E(3) + 1)) < 1e-14
    assert abs(o[2] - (E(3) + 2) / (E(3) + 1)) < 1e-14
    assert abs(o[3] - (E(3) + 2) / (E(3) + 1)) < 1e-14
    # lambda = e^-2: row 3's gap -1 keeps the tile for both rows
    r = oracle.prefill(q, k, v, causal=True, lam=E(-2), tile_q=2, tile_k=2, scale=1.0)
    assert r.mask[0, 0].tolist() == [[0, -1], [0, 0]]
    o = r.o[0, 0, :, 0]
    assert abs(o[2] - (E(3) + 2 + 3 * E(-10)) / (E(3) + 1 + E(-10))) < 1e-14
    assert abs(o[3] - (E(3) + 2 + 3 * E(-10) + 4 * E(2)) / (E(3) + 1 + E(-10) + E(2))) < 1e-14


def test_worked_decode_split_restart():
    # two heads (q = 1, 2) share one kv head; 6 keys, tiles of 2, 2 splits -> tiles {0,1} | {2}
    q = np.array([[[1.0], [2.0]]])
    kk = np.array([3.0, 0.0, -10.0, 1.0, 0.5, 0.0])
    k = kk.reshape(1, 1, 6, 1)
    v = np.arange(1.0, 7.0).reshape(1, 1, 6, 1)
    lam = E(-1.5)
    r = oracle.decode(q, k, v, lam=lam, num_splits=2, tile_k=2, scale=1.0)
    # tile 1: gaps 1-3 = -2 and 2-6 = -4 -> skipped; tile 2 opens split 1 -> kept
    assert r.mask[0, 0].tolist() == [0, 1, 0]
    assert r.num_splits == 2
    for h, qq in enumerate([1.0, 2.0]):
        keys = [0, 1, 4, 5]
        want = sum(E(qq * kk[c]) * (c + 1) for c in keys) / sum(E(qq * kk[c]) for c in keys)
        assert abs(r.o[0, h, 0] - want) < 1e-14
    # one split: tile 2 is judged against running max 3 / 6: gaps -2.5 / -5 -> skipped too
    r1 = oracle.decode(q, k, v, lam=lam, num_splits=1, tile_k=2, scale=1.0)
    assert r1.mask[0, 0].tolist() == [0, 1, 1]
    assert r1.skip_counts.tolist() == [2, 2]


def test_worked_one_row_keeps_tile():
    # a tile is kept when any single row is above the threshold
    q = np.array([[[[1.0], [-1.0]]]])
    k = np.array([[[[2.0], [1.5]]]])
    v = np.array([[[[1.0], [5.0]]]])
    # tile 0 = key 0, tile 1 = key 1. row 0 gap -0.5; row 1: logits -2, -1.5 -> gap +0.5
    r = oracle.prefill(q, k, v, causal=False, lam=E(-0.25), tile_q=2, tile_k=1, scale=1.0)
    assert r.mask[0, 0, 0].tolist() == [0, 0]
    r = oracle.prefill(q[:, :, :1], k, v, causal=False, lam=E(-0.25), tile_q=1, tile_k=1, scale=1.0)
    assert r.mask[0, 0, 0].tolist() == [0, 1]


def test_lambda_one_skips_only_lower_tiles():
    # lambda = 1 skips a tile iff every row's local max is strictly below its running max
    q = np.array([[[[1.0]]]])
    k = np.array([[[[1.0], [1.0], [0.5], [2.0]]]])
    v = np.array([[[[1.0], [2.0], [3.0], [4.0]]]])
    r = oracle.prefill(q, k, v, causal=False, lam=1.0, tile_q=1, tile_k=1, scale=1.0)
    # gaps: +inf, 0 (not < 0), -0.5, +1
    assert r.mask[0, 0, 0].tolist() == [0, 0, 1, 0]


# ---------------------------------------------------------------------------
# random small problems: every pin, tails, GQA, causal / non-causal
# ---------------------------------------------------------------------------
PREFILL_CASES = [
    # B, Hq, Hkv, Sq, Skv, D, causal, tile_q, tile_k
    (1, 1, 1, 7, 7, 4, True, 2, 2),
    (1, 2, 1, 37, 53, 8, True, 8, 16),
    (2, 4, 2, 33, 33, 8, False, 16, 8),
    (1, 2, 2, 40, 64, 16, True, 16, 16),
    (1, 8, 1, 19, 45, 4, True, 4, 8),
    (1, 1, 1, 1, 1, 4, True, 4, 4),
    (1, 1, 1, 1, 30, 4, True, 64, 64),
]


@pytest.mark.parametrize("case", PREFILL_CASES)
@pytest.mark.parametrize("lam", [0.0, 1e-3, 0.05, 0.5])
def test_prefill_pins_random(case, lam):
    B, Hq, Hkv, Sq, Skv, D, causal, tq, tk = case
    rng = np.random.default_rng(hash((case, lam)) % 2**32)
    q = _rand(rng, B, Hq, Sq, D, scale=1.5)
    k = _rand(rng, B, Hkv, Skv, D, scale=1.5)
    v = _rand(rng, B, Hkv, Skv, D)
    check_prefill(q, k, v, causal=causal, lam=lam, tile_q=tq, tile_k=tk,
                  lam_grid=[0.0, 1e-4, 1e-3, 1e-2, 0.05, 0.2, 0.5, 1.0] if lam == 0.05 else None)


DECODE_CASES = [
    # B, Hq, Hkv, Skv, D, splits, tile_k
    (1, 2, 1, 6, 4, 2, 2),
    (2, 8, 1, 200, 8, 3, 16),
    (1, 8, 2, 131, 8, 5, 8),
    (1, 4, 4, 64, 16, 1, 64),
    (1, 8, 1, 7, 4, 7, 64),
]


@pytest.mark.parametrize("case", DECODE_CASES)
@pytest.mark.parametrize("lam", [0.0, 1e-3, 0.1])
def test_decode_pins_random(case, lam):
    B, Hq, Hkv, Skv, D, splits, tk = case
    rng = np.random.default_rng(hash((case, lam)) % 2**32)
    q = _rand(rng, B, Hq, D, scale=2.0)
    k = _rand(rng, B, Hkv, Skv, D, scale=2.0)
    v = _rand(rng, B, Hkv, Skv, D)
    check_decode(q, k, v, lam=lam, num_splits=splits, tile_k=tk)


def test_decode_splits_do_not_change_dense():
    rng = np.random.default_rng(5)
    q, k, v = _rand(rng, 1, 8, 16), _rand(rng, 1, 1, 300, 16), _rand(rng, 1, 1, 300, 16)
    outs = [oracle.decode(q, k, v, lam=0.0, num_splits=s, tile_k=32).o for s in (1, 2, 3, 10)]
    for o in outs[1:]:
        assert np.max(np.abs(o - outs[0])) < 1e-13


def test_split_geometry():
    assert oracle.decode_split_geometry(131072, 64, 64) == (2048, 32, 64)
    assert oracle.decode_split_geometry(130, 64, 16) == (3, 1, 3)     # empty splits dropped
    assert oracle.decode_split_geometry(64 * 10, 64, 4) == (10, 3, 4)
    assert oracle.decode_split_geometry(64 * 9, 64, 4) == (9, 3, 3)


# ---------------------------------------------------------------------------
# the planted workloads: pins at the small configuration, skipping really happens
# ---------------------------------------------------------------------------
def _planted_prefill(name, **over):
    w = synth.WORKLOADS[name].with_(**over)
    _, qb, kb, vb = synth.gen_all(w)
    return w, synth.bf16_bits_to_f64(qb), synth.bf16_bits_to_f64(kb), synth.bf16_bits_to_f64(vb)


def test_planted_prefill_small_pins():
    w, q, k, v = _planted_prefill("prefill_1k_d64", Sq=384, Skv=384)
    res = {}
    for lam in w.lambdas:
        res[lam] = check_prefill(q, k, v, causal=True, lam=lam, tile_q=64, tile_k=64)
    # the planted structure makes lambda = 1e-2 skip tiles and lambda = 0 none
    assert (res[1e-2].mask == 1).sum() > 0
    assert (res[0.0].mask == 1).sum() == 0


def test_planted_decode_small_pins():
    w = synth.WORKLOADS["decode_32k_gqa8"].with_(B=1, Hq=16, Hkv=2, Skv=4096)
    _, qb, kb, vb = synth.gen_all(w)
    q, k, v = (synth.bf16_bits_to_f64(x) for x in (qb, kb, vb))
    r = check_decode(q, k, v, lam=1e-2, num_splits=4, tile_k=64)
    assert 0 < (r.mask == 1).mean() < 1


def test_dense_attention_matches_sdpa():
    rng = np.random.default_rng(9)
    q, k, v = _rand(rng, 9, 8), _rand(rng, 13, 8), _rand(rng, 13, 8)
    o, lse, p = oracle.dense_attention(q, k, v, causal=True, scale=0.3)
    ref = sdpa(q, k, v, causal_allowed(9, 13, True), 0.3)
    assert np.max(np.abs(o - ref)) < 1e-13
    assert np.allclose(p.sum(axis=1), 1.0)
