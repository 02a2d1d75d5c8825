"""Pins of the oracle's block mask, decode and prefill ("NVIDIA Introduces Skip Softmax ...",
"Benefits and Implementation": Skip Softmax combined with another sparse-attention
method).  Tiles outside the mask are not visited; the skip rule runs over the selected
tiles of each split.  Checked against SDPA restricted to the selected keys (a library
routine), invariances, and hand-worked examples (D = 1, scale = 1: logit = q * k).
"""

import math

import numpy as np
import pytest

import oracle
from oracle import skipsm_oracle as so
from pins import sdpa


def E(x):
    return math.exp(x)


def _dec(q, k, v, lam, splits, mask, tile_k=2):
    return oracle.decode(q, k, v, lam=lam, num_splits=splits, tile_k=tile_k, scale=1.0,
                         block_mask=mask)


def test_worked_unselected_tile_does_not_raise_the_running_max():
    # one head, keys [0, 1 | 9, 9 | 2, -3], tiles of 2, one split, tile 1 not selected.
    # Running max before tile 2 is 1 (tile 0 only), tile 2's max is 2: gap +1 -> kept
    # for any lambda <= 1.  Had tile 1 been visited, the gap would be 2 - 9 = -7 and
    # lambda = e^-5 would skip it.
    q = np.ones((1, 1, 1))
    k = np.array([0.0, 1.0, 9.0, 9.0, 2.0, -3.0]).reshape(1, 1, 6, 1)
    v = np.array([1.0, 2.0, 100.0, 100.0, 3.0, 4.0]).reshape(1, 1, 6, 1)
    sel = np.array([[[True, False, True]]])
    r = _dec(q, k, v, E(-5), 1, sel)
    assert r.mask[0, 0].tolist() == [0, -1, 0]
    z = E(0) + E(1) + E(2) + E(-3)
    want = (1 * E(0) + 2 * E(1) + 3 * E(2) + 4 * E(-3)) / z
    assert abs(r.o[0, 0, 0] - want) < 1e-14
    assert abs(r.lse[0, 0] - math.log(z)) < 1e-14
    # all tiles selected: tile 2 is skipped at e^-5 (gap -7)
    r = _dec(q, k, v, E(-5), 1, None)
    assert r.mask[0, 0].tolist() == [0, 0, 1]


def test_worked_empty_split_and_empty_group():
    q = np.ones((1, 2, 1))                     # two heads share one kv head
    k = np.array([1.0, 0.0, 2.0, 5.0]).reshape(1, 1, 4, 1)
    v = np.array([1.0, 2.0, 3.0, 4.0]).reshape(1, 1, 4, 1)
    # two splits of one tile each; the second split has no selected tile
    r = _dec(q, k, v, 0.0, 2, np.array([[[True, False]]]))
    want = (1 * E(1) + 2 * E(0)) / (E(1) + E(0))
    assert np.allclose(r.o[0, :, 0], want, rtol=0, atol=1e-14)
    assert r.mask[0, 0].tolist() == [0, -1]
    # no selected tile at all: output 0, log-sum-exp -inf
    r = _dec(q, k, v, 0.0, 2, np.array([[[False, False]]]))
    assert np.all(r.o == 0.0) and np.all(r.lse == -np.inf)


@pytest.mark.parametrize("splits", [1, 3, 7])
@pytest.mark.parametrize("seed", range(3))
def test_lambda0_equals_sdpa_on_selected_keys(splits, seed):
    rng = np.random.default_rng(seed)
    B, Hkv, G, Skv, D, tk = 2, 2, 3, 37, 8, 4
    q = rng.standard_normal((B, Hkv * G, D))
    k = rng.standard_normal((B, Hkv, Skv, D)) * 2
    v = rng.standard_normal((B, Hkv, Skv, D))
    nblk = -(-Skv // tk)
    sel = rng.random((B, Hkv, nblk)) < 0.5
    sel[0, 0, :] = False
    sel[0, 0, 3] = True                         # a group with a single selected tile
    r = oracle.decode(q, k, v, lam=0.0, num_splits=splits, tile_k=tk, block_mask=sel)
    for b in range(B):
        for hk in range(Hkv):
            keys = np.repeat(sel[b, hk], tk)[:Skv]
            allowed = np.broadcast_to(keys, (G, Skv))
            want = sdpa(q[b, hk * G:(hk + 1) * G], k[b, hk], v[b, hk], allowed, 1 / math.sqrt(D))
            assert np.max(np.abs(r.o[b, hk * G:(hk + 1) * G] - want)) < 1e-12


def test_all_selected_equals_no_mask_and_counts_only_selected():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((1, 4, 8))
    k = rng.standard_normal((1, 2, 50, 8)) * 3
    v = rng.standard_normal((1, 2, 50, 8))
    a = oracle.decode(q, k, v, lam=0.05, num_splits=3, tile_k=4)
    b = oracle.decode(q, k, v, lam=0.05, num_splits=3, tile_k=4,
                      block_mask=np.ones((1, 2, 13), dtype=bool))
    assert np.array_equal(a.o, b.o) and np.array_equal(a.mask, b.mask)
    sel = rng.random((1, 2, 13)) < 0.6
    c = oracle.decode(q, k, v, lam=0.05, num_splits=3, tile_k=4, block_mask=sel)
    assert np.all((c.mask == -1) == ~sel)
    assert np.array_equal(c.skip_counts, np.repeat((c.mask == 1).sum(axis=(0, 2)), 2))


def test_unselected_keys_do_not_matter():
    rng = np.random.default_rng(11)
    q = rng.standard_normal((1, 2, 8))
    k = rng.standard_normal((1, 1, 40, 8)) * 2
    v = rng.standard_normal((1, 1, 40, 8))
    sel = rng.random((1, 1, 10)) < 0.5
    a = oracle.decode(q, k, v, lam=0.02, num_splits=2, tile_k=4, block_mask=sel)
    k2, v2 = k.copy(), v.copy()
    for j in np.where(~sel[0, 0])[0]:
        k2[0, 0, 4 * j:4 * j + 4] += 50.0       # would dominate every softmax if visited
        v2[0, 0, 4 * j:4 * j + 4] = 1e6
    b = oracle.decode(q, k2, v2, lam=0.02, num_splits=2, tile_k=4, block_mask=sel)
    assert np.array_equal(a.o, b.o) and np.array_equal(a.mask, b.mask)


# planted mistakes in the oracle must fail a pin above
def _mutant_max_over_unselected(qg, kh, vh, *, lam, num_splits, tile_k=64, scale=None,
                                block_mask=None):
    # visits unselected tiles for the running max (but adds nothing for them)
    if block_mask is None:
        return _ORIG(qg, kh, vh, lam=lam, num_splits=num_splits, tile_k=tile_k, scale=scale)
    vh2 = vh.copy()
    for j in np.where(~np.asarray(block_mask))[0]:
        vh2[j * tile_k:(j + 1) * tile_k] = 0.0
    o, lse, mask, margin, parts = _ORIG(qg, kh, vh2, lam=lam, num_splits=num_splits,
                                        tile_k=tile_k, scale=scale)
    mask = np.where(np.asarray(block_mask), mask, -1).astype(np.int8)
    return o, lse, mask, margin, parts


def _mutant_ignore_mask(qg, kh, vh, *, lam, num_splits, tile_k=64, scale=None, block_mask=None):
    return _ORIG(qg, kh, vh, lam=lam, num_splits=num_splits, tile_k=tile_k, scale=scale)


_ORIG = so.decode_group


@pytest.mark.parametrize("fn", [_mutant_max_over_unselected, _mutant_ignore_mask])
def test_blockmask_mutants_are_caught(monkeypatch, fn):
    monkeypatch.setattr(so, "decode_group", fn)
    caught = 0
    for pin in (test_worked_unselected_tile_does_not_raise_the_running_max,
                test_worked_empty_split_and_empty_group):
        try:
            pin()
        except (AssertionError, FloatingPointError, ValueError):
            caught += 1
    assert caught > 0


# ---------------------------------------------------------------------------
# prefill: a mask over (query tile, key tile) pairs
# ---------------------------------------------------------------------------
def test_worked_prefill_unselected_tile_not_in_running_max():
    # one row of logits [9, 9 | 1, 0 | 2, -3] (D = 1, q = 1), tiles of 2 keys, non-causal.
    # With key tile 0 unselected the running max before tile 2 is 1, tile 2's gap is +1:
    # kept.  With every tile selected, tiles 1 and 2 have gaps 1 - 9 and 2 - 9, and
    # lambda = e^-5 skips both.
    q = np.ones((1, 1, 1, 1))
    k = np.array([9.0, 9.0, 1.0, 0.0, 2.0, -3.0]).reshape(1, 1, 6, 1)
    v = np.array([100.0, 100.0, 1.0, 2.0, 3.0, 4.0]).reshape(1, 1, 6, 1)
    sel = np.array([False, True, True]).reshape(1, 1, 1, 3)
    r = oracle.prefill(q, k, v, causal=False, lam=E(-5), tile_q=1, tile_k=2, scale=1.0,
                       block_mask=sel)
    assert r.mask[0, 0, 0].tolist() == [-1, 0, 0]
    z = E(1) + E(0) + E(2) + E(-3)
    assert abs(r.o[0, 0, 0, 0] - (E(1) + 2 + 3 * E(2) + 4 * E(-3)) / z) < 1e-14
    r = oracle.prefill(q, k, v, causal=False, lam=E(-5), tile_q=1, tile_k=2, scale=1.0)
    assert r.mask[0, 0, 0].tolist() == [0, 1, 1]


def test_worked_prefill_row_without_selected_keys():
    # causal Sq = Skv = 4, tiles 2 x 2: query tile 1 selects only key tile 1; its rows
    # 2 and 3 see keys 2 and 2..3.  Query tile 0 selects nothing: output 0, lse -inf.
    q = np.ones((1, 1, 4, 1))
    k = np.array([5.0, 5.0, 0.0, 1.0]).reshape(1, 1, 4, 1)
    v = np.array([9.0, 9.0, 1.0, 2.0]).reshape(1, 1, 4, 1)
    sel = np.array([[False, False], [False, True]]).reshape(1, 1, 2, 2)
    r = oracle.prefill(q, k, v, causal=True, lam=0.0, tile_q=2, tile_k=2, scale=1.0,
                       block_mask=sel)
    o = r.o[0, 0, :, 0]
    assert o[0] == 0.0 and o[1] == 0.0 and np.all(r.lse[0, 0, :2] == -np.inf)
    assert abs(o[2] - 1.0) < 1e-15
    assert abs(o[3] - (1 * E(0) + 2 * E(1)) / (E(0) + E(1))) < 1e-14
    assert r.mask[0, 0].tolist() == [[-1, -1], [-1, 0]]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("seed", range(3))
def test_prefill_lambda0_equals_sdpa_on_selected_keys(causal, seed):
    rng = np.random.default_rng(seed)
    B, Hq, Hkv, Sq, Skv, D, tq, tk = 1, 2, 1, 11, 14, 8, 3, 4
    q = rng.standard_normal((B, Hq, Sq, D))
    k = rng.standard_normal((B, Hkv, Skv, D)) * 2
    v = rng.standard_normal((B, Hkv, Skv, D))
    nqt, nkt = -(-Sq // tq), -(-Skv // tk)
    sel = rng.random((B, Hq, nqt, nkt)) < 0.6
    r = oracle.prefill(q, k, v, causal=causal, lam=0.0, tile_q=tq, tile_k=tk,
                       block_mask=sel)
    for h in range(Hq):
        rows_sel = np.repeat(np.repeat(sel[0, h], tq, axis=0)[:Sq], tk, axis=1)[:, :Skv]
        from pins import causal_allowed
        allowed = rows_sel & causal_allowed(Sq, Skv, causal)
        has = allowed.any(axis=1)
        want = sdpa(q[0, h][has], k[0, 0], v[0, 0], allowed[has], 1 / math.sqrt(D))
        assert np.max(np.abs(r.o[0, h][has] - want)) < 1e-12
        assert np.all(r.o[0, h][~has] == 0.0) and np.all(r.lse[0, h][~has] == -np.inf)


def test_prefill_all_selected_equals_no_mask_and_unselected_keys_do_not_matter():
    rng = np.random.default_rng(9)
    q = rng.standard_normal((1, 2, 12, 8))
    k = rng.standard_normal((1, 1, 12, 8)) * 3
    v = rng.standard_normal((1, 1, 12, 8))
    a = oracle.prefill(q, k, v, causal=True, lam=0.05, tile_q=4, tile_k=4)
    b = oracle.prefill(q, k, v, causal=True, lam=0.05, tile_q=4, tile_k=4,
                       block_mask=np.ones((1, 2, 3, 3), dtype=bool))
    assert np.array_equal(a.o, b.o) and np.array_equal(a.mask, b.mask)
    # key tile 1 selected by no query tile: changing its keys and values changes nothing
    sel = np.ones((1, 2, 3, 3), dtype=bool)
    sel[:, :, :, 1] = False
    c = oracle.prefill(q, k, v, causal=True, lam=0.05, tile_q=4, tile_k=4, block_mask=sel)
    k2, v2 = k.copy(), v.copy()
    k2[0, 0, 4:8] += 40.0
    v2[0, 0, 4:8] = 1e6
    d = oracle.prefill(q, k2, v2, causal=True, lam=0.05, tile_q=4, tile_k=4, block_mask=sel)
    assert np.array_equal(c.o, d.o) and np.array_equal(c.mask, d.mask)
