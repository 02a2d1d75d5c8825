"""Prefill with a caller-supplied block mask against the oracle, through the C ABI.

"NVIDIA Introduces Skip Softmax ...", "Benefits and Implementation": Skip Softmax
combined with a block selector.  Unselected (vote tile, key tile) pairs are not
visited: no exponentials, no P.V, no vote, no running-max update.
"""

import numpy as np
import pytest
import torch

import block_sparse_long_softmax_b300 as bs
import oracle
import synth
from gpu_helpers import assert_close, assert_masks, device_inputs, to_f64

pytestmark = pytest.mark.gpu


def _mask(w, tq, tk, density, seed, empty_tile=False):
    nqt, nkt = -(-w.Sq // tq), -(-w.Skv // tk)
    rng = np.random.default_rng(seed)
    m = rng.random((w.B, w.Hq, nqt, nkt)) < density
    if empty_tile:
        m[0, 0, nqt // 2, :] = False          # a query tile with no selected key tile
    return m


def _run(w, lam, tq, tk, sel, heads=None, qtiles=None):
    q, k, v, _ = device_inputs(w)
    bm = torch.tensor(sel.astype(np.uint8), device=q.device)
    out = bs.prefill(q, k, v, lam, causal=w.causal, tile_q=tq, tile_k=tk, return_lse=True,
                     return_mask=True, return_visited=True, block_mask=bm)
    assert bs.check() == 0
    G = w.Hq // w.Hkv
    mask = out.skip_mask.cpu().numpy().astype(np.int8)
    mask = np.where(mask == 2, -1, mask).astype(np.int8)
    lse = out.lse.cpu().numpy()
    heads = heads or [(b, h) for b in range(w.B) for h in range(w.Hq)]
    for (b, h) in heads:
        qh, kh, vh = to_f64(q[b, h]), to_f64(k[b, h // G]), to_f64(v[b, h // G])
        nqt = -(-w.Sq // tq)
        for t in (range(nqt) if qtiles is None else qtiles):
            r0, r1 = t * tq, min((t + 1) * tq, w.Sq)
            ot, lt, mt, gt, _ = oracle.prefill_qtile(qh, kh, vh, t, tile_q=tq, tile_k=tk,
                                                     causal=w.causal, lam=lam,
                                                     scale=1.0 / np.sqrt(w.D),
                                                     block_mask_row=sel[b, h, t])
            og = to_f64(out.o[b, h, r0:r1])
            assert np.all(np.isfinite(og))
            assert_close(og, ot, f"o[b={b},h={h},t={t}]")
            fin = np.isfinite(lt)
            assert np.all(lse[b, h, r0:r1][~fin] == -np.inf), f"lse -inf rows b={b},h={h},t={t}"
            assert np.all(np.abs(lse[b, h, r0:r1][fin] - lt[fin]) < 2e-2), f"lse[b={b},h={h},t={t}]"
            assert_masks(mask[b, h, t], mt, gt, f"mask[b={b},h={h},t={t}]")
    vis = out.visited_counts.cpu().numpy()
    assert np.array_equal(vis, (mask >= 0).sum(axis=(0, 2, 3)))
    assert np.array_equal(out.skip_counts.cpu().numpy(), (mask == 1).sum(axis=(0, 2, 3)))
    return out


CASES = [
    (dict(B=1, Hq=4, Hkv=2, Sq=700, Skv=700, D=128, window=128), 128, 128, 0.5, True),
    (dict(B=1, Hq=4, Hkv=2, Sq=700, Skv=700, D=128, window=128), 64, 64, 0.4, True),
    (dict(B=1, Hq=4, Hkv=2, Sq=700, Skv=700, D=128, window=128), 64, 128, 0.6, False),
    (dict(B=1, Hq=4, Hkv=2, Sq=700, Skv=700, D=128, window=128), 128, 64, 0.3, False),
    (dict(B=2, Hq=2, Hkv=1, Sq=520, Skv=520, D=64, window=64), 128, 128, 0.5, True),
    (dict(B=1, Hq=2, Hkv=2, Sq=200, Skv=777, D=128, window=128), 128, 128, 0.5, False),
    (dict(B=1, Hq=2, Hkv=1, Sq=300, Skv=520, D=128, window=128, causal=False), 128, 128, 0.5, True),
]


@pytest.mark.parametrize("lam", [0.0, 1e-2])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_blockmask_prefill_parity(case, lam):
    over, tq, tk, density, empty = CASES[case]
    w = synth.WORKLOADS["prefill_32k_gqa8"].with_(**over)
    _run(w, lam, tq, tk, _mask(w, tq, tk, density, case, empty))


def test_blockmask_prefill_all_selected_equals_no_mask():
    w = synth.WORKLOADS["prefill_32k_gqa8"].with_(B=1, Hq=4, Hkv=1, Sq=900, Skv=900, window=128)
    q, k, v, _ = device_inputs(w)
    ref = bs.prefill(q, k, v, 1e-3, return_mask=True)
    ones = torch.ones((1, 4, 8, 8), dtype=torch.uint8, device=q.device)
    out = bs.prefill(q, k, v, 1e-3, return_mask=True, block_mask=ones)
    assert torch.equal(out.o, ref.o) and torch.equal(out.skip_mask, ref.skip_mask)


def test_blockmask_prefill_32k_sampled():
    w = synth.WORKLOADS["prefill_32k_gqa8"]
    sel = _mask(w, 128, 128, 0.5, 99)
    _run(w, 1e-3, 128, 128, sel, heads=[(0, 3)], qtiles=[0, 61, w.Sq // 128 - 1])
