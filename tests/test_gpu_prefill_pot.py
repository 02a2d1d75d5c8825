"""GPU parity of the Rowmax-PoT prefill weights against the oracle.

"Approximating Softmax in Pretrained LLMs: Model Sensitivity and Kernel
Acceleration" (AI Summary, Abstract): powers of two anchored at each row maximum.
The oracle computes the exponents in fp64 and reports, per row, the share of the
weight sum carried by keys whose exponent lies within 1e-4 of a rounding boundary,
where fp32 logits may round the other way (each such key's weight may then be off by
a factor of 2).  The kernel rounds the factor from the running max to the
accumulator's reference to bf16 (relative error <= 2^-9, common to one row and tile).
Tolerance per output element, from that arithmetic:
    1e-2 + 1e-2 |o| + (2^-9 + ambiguous share) * 2 max|v|.
Skip masks are unchanged by PoT and must match on every tile with margin > 1e-3.
"""

import numpy as np
import pytest
import torch

import block_sparse_long_softmax_b300 as bs
import oracle
import synth
from gpu_helpers import ATOL, RTOL, assert_masks, device_inputs, to_f64

pytestmark = pytest.mark.gpu


def _compare(w, q, k, v, out, lam, heads, qtiles=None):
    G = w.Hq // w.Hkv
    mask = out.skip_mask.cpu().numpy().astype(np.int8)
    mask = np.where(mask == 2, -1, mask).astype(np.int8)
    lse = out.lse.cpu().numpy()
    for (b, h) in heads:
        qh, kh, vh = to_f64(q[b, h]), to_f64(k[b, h // G]), to_f64(v[b, h // G])
        vmax = float(np.max(np.abs(vh)))
        nqt = -(-w.Sq // out.tile_q)
        for t in (range(nqt) if qtiles is None else qtiles):
            r0, r1 = t * out.tile_q, min((t + 1) * out.tile_q, w.Sq)
            ot, lt, mt, gt, amb = oracle.prefill_qtile(qh, kh, vh, t, tile_q=out.tile_q,
                                                       tile_k=out.tile_k, causal=w.causal,
                                                       lam=lam, scale=1.0 / np.sqrt(w.D),
                                                       pot=True)
            og = to_f64(out.o[b, h, r0:r1])
            bound = ATOL + RTOL * np.abs(ot) + (2.0 ** -9 + amb[:, None]) * 2 * vmax
            bad = np.abs(og - ot) > bound
            assert not bad.any(), (f"o[b={b},h={h},t={t}]: {bad.sum()} elements out of "
                                   f"tolerance, max err {np.abs(og - ot).max():.3e}")
            lbound = 2e-2 + 2.0 ** -8 + 2 * amb
            assert np.all(np.abs(lse[b, h, r0:r1] - lt) < lbound), f"lse[b={b},h={h},t={t}]"
            assert_masks(mask[b, h, t], mt, gt, f"mask[b={b},h={h},t={t}]")


def _run(w, lam, tq=0, tk=0):
    q, k, v, _ = device_inputs(w)
    out = bs.prefill(q, k, v, lam, causal=w.causal, tile_q=tq, tile_k=tk, return_lse=True,
                     return_mask=True, return_visited=True, exp_mode="pot")
    assert bs.check() == 0
    return q, k, v, out


@pytest.mark.parametrize("lam", [0.0, 1e-2])
def test_pot_prefill_1k_d64_full(lam):
    w = synth.WORKLOADS["prefill_1k_d64"]
    q, k, v, out = _run(w, lam, 64, 64)
    _compare(w, q, k, v, out, lam, [(0, 0)])


CASES = [
    (dict(B=1, Hq=4, Hkv=2, Sq=700, Skv=700, D=128, window=128), 128, 128),
    (dict(B=1, Hq=4, Hkv=2, Sq=700, Skv=700, D=128, window=128), 64, 64),
    (dict(B=2, Hq=2, Hkv=1, Sq=520, Skv=520, D=64, window=64), 128, 128),
    (dict(B=1, Hq=2, Hkv=2, Sq=200, Skv=777, D=128, window=128), 128, 128),
    (dict(B=1, Hq=2, Hkv=1, Sq=300, Skv=520, D=128, window=128, causal=False), 128, 128),
]


@pytest.mark.parametrize("lam", [0.0, 1e-3, 1e-2])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_pot_prefill_parity_small(case, lam):
    over, tq, tk = CASES[case]
    w = synth.WORKLOADS["prefill_32k_gqa8"].with_(**over)
    q, k, v, out = _run(w, lam, tq, tk)
    _compare(w, q, k, v, out, lam, [(b, h) for b in range(w.B) for h in range(w.Hq)])


def test_pot_prefill_32k_sampled_and_masks_match_exact():
    w = synth.WORKLOADS["prefill_32k_gqa8"]
    q, k, v, _ = device_inputs(w)
    lam = 1e-3
    out = bs.prefill(q, k, v, lam, return_lse=True, return_mask=True, return_visited=True,
                     exp_mode="pot")
    assert bs.check() == 0
    nqt = w.Sq // 128
    _compare(w, q, k, v, out, lam, [(0, 5)], qtiles=[0, 101, nqt - 1])
    # the vote only looks at exact maxima: the same tiles are skipped as without PoT
    ref = bs.prefill(q, k, v, lam, return_mask=True)
    assert torch.equal(out.skip_mask, ref.skip_mask)
    assert torch.equal(out.skip_counts, ref.skip_counts)
