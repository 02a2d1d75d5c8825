"""The prefill with V loads after the vote (v_load="after_vote") against the oracle and
against the default schedule ("NVIDIA Introduces Skip Softmax ...", "Benefits and
Implementation": a skipped block's values need not be read).

Loading V_j only once a query tile of the CTA keeps key tile j changes when the V rows
arrive in shared memory, not what is computed: outputs, LSE, masks and counts must be
bit-identical to the default schedule, and match the oracle at the usual tolerances.
"""

import numpy as np
import pytest
import torch

import block_sparse_long_softmax_b300 as bs
import oracle
import synth
from gpu_helpers import assert_close, assert_masks, device_inputs, to_f64

pytestmark = pytest.mark.gpu

CASES = [
    (dict(B=1, Hq=4, Hkv=2, Sq=700, Skv=700, D=128, window=128), 128),
    (dict(B=1, Hq=4, Hkv=2, Sq=700, Skv=700, D=128, window=128), 64),
    (dict(B=2, Hq=2, Hkv=1, Sq=200, Skv=777, D=128, window=128), 128),
    (dict(B=1, Hq=2, Hkv=1, Sq=300, Skv=520, D=128, window=128, causal=False), 128),
    (dict(B=1, Hq=4, Hkv=2, Sq=700, Skv=700, D=128, window=128, sink=0, bump=20.0), 128),
]


def _pair(w, lam, tq, **kw):
    q, k, v, _ = device_inputs(w)
    outs = [bs.prefill(q, k, v, lam, causal=w.causal, tile_q=tq, return_lse=True,
                       return_mask=True, return_visited=True, v_load=mode, **kw)
            for mode in ("ahead", "after_vote")]
    assert bs.check() == 0
    a, b = outs
    assert torch.equal(a.o, b.o) and torch.equal(a.lse, b.lse)
    assert torch.equal(a.skip_mask, b.skip_mask) and torch.equal(a.skip_counts, b.skip_counts)
    return q, k, v, b


@pytest.mark.parametrize("lam", [0.0, 1e-3, 1e-2])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_v_after_vote_parity_small(case, lam):
    over, tq = CASES[case]
    w = synth.WORKLOADS["prefill_32k_gqa8"].with_(**over)
    q, k, v, out = _pair(w, lam, tq)
    G = w.Hq // w.Hkv
    mask = out.skip_mask.cpu().numpy().astype(np.int8)
    mask = np.where(mask == 2, -1, mask)
    lse = out.lse.cpu().numpy()
    for b in range(w.B):
        for h in range(w.Hq):
            qh, kh, vh = to_f64(q[b, h]), to_f64(k[b, h // G]), to_f64(v[b, h // G])
            for t in range(-(-w.Sq // tq)):
                r0, r1 = t * tq, min((t + 1) * tq, w.Sq)
                ot, lt, mt, gt, _ = oracle.prefill_qtile(qh, kh, vh, t, tile_q=tq, tile_k=128,
                                                         causal=w.causal, lam=lam,
                                                         scale=1.0 / np.sqrt(w.D))
                assert_close(to_f64(out.o[b, h, r0:r1]), ot, f"o[b={b},h={h},t={t}]")
                assert np.all(np.abs(lse[b, h, r0:r1] - lt) < 2e-2)
                assert_masks(mask[b, h, t], mt, gt, f"mask[b={b},h={h},t={t}]")


def test_v_after_vote_block_mask_identical():
    w = synth.WORKLOADS["prefill_32k_gqa8"].with_(B=1, Hq=4, Hkv=2, Sq=1000, Skv=1000, window=128)
    nqt = -(-w.Sq // 128)
    rng = np.random.default_rng(3)
    bm = torch.tensor((rng.random((w.B, w.Hq, nqt, nqt)) < 0.6).astype(np.uint8), device="cuda")
    _pair(w, 1e-3, 128, block_mask=bm)


@pytest.mark.parametrize("lam", [0.0, 3e-3, 1e-2])
def test_v_after_vote_32k_identical(lam):
    w = synth.WORKLOADS["prefill_32k_gqa8"]
    _pair(w, lam, 128)
