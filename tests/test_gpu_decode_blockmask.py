"""Decode with a caller-supplied block mask against the oracle, through the C ABI.

"NVIDIA Introduces Skip Softmax ...", "Benefits and Implementation": Skip Softmax
combined with a block selector.  Unselected 64-key tiles are never read or voted on;
the skip rule runs over the selected tiles of each split.
"""

import numpy as np
import pytest
import torch

import block_sparse_long_softmax_b300 as bs
import oracle
import synth
from gpu_helpers import assert_close, assert_masks, device_inputs, to_f64

pytestmark = pytest.mark.gpu


def _mask(w, density, seed, empty_group=False):
    nblk = -(-w.Skv // 64)
    rng = np.random.default_rng(seed)
    m = rng.random((w.B, w.Hkv, nblk)) < density
    if empty_group:
        m[0, 0, :] = False
    return m


def _run_and_compare(w, lam, splits, sel, groups=None):
    q, k, v, _ = device_inputs(w)
    bm = torch.tensor(sel.astype(np.uint8), device=q.device)
    out = bs.decode(q, k, v, lam, num_splits=splits, return_lse=True, return_mask=True,
                    block_mask=bm)
    assert bs.check() == 0
    o = to_f64(out.o)
    assert np.all(np.isfinite(o))
    mask = out.skip_mask.cpu().numpy().astype(np.int8)
    mask = np.where(mask == 2, -1, mask).astype(np.int8)
    lse = out.lse.cpu().numpy()
    counts = out.skip_counts.cpu().numpy()
    G = w.Hq // w.Hkv
    groups = groups or [(b, h) for b in range(w.B) for h in range(w.Hkv)]
    for (b, h) in groups:
        qg = to_f64(q[b, h * G:(h + 1) * G])
        og, lg, mg, gg, _ = oracle.decode_group(qg, to_f64(k[b, h]), to_f64(v[b, h]), lam=lam,
                                                num_splits=out.num_splits, tile_k=64,
                                                block_mask=sel[b, h])
        assert np.array_equal(mask[b, h] == -1, ~sel[b, h]), f"unselected tiles b={b} h={h}"
        assert_close(o[b, h * G:(h + 1) * G], og, f"o[b={b},hkv={h}]")
        if np.all(np.isinf(lg)):
            assert np.all(lse[b, h * G:(h + 1) * G] == -np.inf)
            assert np.all(o[b, h * G:(h + 1) * G] == 0.0)
        else:
            assert np.all(np.abs(lse[b, h * G:(h + 1) * G] - lg) < 1e-2)
        assert_masks(mask[b, h], mg, gg, f"mask[b={b},hkv={h}]")
    per_group = (mask == 1).sum(axis=(0, 2))
    assert np.array_equal(counts, np.repeat(per_group, G))
    return out


CASES = [
    # (workload overrides, splits, density, empty group)
    (dict(B=2, Hq=16, Hkv=2, Skv=3000, D=128, window=256), 0, 0.5, False),
    (dict(B=2, Hq=16, Hkv=2, Skv=3000, D=128, window=256), 3, 0.3, True),
    (dict(B=2, Hq=16, Hkv=2, Skv=3000, D=128, window=256), 1, 0.8, False),
    (dict(B=1, Hq=8, Hkv=8, Skv=1000, D=64, window=128), 0, 0.5, True),
    (dict(B=3, Hq=8, Hkv=2, Skv=2500, D=128, window=128), 7, 0.1, False),
    (dict(B=1, Hq=8, Hkv=1, Skv=65, D=128, window=16), 2, 0.5, False),
]


@pytest.mark.parametrize("lam", [0.0, 1e-3, 1e-2])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_blockmask_decode_parity(case, lam):
    over, splits, density, empty = CASES[case]
    w = synth.WORKLOADS["decode_32k_gqa8"].with_(**over)
    _run_and_compare(w, lam, splits, _mask(w, density, case, empty))


def test_blockmask_all_selected_equals_no_mask():
    w = synth.WORKLOADS["decode_32k_gqa8"].with_(B=2, Hq=16, Hkv=2, Skv=5000, window=256)
    q, k, v, _ = device_inputs(w)
    ref = bs.decode(q, k, v, 1e-3, return_mask=True)
    ones = torch.ones((w.B, w.Hkv, -(-w.Skv // 64)), dtype=torch.uint8, device=q.device)
    out = bs.decode(q, k, v, 1e-3, return_mask=True, block_mask=ones)
    assert torch.equal(out.o, ref.o) and torch.equal(out.skip_mask, ref.skip_mask)
    assert torch.equal(out.skip_counts, ref.skip_counts)


def test_blockmask_decode_32k_sampled():
    w = synth.WORKLOADS["decode_32k_gqa8"]
    _run_and_compare(w, 1e-3, 0, _mask(w, 0.5, 7), groups=[(0, 0), (w.B - 1, w.Hkv - 1)])


def test_blockmask_rejects_bad_tensor():
    w = synth.WORKLOADS["decode_32k_gqa8"].with_(B=1, Hq=8, Hkv=1, Skv=1000, window=128)
    q, k, v, _ = device_inputs(w)
    with pytest.raises(TypeError):
        bs.decode(q, k, v, 0.0, block_mask=torch.ones((1, 1, 3), dtype=torch.uint8,
                                                      device=q.device))
