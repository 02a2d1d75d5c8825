"""Decode kernels (split-KV + combine) against the fp64 oracle, through the C ABI."""

import numpy as np
import pytest
import torch

import block_sparse_long_softmax_b300 as bs
import oracle
import synth
from gpu_helpers import assert_close, assert_masks, device_inputs, to_f64

pytestmark = pytest.mark.gpu

SMALL = [
    # (workload overrides, splits)
    (dict(B=2, Hq=16, Hkv=2, Skv=4096 + 37, D=128, window=256), 0),
    (dict(B=2, Hq=16, Hkv=2, Skv=4096 + 37, D=128, window=256), 5),
    (dict(B=1, Hq=8, Hkv=8, Skv=1000, D=64, window=128), 0),
    (dict(B=3, Hq=8, Hkv=2, Skv=2500, D=128, window=128), 1),
    (dict(B=1, Hq=4, Hkv=2, Skv=700, D=64, window=64), 3),
    (dict(B=1, Hq=8, Hkv=1, Skv=1, D=128, window=0, sink=1), 0),
    (dict(B=1, Hq=8, Hkv=1, Skv=65, D=128, window=16), 2),
]


def _run_and_compare(w, lam, splits, groups=None):
    q, k, v, _ = device_inputs(w)
    out = bs.decode(q, k, v, lam, num_splits=splits, return_lse=True, return_mask=True)
    assert bs.check() == 0
    o = to_f64(out.o)
    mask = out.skip_mask.cpu().numpy().astype(np.int8)
    counts = out.skip_counts.cpu().numpy()
    G = w.Hq // w.Hkv
    groups = groups or [(b, h) for b in range(w.B) for h in range(w.Hkv)]
    low = 0
    for (b, h) in groups:
        qg = to_f64(q[b, h * G:(h + 1) * G])
        og, lg, mg, gg, _ = oracle.decode_group(qg, to_f64(k[b, h]), to_f64(v[b, h]), lam=lam,
                                                num_splits=out.num_splits, tile_k=64)
        assert_close(o[b, h * G:(h + 1) * G], og, f"o[b={b},hkv={h}]")
        assert np.all(np.abs(out.lse.cpu().numpy()[b, h * G:(h + 1) * G] - lg) < 1e-2)
        low += assert_masks(mask[b, h], mg, gg, f"mask[b={b},hkv={h}]")
    # skip counts: group count (summed over batch) given to each query head
    per_group = (mask == 1).sum(axis=(0, 2))
    assert np.array_equal(counts, np.repeat(per_group, G))
    return out, low


@pytest.mark.parametrize("lam", [0.0, 1e-4, 1e-3, 1e-2])
@pytest.mark.parametrize("case", range(len(SMALL)))
def test_decode_parity_small(case, lam):
    over, splits = SMALL[case]
    w = synth.WORKLOADS["decode_32k_gqa8"].with_(**over)
    out, _ = _run_and_compare(w, lam, splits)
    if lam == 0.0:
        assert int(out.skip_counts.sum()) == 0


@pytest.mark.parametrize("name", ["decode_32k_gqa8", "decode_128k_gqa8"])
def test_decode_full_size_sampled(name):
    w = synth.WORKLOADS[name]
    for lam in w.lambdas:
        out, low = _run_and_compare(w, lam, 0, groups=[(0, 0), (w.B - 1, w.Hkv - 1), (w.B // 2, 3)])
        if lam >= 1e-3:
            assert out.skip_mask.float().mean().item() > 0.1  # planted structure is sparse


def test_decode_matches_dense_at_lambda_zero_any_splits():
    w = synth.WORKLOADS["decode_32k_gqa8"].with_(B=1, Hq=8, Hkv=1, Skv=5000, window=256)
    q, k, v, _ = device_inputs(w)
    ref = bs.decode(q, k, v, 0.0, num_splits=1).o.float()
    for s in (2, 7, 40):
        o = bs.decode(q, k, v, 0.0, num_splits=s).o.float()
        assert torch.allclose(o, ref, atol=1e-2, rtol=1e-2)


def test_decode_on_side_stream():
    w = synth.WORKLOADS["decode_32k_gqa8"].with_(B=2, Hq=16, Hkv=2, Skv=3000, window=256)
    q, k, v, _ = device_inputs(w)
    ref = bs.decode(q, k, v, 1e-3).o.clone()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out = bs.decode(q, k, v, 1e-3)
    s.synchronize()
    assert torch.equal(out.o, ref)


def test_decode_bounded_wait_reports_timeout():
    """A wait that nothing satisfies ends with a status code, not a hang or trap."""
    w = synth.WORKLOADS["decode_32k_gqa8"].with_(B=1, Hq=8, Hkv=1, Skv=1024, window=128)
    q, k, v, _ = device_inputs(w)
    bs.decode(q, k, v, 1e-3, num_splits=1, wait_limit_ms=20, inject_wait_timeout=True)
    assert bs.check() == 7
    assert bs.check() == 0  # cleared
    # the context is still usable and results are correct again
    _run_and_compare(w, 1e-3, 1)


@pytest.mark.parametrize("G", [1, 2, 4])
def test_decode_gqa_groups_full_length_sampled(G):
    # every supported group size at a 32K cache, sampled groups
    w = synth.WORKLOADS["decode_32k_gqa8"].with_(B=4, Hq=8 * G, Hkv=8)
    for lam in (0.0, 1e-3, 1e-2):
        _run_and_compare(w, lam, 0, groups=[(0, 0), (w.B - 1, w.Hkv - 1), (2, 5)])
