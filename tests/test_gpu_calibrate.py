"""Threshold calibration to a target skip ratio, through the C ABI."""

import pytest
import torch

import block_sparse_long_softmax_b300 as bs
import synth
from gpu_helpers import device_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("target", [0.25, 0.5])
def test_prefill_calibration_hits_target(target):
    w = synth.WORKLOADS["prefill_32k_gqa8"].with_(Hq=16, Hkv=2, Sq=4096, Skv=4096, window=512)
    q, k, v, _ = device_inputs(w)
    lam, ratio, launches = bs.calibrate_prefill(q, k, v, target)
    assert launches == 14 and 0.0 < lam <= 1.0
    assert abs(ratio - target) < 0.03
    # the reported ratio is what a plain call at that lambda measures
    out = bs.prefill(q, k, v, lam, return_visited=True)
    again = out.skip_counts.sum().item() / out.visited_counts.sum().item()
    assert abs(again - ratio) < 1e-6
    assert bs.check() == 0


def test_decode_calibration_hits_target():
    w = synth.WORKLOADS["decode_32k_gqa8"].with_(B=4, Skv=8192, window=512)
    q, k, v, _ = device_inputs(w)
    lam, ratio, launches = bs.calibrate_decode(q, k, v, 0.5, max_iters=16)
    assert launches == 16 and abs(ratio - 0.5) < 0.03
    out = bs.decode(q, k, v, lam)
    nblk = w.B * w.Hkv * (w.Skv // 64)
    again = out.skip_counts[:: w.G].sum().item() / nblk
    assert abs(again - ratio) < 1e-6
    assert bs.check() == 0


def test_skip_ratio_is_monotone_in_lambda():
    w = synth.WORKLOADS["prefill_32k_gqa8"].with_(Hq=8, Hkv=1, Sq=2048, Skv=2048, window=256)
    q, k, v, _ = device_inputs(w)
    prev = -1
    for lam in (0.0, 1e-6, 1e-4, 1e-3, 3e-3, 1e-2, 3e-2, 0.1, 0.5, 1.0):
        s = bs.prefill(q, k, v, lam).skip_counts.sum().item()
        assert s >= prev
        prev = s
