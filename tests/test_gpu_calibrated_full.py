"""Full-size parity at the thresholds the benchmark runs at.

The benchmark calibrates lambda on the 128K prefill for tile skip ratios of about
30%, 50% and 70%, and on the 128K decode for 50% ("NVIDIA Introduces Skip Softmax
...", "Accuracy and Sparsity Trade-offs"; "Accelerating Long-Context Inference with
Skip Softmax in NVIDIA TensorRT-LLM", "Impact on Accuracy vs. Speed").  Here the
same calibration runs, and at each calibrated lambda sampled query tiles (first,
middle, last) of two heads of the 128K prefill, and three GQA groups of the 128K
decode, are compared with the oracle element by element: outputs within
1e-2 + 1e-2 |o|, LSE within 2e-2 (decode 1e-2), masks equal on every tile decided by
more than 1e-3 nats.  The error of the same rows against the oracle's dense
attention (lambda = 0) is printed: the sparsity-versus-error curve of these inputs.
"""

import numpy as np
import pytest

import block_sparse_long_softmax_b300 as bs
import oracle
import synth
from gpu_helpers import assert_close, assert_masks, device_inputs, to_f64

pytestmark = pytest.mark.gpu


def test_prefill_128k_parity_at_calibrated_lambdas():
    w = synth.WORKLOADS["prefill_128k_gqa8"]
    q, k, v, _ = device_inputs(w)
    G = w.Hq // w.Hkv
    nqt = w.Sq // 128
    tiles = [0, nqt // 2, nqt - 1]
    heads = [(0, 5), (0, w.Hq - 2)]
    host = {h: (to_f64(q[0, h]), to_f64(k[0, h // G]), to_f64(v[0, h // G])) for _, h in heads}
    dense = {(h, t): oracle.prefill_qtile(*host[h], t, tile_q=128, tile_k=128, causal=True,
                                          lam=0.0, scale=1.0 / np.sqrt(w.D))[0]
             for _, h in heads for t in tiles}
    for target in (0.3, 0.5, 0.7):
        lam, rho, _ = bs.calibrate_prefill(q, k, v, target)
        assert abs(rho - target) < 0.05, (target, rho)
        out = bs.prefill(q, k, v, lam, return_lse=True, return_mask=True, return_visited=True)
        assert bs.check() == 0
        mask = out.skip_mask.cpu().numpy().astype(np.int8)
        mask = np.where(mask == 2, -1, mask)
        lse = out.lse.cpu().numpy()
        errs = []
        for b, h in heads:
            for t in tiles:
                r0, r1 = 128 * t, 128 * t + 128
                ot, lt, mt, gt, _ = oracle.prefill_qtile(*host[h], t, tile_q=128, tile_k=128,
                                                         causal=True, lam=lam,
                                                         scale=1.0 / np.sqrt(w.D))
                og = to_f64(out.o[b, h, r0:r1])
                what = f"rho={target} lam={lam:.3e} h={h} t={t}"
                assert_close(og, ot, "o " + what)
                assert np.all(np.abs(lse[b, h, r0:r1] - lt) < 2e-2), "lse " + what
                assert_masks(mask[b, h, t], mt, gt, "mask " + what)
                errs.append(np.abs(og - dense[(h, t)]))
        e = np.concatenate(errs)
        print(f"prefill 128K rho={rho:.3f} lambda={lam:.3e}: error vs dense oracle on sampled "
              f"rows max {e.max():.3e} mean {e.mean():.3e}")


def test_decode_128k_parity_at_calibrated_lambda():
    w = synth.WORKLOADS["decode_128k_gqa8"]
    q, k, v, _ = device_inputs(w)
    G = w.Hq // w.Hkv
    for target in (0.5, 0.8):
        lam, rho, _ = bs.calibrate_decode(q, k, v, target)
        assert abs(rho - target) < 0.05, (target, rho)
        out = bs.decode(q, k, v, lam, return_lse=True, return_mask=True)
        assert bs.check() == 0
        o = to_f64(out.o)
        mask = out.skip_mask.cpu().numpy().astype(np.int8)
        errs = []
        for b, h in [(0, 0), (w.B - 1, w.Hkv - 1), (w.B // 2, 3)]:
            qg, kh, vh = to_f64(q[b, h * G:(h + 1) * G]), to_f64(k[b, h]), to_f64(v[b, h])
            og, lg, mg, gg, _ = oracle.decode_group(qg, kh, vh, lam=lam,
                                                    num_splits=out.num_splits, tile_k=64)
            what = f"rho={target} lam={lam:.3e} b={b} hkv={h}"
            assert_close(o[b, h * G:(h + 1) * G], og, "o " + what)
            assert np.all(np.abs(out.lse.cpu().numpy()[b, h * G:(h + 1) * G] - lg) < 1e-2)
            assert_masks(mask[b, h], mg, gg, "mask " + what)
            dense = oracle.decode_group(qg, kh, vh, lam=0.0, num_splits=out.num_splits,
                                        tile_k=64)[0]
            errs.append(np.abs(o[b, h * G:(h + 1) * G] - dense))
        e = np.concatenate(errs)
        print(f"decode 128K rho={rho:.3f} lambda={lam:.3e}: error vs dense oracle max "
              f"{e.max():.3e} mean {e.mean():.3e}")
