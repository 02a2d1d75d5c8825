"""Error of the kernels' Skip Softmax output against dense attention, at full size.

"Accelerating Long-Context Inference with Skip Softmax in NVIDIA TensorRT-LLM", "Impact on
Accuracy vs. Speed", and "NVIDIA Introduces Skip Softmax ...", "Accuracy and Sparsity
Trade-offs": skipping gives up a little accuracy for speed.  How much is fixed by the rule:
a tile is skipped only when every row's exp(local max - running max) is below lambda, and the
running max is at most the row's final max, so each skipped key's dense probability is below
lambda.  The output of a row then moves, per dimension, by at most eps * (max v - min v),
where eps is the dense probability mass on the row's skipped keys.

Here the skipped tiles come from the kernel's own mask and the dense output and
probabilities from the oracle.  On sampled rows of the 128K prefill and decode workloads
each output element must satisfy that bound, widened by the kernel's rounding tolerance,
and eps must stay below lambda times the number of skipped keys (with a factor e^0.01 for
decisions the fp32 logits take within that margin).  The measured errors are printed.
"""

import math

import numpy as np
import pytest
import torch

import block_sparse_long_softmax_b300 as bs
import oracle
import synth
from gpu_helpers import ATOL, RTOL, device_inputs, to_f64

pytestmark = pytest.mark.gpu

DECISION_SLACK = math.exp(0.01)


def _check_rows(o_gpu, o_dense, p, skipped, vh, lam, what):
    eps = oracle.skipped_mass(p, skipped)
    vrange = vh.max(axis=0) - vh.min(axis=0)
    err = np.abs(o_gpu - o_dense)
    bound = eps[:, None] * vrange[None, :] + ATOL + RTOL * np.abs(o_dense)
    bad = err > bound
    assert not bad.any(), f"{what}: {bad.sum()} elements above the bound, max err {err.max():.3e}"
    nsk = skipped.sum(axis=1)
    assert np.all((eps < lam * nsk * DECISION_SLACK) | (nsk == 0)), f"{what}: eps above lambda*n"
    return float(err.max()), float(err.mean()), float(eps.max())


@pytest.mark.parametrize("lam", [3e-3, 1e-2])
def test_prefill_128k_error_against_dense_within_bound(lam):
    w = synth.WORKLOADS["prefill_128k_gqa8"]
    q, k, v, _ = device_inputs(w)
    out = bs.prefill(q, k, v, lam, causal=True, return_mask=True, return_visited=True)
    assert bs.check() == 0
    rho = out.skip_counts.sum().item() / out.visited_counts.sum().item()
    assert rho > 0.3
    G = w.Hq // w.Hkv
    tq, tk = out.tile_q, out.tile_k
    nqt = w.Sq // tq
    keys = np.arange(w.Skv)
    stats = []
    for (b, h) in [(0, 5), (0, w.Hq - 1)]:
        mask = out.skip_mask[b, h].cpu().numpy()
        kh, vh = to_f64(k[b, h // G]), to_f64(v[b, h // G])
        for t in (1, nqt // 2, nqt - 1):
            r0, r1 = t * tq, (t + 1) * tq
            qh = to_f64(q[b, h, r0:r1])
            visible = keys[None, :] <= np.arange(r0, r1)[:, None]   # Sq = Skv: causal
            o_dense, _, p = oracle.dense_attention(qh, kh, vh, causal=False, key_keep=visible)
            skipped = np.repeat(mask[t] == 1, tk)[None, : w.Skv] & visible
            o_gpu = to_f64(out.o[b, h, r0:r1])
            stats.append(_check_rows(o_gpu, o_dense, p, skipped, vh, lam,
                                     f"prefill b={b} h={h} t={t}"))
    mx = max(s[0] for s in stats)
    print(f"\nprefill 128K lambda={lam:g}: skip ratio {rho:.3f}, sampled rows: max |o - o_dense| "
          f"{mx:.3e}, mean {np.mean([s[1] for s in stats]):.3e}, max eps "
          f"{max(s[2] for s in stats):.3e}")


@pytest.mark.parametrize("lam", [2.2e-3, 1e-2])
def test_decode_128k_error_against_dense_within_bound(lam):
    w = synth.WORKLOADS["decode_128k_gqa8"]
    q, k, v, _ = device_inputs(w)
    out = bs.decode(q, k, v, lam, return_mask=True)
    assert bs.check() == 0
    mask_all = out.skip_mask.cpu().numpy()
    rho = float((mask_all == 1).mean())
    assert rho > 0.3
    G = w.Hq // w.Hkv
    stats = []
    for (b, h) in [(0, 0), (3, 5), (w.B - 1, w.Hkv - 1)]:
        qg = to_f64(q[b, h * G:(h + 1) * G])
        kh, vh = to_f64(k[b, h]), to_f64(v[b, h])
        o_dense, _, p = oracle.dense_attention(qg, kh, vh, causal=False)
        skipped = np.broadcast_to(np.repeat(mask_all[b, h] == 1, 64)[: w.Skv], p.shape)
        o_gpu = to_f64(out.o[b, h * G:(h + 1) * G])
        stats.append(_check_rows(o_gpu, o_dense, p, skipped, vh, lam, f"decode b={b} hkv={h}"))
    print(f"\ndecode 128K lambda={lam:g}, {out.num_splits} splits: skip ratio {rho:.3f}, sampled "
          f"groups: max |o - o_dense| {max(s[0] for s in stats):.3e}, mean "
          f"{np.mean([s[1] for s in stats]):.3e}, max eps {max(s[2] for s in stats):.3e}")
    del out
    torch.cuda.synchronize()
