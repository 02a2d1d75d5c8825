"""GPU parity of the FP8/BF16 mixed-precision prefill (e4m3 Q and K, bf16 V) against
the oracle ("Approximating Softmax in Pretrained LLMs: ...", AI Summary: FP8/BF16
mixed-precision tensor cores).

The e4m3 inputs are the bf16 planted-structure inputs rounded to E4M3 (ties to even):
on the GPU by torch's float8_e4m3fn cast, on the host by synth.e4m3_round; the test
first checks that both give the same values, and the oracle then takes the host
values exactly.  Q.K^T of e4m3 values is exact per product and accumulated in fp32,
like the bf16 path, so the bf16 tolerances and mask rule apply unchanged.
"""

import math

import numpy as np
import pytest
import torch

import block_sparse_long_softmax_b300 as bs
import oracle
import synth
from gpu_helpers import assert_close, assert_masks, device_inputs, to_f64

pytestmark = pytest.mark.gpu


def _fp8_inputs(w, q_scale=1.0, k_scale=1.0):
    q, k, v, _ = device_inputs(w)
    q8 = (q.float() / q_scale).to(torch.float8_e4m3fn)
    k8 = (k.float() / k_scale).to(torch.float8_e4m3fn)
    return q, k, v, q8, k8


def _host_e4m3(t_bf16, scale):
    return synth.e4m3_round(to_f64(t_bf16) / scale)


def _check(w, lam, q, k, v, q8, k8, out, q_scale, k_scale, heads, qtiles=None):
    G = w.Hq // w.Hkv
    mask = out.skip_mask.cpu().numpy().astype(np.int8)
    mask = np.where(mask == 2, -1, mask).astype(np.int8)
    lse = out.lse.cpu().numpy()
    scale = q_scale * k_scale / math.sqrt(w.D)
    for (b, h) in heads:
        qh = _host_e4m3(q[b, h], q_scale)
        kh = _host_e4m3(k[b, h // G], k_scale)
        # the device cast gave the same e4m3 values
        assert np.array_equal(q8[b, h].double().cpu().numpy(), qh)
        assert np.array_equal(k8[b, h // G].double().cpu().numpy(), kh)
        vh = to_f64(v[b, h // G])
        nqt = -(-w.Sq // out.tile_q)
        for t in (range(nqt) if qtiles is None else qtiles):
            r0, r1 = t * out.tile_q, min((t + 1) * out.tile_q, w.Sq)
            ot, lt, mt, gt, _ = oracle.prefill_qtile(qh, kh, vh, t, tile_q=out.tile_q,
                                                     tile_k=out.tile_k, causal=w.causal,
                                                     lam=lam, scale=scale)
            assert_close(to_f64(out.o[b, h, r0:r1]), ot, f"o[b={b},h={h},t={t}]")
            assert np.all(np.abs(lse[b, h, r0:r1] - lt) < 2e-2), f"lse[b={b},h={h},t={t}]"
            assert_masks(mask[b, h, t], mt, gt, f"mask[b={b},h={h},t={t}]")


CASES = [
    (dict(B=1, Hq=4, Hkv=2, Sq=700, Skv=700, D=128, window=128), 128, 1.0, 1.0),
    (dict(B=1, Hq=4, Hkv=2, Sq=700, Skv=700, D=128, window=128), 64, 0.5, 2.0),
    (dict(B=2, Hq=2, Hkv=1, Sq=300, Skv=777, D=128, window=128), 128, 1.0, 1.0),
    (dict(B=1, Hq=2, Hkv=1, Sq=300, Skv=520, D=128, window=128, causal=False), 128, 4.0, 1.0),
]


@pytest.mark.parametrize("lam", [0.0, 1e-3, 1e-2])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_fp8_prefill_parity_small(case, lam):
    over, tq, qs, ks = CASES[case]
    w = synth.WORKLOADS["prefill_32k_gqa8"].with_(**over)
    q, k, v, q8, k8 = _fp8_inputs(w, qs, ks)
    out = bs.prefill(q8, k8, v, lam, causal=w.causal, tile_q=tq, return_lse=True,
                     return_mask=True, qk_descale=qs * ks)
    assert bs.check() == 0
    assert out.o.dtype == torch.bfloat16
    _check(w, lam, q, k, v, q8, k8, out, qs, ks, [(b, h) for b in range(w.B) for h in range(w.Hq)])


def test_fp8_prefill_32k_sampled():
    w = synth.WORKLOADS["prefill_32k_gqa8"]
    q, k, v, q8, k8 = _fp8_inputs(w)
    out = bs.prefill(q8, k8, v, 1e-3, return_lse=True, return_mask=True)
    assert bs.check() == 0
    _check(w, 1e-3, q, k, v, q8, k8, out, 1.0, 1.0, [(0, 9)], qtiles=[0, 77, w.Sq // 128 - 1])


def test_fp8_rejects_mixed_dtypes():
    w = synth.WORKLOADS["prefill_32k_gqa8"].with_(B=1, Hq=2, Hkv=1, Sq=256, Skv=256)
    q, k, v, q8, k8 = _fp8_inputs(w)
    with pytest.raises(TypeError):
        bs.prefill(q8, k, v, 0.0)
