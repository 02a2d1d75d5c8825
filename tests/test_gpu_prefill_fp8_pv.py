"""GPU parity of the all-e4m3 prefill (e4m3 Q, K and V; P quantised to e4m3 for P.V)
against the oracle's FP8 P.V reading ("Approximating Softmax in Pretrained LLMs: ...",
AI Summary: FP8/BF16 mixed-precision tensor cores).

Inputs are the bf16 planted-structure inputs divided by a quantisation scale and
rounded to E4M3 (ties to even): on the GPU by torch's float8_e4m3fn cast, on the host
by synth.e4m3_round; the test checks both agree and feeds the oracle the host values
(V multiplied back by its scale, which the kernel applies to the output).  V goes to
the kernel transposed, [B][Hkv][D][Skv].

The oracle quantises each kept weight as e4m3(2^8 p) 2^-8 with p = exp(s - m') in fp64;
the kernel does the same in fp32, so a weight whose 2^8 p lies within a relative 2e-4 of
an e4m3 rounding midpoint may round to the neighbouring e4m3 value (one step, at most
2^-3 of the weight).  The oracle reports, per row, the share of the row sum carried by
such weights, and the tolerance per output element is
    1e-2 + 1e-2 |o| + ambiguous share * 2^-2 * max|v|.
LSE (the row sums keep the unquantised weights) and skip masks follow the rules of the
other parity tests.
"""

import math

import numpy as np
import pytest
import torch

import block_sparse_long_softmax_b300 as bs
import oracle
import synth
from gpu_helpers import ATOL, RTOL, assert_masks, device_inputs, to_f64

pytestmark = pytest.mark.gpu


def _inputs(w, qs=1.0, ks=1.0, vs=1.0):
    q, k, v, _ = device_inputs(w)
    q8 = (q.float() / qs).to(torch.float8_e4m3fn)
    k8 = (k.float() / ks).to(torch.float8_e4m3fn)
    v8 = (v.float() / vs).to(torch.float8_e4m3fn)
    v8t = v8.transpose(2, 3).contiguous()
    return q, k, v, q8, k8, v8, v8t


def _host(t_bf16, scale):
    return synth.e4m3_round(to_f64(t_bf16) / scale)


def _run_and_check(w, lam, tq, qs=1.0, ks=1.0, vs=1.0, heads=None, qtiles=None, sel=None):
    q, k, v, q8, k8, v8, v8t = _inputs(w, qs, ks, vs)
    kw = {}
    if sel is not None:
        kw["block_mask"] = torch.tensor(sel.astype(np.uint8), device=q.device)
    out = bs.prefill(q8, k8, v8t, lam, causal=w.causal, tile_q=tq, return_lse=True,
                     return_mask=True, return_visited=True, qk_descale=qs * ks, v_descale=vs,
                     **kw)
    assert bs.check() == 0
    assert out.o.dtype == torch.bfloat16
    G = w.Hq // w.Hkv
    mask = out.skip_mask.cpu().numpy().astype(np.int8)
    mask = np.where(mask == 2, -1, mask).astype(np.int8)
    lse = out.lse.cpu().numpy()
    scale = qs * ks / math.sqrt(w.D)
    heads = heads or [(b, h) for b in range(w.B) for h in range(w.Hq)]
    for (b, h) in heads:
        qh, kh = _host(q[b, h], qs), _host(k[b, h // G], ks)
        vh8 = _host(v[b, h // G], vs)
        assert np.array_equal(q8[b, h].double().cpu().numpy(), qh)
        assert np.array_equal(k8[b, h // G].double().cpu().numpy(), kh)
        assert np.array_equal(v8[b, h // G].double().cpu().numpy(), vh8)
        vh = vh8 * vs
        vmax = float(np.max(np.abs(vh)))
        nqt = -(-w.Sq // tq)
        for t in (range(nqt) if qtiles is None else qtiles):
            r0, r1 = t * tq, min((t + 1) * tq, w.Sq)
            ot, lt, mt, gt, amb = oracle.prefill_qtile(
                qh, kh, vh, t, tile_q=tq, tile_k=128, causal=w.causal, lam=lam, scale=scale,
                fp8_pv=True, block_mask_row=None if sel is None else sel[b, h, t])
            og = to_f64(out.o[b, h, r0:r1])
            bound = ATOL + RTOL * np.abs(ot) + amb[:, None] * 0.25 * vmax
            bad = np.abs(og - ot) > bound
            assert not bad.any(), (f"o[b={b},h={h},t={t}]: {bad.sum()} elements out of "
                                   f"tolerance, max err {np.abs(og - ot).max():.3e}")
            fin = np.isfinite(lt)
            assert np.all(lse[b, h, r0:r1][~fin] == -np.inf)
            assert np.all(np.abs(lse[b, h, r0:r1][fin] - lt[fin]) < 2e-2), f"lse[b={b},h={h},t={t}]"
            assert_masks(mask[b, h, t], mt, gt, f"mask[b={b},h={h},t={t}]")
    return out


CASES = [
    (dict(B=1, Hq=4, Hkv=2, Sq=704, Skv=704, D=128, window=128), 128, 1.0, 1.0, 1.0),
    (dict(B=1, Hq=4, Hkv=2, Sq=704, Skv=704, D=128, window=128), 64, 0.5, 2.0, 0.25),
    (dict(B=2, Hq=2, Hkv=1, Sq=200, Skv=784, D=128, window=128), 128, 1.0, 1.0, 2.0),
    (dict(B=1, Hq=2, Hkv=1, Sq=300, Skv=528, D=128, window=128, causal=False), 128, 4.0, 1.0,
     1.0),
    (dict(B=1, Hq=4, Hkv=2, Sq=704, Skv=704, D=128, window=128, sink=0, bump=20.0), 128, 1.0,
     1.0, 1.0),
]


@pytest.mark.parametrize("lam", [0.0, 1e-3, 1e-2])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_fp8_pv_prefill_parity_small(case, lam):
    over, tq, qs, ks, vs = CASES[case]
    _run_and_check(synth.WORKLOADS["prefill_32k_gqa8"].with_(**over), lam, tq, qs, ks, vs)


@pytest.mark.parametrize("lam", [0.0, 1e-3])
def test_fp8_pv_prefill_block_mask(lam):
    w = synth.WORKLOADS["prefill_32k_gqa8"].with_(B=1, Hq=4, Hkv=2, Sq=704, Skv=704, window=128)
    rng = np.random.default_rng(5)
    nqt = -(-w.Sq // 128)
    sel = rng.random((w.B, w.Hq, nqt, nqt)) < 0.6
    _run_and_check(w, lam, 128, sel=sel)


def test_fp8_pv_prefill_32k_sampled():
    w = synth.WORKLOADS["prefill_32k_gqa8"]
    nqt = w.Sq // 128
    out = _run_and_check(w, 1e-3, 128, heads=[(0, 9)], qtiles=[0, 77, nqt - 1])
    # the skip decisions only see Q.K^T: the same tiles as the bf16-V e4m3 path
    q, k, v, q8, k8, _, _ = _inputs(w)
    ref = bs.prefill(q8, k8, v, 1e-3, return_mask=True)
    assert torch.equal(out.skip_mask, ref.skip_mask)


def test_fp8_pv_rejects_bad_layouts():
    w = synth.WORKLOADS["prefill_32k_gqa8"].with_(B=1, Hq=2, Hkv=1, Sq=256, Skv=256)
    q, k, v, q8, k8, v8, v8t = _inputs(w)
    with pytest.raises(TypeError):
        bs.prefill(q8, k8, v8, 0.0)      # not transposed (D != Skv here only by shape)
    w2 = w.with_(Sq=250, Skv=250)        # Skv not a multiple of 16: the row stride of v^T
    q, k, v, q8, k8, v8, v8t = _inputs(w2)
    with pytest.raises(bs.SkipsmError):
        bs.prefill(q8, k8, v8t, 0.0)
