"""GPU parity of the online-softmax rescale of the prefill accumulator, and of a
caller-given softmax scale, against the fp64 oracle.

The update of a kept tile (the FlashAttention recurrence that Skip Softmax
builds on: "Approximating Softmax in Pretrained LLMs ...", Abstract; the running
maximum of "Accelerating Long-Context Inference with Skip Softmax in NVIDIA
TensorRT-LLM", "Skip Softmax Mechanism") multiplies the earlier output and row
sum by alpha = exp(m - m') whenever the running maximum m grows to m'.  The
prefill kernel defers that multiplication until the maximum has grown by more
than 2^8 in exp2 units (8 ln 2 nats) since the accumulator was last scaled.
Every case below first shows, from fp64 logits computed here, that some row's
maximum over its visited keys exceeds the maximum of its first visited tile by
more than 8 ln 2 + 0.5 nats — so the deferred rescale of O and l runs — and
then compares outputs, LSE and skip masks element by element with the oracle
at the tolerances of the other parity tests.

Two kinds of input make the maximum climb: planted structure with no sink keys
and a logit bump of 20 (the first tiles are noise, later window and random
blocks carry the bump), and the default planted structure with a softmax scale
of 4/sqrt(D) passed through the ABI.  Every prefill variant runs the rescale:
exact exponentials (128- and 64-row votes, D = 128 and 64), Rowmax-PoT, e4m3
Q/K and a caller block mask.  The decode, which rescales on every kept tile,
gets the softmax-scale case.
"""

import math

import numpy as np
import pytest
import torch

import block_sparse_long_softmax_b300 as bs
import oracle
import synth
from gpu_helpers import ATOL, RTOL, assert_close, assert_masks, device_inputs, to_f64

pytestmark = pytest.mark.gpu

CLIMB = 8.0 * math.log(2.0) + 0.5   # nats: comfortably past the kernel's deferral threshold
BASE = synth.WORKLOADS["prefill_32k_gqa8"]
NO_SINK = dict(sink=0, bump=20.0)


def _climbing_rows(qh, kh, *, scale, causal, tile_k, first_tile=None):
    """Rows whose maximum logit over visited keys exceeds the maximum over their first
    visited key tile by more than CLIMB nats.  first_tile[r] is that tile's index
    (default 0); sel[r, c] (optional, via first_tile) restricts the keys."""
    Sq, Skv = qh.shape[0], kh.shape[0]
    s = (qh @ kh.T) * scale
    if causal:
        qpos = np.arange(Sq) + (Skv - Sq)
        s = np.where(np.arange(Skv)[None, :] <= qpos[:, None], s, -np.inf)
    if first_tile is None:
        first = s[:, :tile_k].max(axis=1)
        top = s.max(axis=1)
    else:
        ft, keep = first_tile
        s = np.where(keep, s, -np.inf)
        cols = np.arange(Skv)[None, :] // tile_k
        first = np.where(cols == ft[:, None], s, -np.inf).max(axis=1)
        top = s.max(axis=1)
    with np.errstate(invalid="ignore"):
        return int(np.sum(np.isfinite(first) & (top - first > CLIMB)))


def _prefill_case(w, lam, *, tq, tk, mult=1.0, mode="exact", qs=1.0, ks=1.0, density=None):
    q, k, v, _ = device_inputs(w)
    scale_given = mult / math.sqrt(w.D) if mult != 1.0 else 0.0
    scale = mult / math.sqrt(w.D)
    kw = dict(causal=w.causal, tile_q=tq, tile_k=tk, return_lse=True, return_mask=True,
              return_visited=True, softmax_scale=scale_given)
    sel = None
    if mode == "pot":
        kw["exp_mode"] = "pot"
    if mode == "bm":
        nqt, nkt = -(-w.Sq // tq), -(-w.Skv // tk)
        rng = np.random.default_rng(11)
        sel = rng.random((w.B, w.Hq, nqt, nkt)) < density
        kw["block_mask"] = torch.tensor(sel.astype(np.uint8), device=q.device)
    if mode == "fp8":
        q8 = (q.float() / qs).to(torch.float8_e4m3fn)
        k8 = (k.float() / ks).to(torch.float8_e4m3fn)
        out = bs.prefill(q8, k8, v, lam, qk_descale=qs * ks, **kw)
    else:
        out = bs.prefill(q, k, v, lam, **kw)
    assert bs.check() == 0
    G = w.Hq // w.Hkv
    mask = out.skip_mask.cpu().numpy().astype(np.int8)
    mask = np.where(mask == 2, -1, mask).astype(np.int8)
    lse = out.lse.cpu().numpy()
    climbing = 0
    for b in range(w.B):
        for h in range(w.Hq):
            if mode == "fp8":
                qh = synth.e4m3_round(to_f64(q[b, h]) / qs)
                kh = synth.e4m3_round(to_f64(k[b, h // G]) / ks)
                sc = scale * qs * ks
            else:
                qh, kh, sc = to_f64(q[b, h]), to_f64(k[b, h // G]), scale
            vh = to_f64(v[b, h // G])
            vmax = float(np.max(np.abs(vh)))
            nqt = -(-w.Sq // tq)
            first = None
            if sel is not None:
                # each row's first selected key tile, and the keys its query tile visits
                rows_t = np.arange(w.Sq) // tq
                srow = sel[b, h][rows_t]                                  # [Sq][nkt]
                ft = np.where(srow.any(axis=1), srow.argmax(axis=1), -1)
                keep = np.repeat(srow, tk, axis=1)[:, :w.Skv]
                first = (ft, keep)
            climbing += _climbing_rows(qh, kh, scale=sc, causal=w.causal, tile_k=tk,
                                       first_tile=first)
            for t in range(nqt):
                r0, r1 = t * tq, min((t + 1) * tq, w.Sq)
                ot, lt, mt, gt, amb = oracle.prefill_qtile(
                    qh, kh, vh, t, tile_q=tq, tile_k=tk, causal=w.causal, lam=lam, scale=sc,
                    pot=mode == "pot",
                    block_mask_row=None if sel is None else sel[b, h, t])
                og = to_f64(out.o[b, h, r0:r1])
                what = f"{mode} o[b={b},h={h},t={t}]"
                if mode == "pot":
                    bound = ATOL + RTOL * np.abs(ot) + (2.0 ** -9 + amb[:, None]) * 2 * vmax
                    bad = np.abs(og - ot) > bound
                    assert not bad.any(), f"{what}: {bad.sum()} out of tolerance"
                    lb = 2e-2 + 2.0 ** -8 + 2 * amb
                else:
                    assert_close(og, ot, what)
                    lb = 2e-2
                fin = np.isfinite(lt)
                lb = np.broadcast_to(lb, lt.shape)
                assert np.all(lse[b, h, r0:r1][~fin] == -np.inf), f"lse -inf rows {what}"
                assert np.all(np.abs(lse[b, h, r0:r1][fin] - lt[fin]) < lb[fin]), f"lse {what}"
                assert_masks(mask[b, h, t], mt, gt, f"mask {what}")
    assert climbing > 0, "no row's running max climbs past the rescale threshold"
    return out


EXACT = [
    (dict(B=1, Hq=4, Hkv=2, Sq=700, Skv=700, D=128, window=128, **NO_SINK), 128, 128),
    (dict(B=1, Hq=4, Hkv=2, Sq=700, Skv=700, D=128, window=128, **NO_SINK), 64, 64),
    (dict(B=2, Hq=2, Hkv=1, Sq=520, Skv=520, D=64, window=64, **NO_SINK), 64, 64),
    (dict(B=2, Hq=2, Hkv=1, Sq=520, Skv=520, D=64, window=64, **NO_SINK), 128, 128),
    (dict(B=1, Hq=2, Hkv=1, Sq=300, Skv=777, D=128, window=128, causal=False, **NO_SINK),
     128, 128),
]


@pytest.mark.parametrize("lam", [0.0, 1e-3])
@pytest.mark.parametrize("case", range(len(EXACT)))
def test_rescale_exact_climbing_max(case, lam):
    over, tq, tk = EXACT[case]
    _prefill_case(BASE.with_(**over), lam, tq=tq, tk=tk)


@pytest.mark.parametrize("lam", [0.0, 1e-3, 1e-2])
@pytest.mark.parametrize("tq", [128, 64])
def test_rescale_exact_softmax_scale(tq, lam):
    w = BASE.with_(B=1, Hq=4, Hkv=2, Sq=700, Skv=700, D=128, window=128)
    _prefill_case(w, lam, tq=tq, tk=128, mult=4.0)


@pytest.mark.parametrize("lam", [0.0, 1e-3])
@pytest.mark.parametrize("over,tq,tk,mult", [
    (dict(B=1, Hq=4, Hkv=2, Sq=700, Skv=700, D=128, window=128, **NO_SINK), 128, 128, 1.0),
    (dict(B=2, Hq=2, Hkv=1, Sq=520, Skv=520, D=64, window=64, **NO_SINK), 64, 64, 1.0),
    (dict(B=1, Hq=4, Hkv=2, Sq=700, Skv=700, D=128, window=128), 128, 128, 4.0),
])
def test_rescale_rowmax_pot(over, tq, tk, mult, lam):
    _prefill_case(BASE.with_(**over), lam, tq=tq, tk=tk, mult=mult, mode="pot")


@pytest.mark.parametrize("lam", [0.0, 1e-3])
@pytest.mark.parametrize("over,tq,mult,qs,ks", [
    (dict(B=1, Hq=4, Hkv=2, Sq=700, Skv=700, D=128, window=128, **NO_SINK), 128, 1.0, 1.0, 1.0),
    (dict(B=1, Hq=4, Hkv=2, Sq=700, Skv=700, D=128, window=128, **NO_SINK), 64, 1.0, 2.0, 0.5),
    (dict(B=1, Hq=4, Hkv=2, Sq=700, Skv=700, D=128, window=128), 128, 4.0, 1.0, 1.0),
])
def test_rescale_fp8_qk(over, tq, mult, qs, ks, lam):
    _prefill_case(BASE.with_(**over), lam, tq=tq, tk=128, mult=mult, mode="fp8", qs=qs, ks=ks)


@pytest.mark.parametrize("lam", [0.0, 1e-3])
@pytest.mark.parametrize("over,tq,tk,mult", [
    (dict(B=1, Hq=4, Hkv=2, Sq=700, Skv=700, D=128, window=128, **NO_SINK), 128, 128, 1.0),
    (dict(B=1, Hq=4, Hkv=2, Sq=700, Skv=700, D=128, window=128, **NO_SINK), 64, 64, 1.0),
    (dict(B=1, Hq=4, Hkv=2, Sq=700, Skv=700, D=128, window=128), 128, 128, 4.0),
])
def test_rescale_block_mask(over, tq, tk, mult, lam):
    _prefill_case(BASE.with_(**over), lam, tq=tq, tk=tk, mult=mult, mode="bm", density=0.7)


@pytest.mark.parametrize("lam", [0.0, 1e-3, 1e-2])
@pytest.mark.parametrize("over,splits", [
    (dict(B=2, Hq=16, Hkv=2, Skv=4096 + 37, D=128, window=256), 0),
    (dict(B=1, Hq=8, Hkv=2, Skv=3000, D=64, window=128, **NO_SINK), 3),
])
def test_decode_softmax_scale(over, splits, lam):
    w = synth.WORKLOADS["decode_32k_gqa8"].with_(**over)
    q, k, v, _ = device_inputs(w)
    scale = 4.0 / math.sqrt(w.D)
    out = bs.decode(q, k, v, lam, num_splits=splits, softmax_scale=scale, return_lse=True,
                    return_mask=True)
    assert bs.check() == 0
    G = w.Hq // w.Hkv
    o = to_f64(out.o)
    mask = out.skip_mask.cpu().numpy().astype(np.int8)
    for b in range(w.B):
        for h in range(w.Hkv):
            og, lg, mg, gg, _ = oracle.decode_group(
                to_f64(q[b, h * G:(h + 1) * G]), to_f64(k[b, h]), to_f64(v[b, h]), lam=lam,
                num_splits=out.num_splits, tile_k=64, scale=scale)
            assert_close(o[b, h * G:(h + 1) * G], og, f"o[b={b},hkv={h}]")
            assert np.all(np.abs(out.lse.cpu().numpy()[b, h * G:(h + 1) * G] - lg) < 1e-2)
            assert_masks(mask[b, h], mg, gg, f"mask[b={b},hkv={h}]")
