"""Seeded sweep of small random shapes through every prefill and decode variant, each
compared element by element with the fp64 oracle.

Shapes, GQA groups, head dims, tiles, causality, thresholds, softmax scales, block
masks and (prefill) weight modes and operand formats are drawn from a fixed seed, so
the sweep is the same on every run.  Tolerances are those of the dedicated parity
tests: outputs within 1e-2 + 1e-2 |o| (Rowmax-PoT and e4m3 P.V widened by their
oracle-reported ambiguous shares), LSE within 2e-2 (decode 1e-2), masks equal on every
tile decided by more than 1e-3 nats, skip counts equal to the GPU's own mask.
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

N_PREFILL = 150
N_DECODE = 100


def _prefill_case(i):
    rng = np.random.default_rng(1000 + i)
    mode = ["exact", "exact", "pot", "fp8", "fp8pv", "bm"][i % 6]
    D = 128 if mode in ("fp8", "fp8pv") else int(rng.choice([64, 128]))
    tk = 128 if mode in ("fp8", "fp8pv") else int(rng.choice([64, 128]))
    tq = int(rng.choice([64, 128]))
    causal = bool(rng.random() < 0.7)
    Hkv = int(rng.choice([1, 2]))
    G = int(rng.choice([1, 2, 4]))
    Skv = int(rng.integers(1, 900))
    if mode == "fp8pv":
        Skv = max(16, Skv // 16 * 16)
    Sq = int(rng.integers(1, Skv + 1)) if causal else int(rng.integers(1, 700))
    lam = float(rng.choice([0.0, 1e-4, 1e-3, 1e-2, 0.1]))
    mult = float(rng.choice([1.0, 1.0, 2.0, 0.5]))
    over = dict(B=int(rng.choice([1, 2])), Hq=Hkv * G, Hkv=Hkv, Sq=Sq, Skv=Skv, D=D,
                window=int(rng.choice([32, 64, 128])), causal=causal, seed=int(i),
                sink=int(rng.choice([0, 16, 64])), bump=float(rng.choice([8.0, 12.0])))
    return mode, over, tq, tk, lam, mult


@pytest.mark.parametrize("i", range(N_PREFILL))
def test_random_prefill_parity(i):
    mode, over, tq, tk, lam, mult = _prefill_case(i)
    w = synth.WORKLOADS["prefill_32k_gqa8"].with_(**over)
    q, k, v, _ = device_inputs(w)
    scale = mult / math.sqrt(w.D)
    kw = dict(causal=w.causal, tile_q=tq, tile_k=tk, return_lse=True, return_mask=True,
              return_visited=True, softmax_scale=scale if mult != 1.0 else 0.0)
    sel = None
    if mode == "pot":
        kw["exp_mode"] = "pot"
    if mode == "bm":
        rng = np.random.default_rng(77 + i)
        nqt, nkt = -(-w.Sq // tq), -(-w.Skv // tk)
        sel = rng.random((w.B, w.Hq, nqt, nkt)) < 0.6
        kw["block_mask"] = torch.tensor(sel.astype(np.uint8), device=q.device)
    if mode in ("fp8", "fp8pv"):
        q8, k8 = q.float().to(torch.float8_e4m3fn), k.float().to(torch.float8_e4m3fn)
        assert np.array_equal(q8.double().cpu().numpy(), synth.e4m3_round(to_f64(q)))
        assert np.array_equal(k8.double().cpu().numpy(), synth.e4m3_round(to_f64(k)))
        if mode == "fp8pv":
            v8t = v.float().to(torch.float8_e4m3fn).transpose(2, 3).contiguous()
            out = bs.prefill(q8, k8, v8t, lam, **kw)
        else:
            out = bs.prefill(q8, k8, v, lam, **kw)
    else:
        out = bs.prefill(q, k, v, lam, **kw)
    assert bs.check() == 0
    G = w.Hq // w.Hkv
    mask = out.skip_mask.cpu().numpy().astype(np.int8)
    mask = np.where(mask == 2, -1, mask).astype(np.int8)
    lse = out.lse.cpu().numpy()
    for b in range(w.B):
        for h in range(w.Hq):
            if mode in ("fp8", "fp8pv"):
                qh = synth.e4m3_round(to_f64(q[b, h]))
                kh = synth.e4m3_round(to_f64(k[b, h // G]))
            else:
                qh, kh = to_f64(q[b, h]), to_f64(k[b, h // G])
            vh = synth.e4m3_round(to_f64(v[b, h // G])) if mode == "fp8pv" else to_f64(v[b, h // G])
            vmax = float(np.max(np.abs(vh)))
            for t in range(-(-w.Sq // tq)):
                r0, r1 = t * tq, min((t + 1) * tq, w.Sq)
                ot, lt, mt, gt, amb = oracle.prefill_qtile(
                    qh, kh, vh, t, tile_q=tq, tile_k=tk, causal=w.causal, lam=lam, scale=scale,
                    pot=mode == "pot", fp8_pv=mode == "fp8pv",
                    block_mask_row=None if sel is None else sel[b, h, t])
                og = to_f64(out.o[b, h, r0:r1])
                bound = ATOL + RTOL * np.abs(ot)
                lb = np.full(lt.shape, 2e-2)
                if mode == "pot":
                    bound = bound + (2.0 ** -9 + amb[:, None]) * 2 * vmax
                    lb = lb + 2.0 ** -8 + 2 * amb
                if mode == "fp8pv":
                    bound = bound + amb[:, None] * 0.25 * vmax
                bad = np.abs(og - ot) > bound
                what = f"case {i} ({mode}, {over}, tq={tq}, tk={tk}, lam={lam}) b={b} h={h} t={t}"
                assert not bad.any(), f"{what}: max err {np.abs(og - ot).max():.3e}"
                fin = np.isfinite(lt)
                assert np.all(lse[b, h, r0:r1][~fin] == -np.inf), what
                assert np.all(np.abs(lse[b, h, r0:r1][fin] - lt[fin]) < lb[fin]), what
                assert_masks(mask[b, h, t], mt, gt, what)
    assert np.array_equal(out.skip_counts.cpu().numpy(), (mask == 1).sum(axis=(0, 2, 3)))
    assert np.array_equal(out.visited_counts.cpu().numpy(), (mask >= 0).sum(axis=(0, 2, 3)))


def _decode_case(i):
    rng = np.random.default_rng(5000 + i)
    Hkv = int(rng.choice([1, 2, 3]))
    G = int(rng.choice([1, 2, 4, 8]))
    D = int(rng.choice([64, 128]))
    Skv = int(rng.integers(1, 6000))
    splits = int(rng.choice([0, 0, 1, 2, 5, 11]))
    lam = float(rng.choice([0.0, 1e-4, 1e-3, 1e-2, 0.1]))
    mult = float(rng.choice([1.0, 1.0, 3.0]))
    masked = bool(rng.random() < 0.3)
    over = dict(B=int(rng.choice([1, 3])), Hq=Hkv * G, Hkv=Hkv, Skv=Skv, D=D, seed=int(i),
                window=int(rng.choice([16, 128, 512])), sink=int(rng.choice([0, 1, 64])))
    return over, splits, lam, mult, masked


@pytest.mark.parametrize("i", range(N_DECODE))
def test_random_decode_parity(i):
    over, splits, lam, mult, masked = _decode_case(i)
    w = synth.WORKLOADS["decode_32k_gqa8"].with_(**over)
    q, k, v, _ = device_inputs(w)
    scale = mult / math.sqrt(w.D)
    nblk = -(-w.Skv // 64)
    sel = None
    kw = dict(num_splits=splits, return_lse=True, return_mask=True,
              softmax_scale=scale if mult != 1.0 else 0.0)
    if masked:
        sel = np.random.default_rng(99 + i).random((w.B, w.Hkv, nblk)) < 0.5
        kw["block_mask"] = torch.tensor(sel.astype(np.uint8), device=q.device)
    out = bs.decode(q, k, v, lam, **kw)
    assert bs.check() == 0
    G = w.Hq // w.Hkv
    o = to_f64(out.o)
    mask = out.skip_mask.cpu().numpy().astype(np.int8)
    mask = np.where(mask == 2, -1, mask).astype(np.int8)
    lse = out.lse.cpu().numpy()
    for b in range(w.B):
        for h in range(w.Hkv):
            og, lg, mg, gg, _ = oracle.decode_group(
                to_f64(q[b, h * G:(h + 1) * G]), to_f64(k[b, h]), to_f64(v[b, h]), lam=lam,
                num_splits=out.num_splits, tile_k=64, scale=scale,
                block_mask=None if sel is None else sel[b, h])
            what = f"case {i} ({over}, splits={splits}, lam={lam}, masked={masked}) b={b} hkv={h}"
            err = np.abs(o[b, h * G:(h + 1) * G] - og)
            assert np.all(err <= ATOL + RTOL * np.abs(og)), f"{what}: max err {err.max():.3e}"
            fin = np.isfinite(lg)
            lgpu = lse[b, h * G:(h + 1) * G]
            assert np.all(lgpu[~fin] == -np.inf), what
            assert np.all(np.abs(lgpu[fin] - lg[fin]) < 1e-2), what
            assert_masks(mask[b, h], mg, gg, what)
    per_group = (mask == 1).sum(axis=(0, 2))
    assert np.array_equal(out.skip_counts.cpu().numpy(), np.repeat(per_group, G))
