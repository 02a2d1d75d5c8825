"""Prefill kernel (tcgen05 / TMEM / TMA) against the fp64 oracle, through the C ABI."""

import numpy as np
import pytest
import torch

import block_sparse_long_softmax_b300 as bs
import oracle
import synth
from gpu_helpers import assert_close, assert_masks, device_inputs, to_f64

pytestmark = pytest.mark.gpu


def _compare_heads(w, q, k, v, out, lam, heads, qtiles=None):
    """Compare sampled (b, hq[, q tile]) of a prefill run with the oracle."""
    G = w.Hq // w.Hkv
    o = out.o
    mask = out.skip_mask.cpu().numpy().astype(np.int8)
    mask = np.where(mask == 2, -1, mask).astype(np.int8)
    lse = out.lse.cpu().numpy()
    low = 0
    for (b, h) in heads:
        qh, kh, vh = to_f64(q[b, h]), to_f64(k[b, h // G]), to_f64(v[b, h // G])
        nqt = -(-w.Sq // out.tile_q)
        for t in (range(nqt) if qtiles is None else qtiles):
            r0, r1 = t * out.tile_q, min((t + 1) * out.tile_q, w.Sq)
            ot, lt, mt, gt, _ = oracle.prefill_qtile(qh, kh, vh, t, tile_q=out.tile_q,
                                                     tile_k=out.tile_k, causal=w.causal, lam=lam,
                                                     scale=1.0 / np.sqrt(w.D))
            assert_close(to_f64(o[b, h, r0:r1]), ot, f"o[b={b},h={h},t={t}]")
            assert np.all(np.abs(lse[b, h, r0:r1] - lt) < 2e-2), f"lse[b={b},h={h},t={t}]"
            low += assert_masks(mask[b, h, t], mt, gt, f"mask[b={b},h={h},t={t}]")
    return low


def _run(w, lam, tile_q=0, tile_k=0):
    q, k, v, _ = device_inputs(w)
    out = bs.prefill(q, k, v, lam, causal=w.causal, tile_q=tile_q, tile_k=tile_k,
                     return_lse=True, return_mask=True, return_visited=True)
    assert bs.check() == 0
    return q, k, v, out


def _check_counts(out):
    mask = out.skip_mask.cpu().numpy()
    assert np.array_equal(out.skip_counts.cpu().numpy(), (mask == 1).sum(axis=(0, 2, 3)))
    assert np.array_equal(out.visited_counts.cpu().numpy(), (mask <= 1).sum(axis=(0, 2, 3)))


@pytest.mark.parametrize("lam", [0.0, 1e-4, 1e-2])
def test_prefill_1k_d64_full(lam):
    """The small configuration (B=1, H=1, S=1024, D=64, causal, 64x64 tiles), every output."""
    w = synth.WORKLOADS["prefill_1k_d64"]
    q, k, v, out = _run(w, lam, 64, 64)
    _compare_heads(w, q, k, v, out, lam, [(0, 0)])
    _check_counts(out)
    if lam == 0.0:
        assert int(out.skip_counts.sum()) == 0
    if lam == 1e-2:
        assert int(out.skip_counts.sum()) > 0


SMALL = [
    # overrides, tile_q, tile_k
    (dict(B=1, Hq=4, Hkv=2, Sq=700, Skv=700, D=128, window=128), 128, 128),
    (dict(B=1, Hq=4, Hkv=2, Sq=700, Skv=700, D=128, window=128), 64, 64),
    (dict(B=1, Hq=4, Hkv=2, Sq=700, Skv=700, D=128, window=128), 128, 64),
    (dict(B=1, Hq=4, Hkv=2, Sq=700, Skv=700, D=128, window=128), 64, 128),
    (dict(B=2, Hq=2, Hkv=1, Sq=520, Skv=520, D=64, window=64), 128, 128),
    (dict(B=1, Hq=2, Hkv=2, Sq=200, Skv=777, D=128, window=128), 128, 128),
    (dict(B=1, Hq=2, Hkv=1, Sq=300, Skv=520, D=128, window=128, causal=False), 128, 128),
    (dict(B=1, Hq=8, Hkv=1, Sq=129, Skv=129, D=64, window=32), 64, 64),
    (dict(B=1, Hq=1, Hkv=1, Sq=1, Skv=1, D=128, window=0, sink=1), 128, 128),
    (dict(B=1, Hq=1, Hkv=1, Sq=1, Skv=300, D=64, window=64), 64, 128),
    # non-causal with more queries than keys: every query tile sees the whole (ragged) cache
    (dict(B=1, Hq=2, Hkv=1, Sq=777, Skv=300, D=128, window=128, causal=False), 128, 128),
    (dict(B=1, Hq=2, Hkv=2, Sq=333, Skv=65, D=64, window=32, causal=False), 64, 64),
]


@pytest.mark.parametrize("lam", [0.0, 1e-3, 1e-2])
@pytest.mark.parametrize("case", range(len(SMALL)))
def test_prefill_parity_small(case, lam):
    over, tq, tk = SMALL[case]
    w = synth.WORKLOADS["prefill_32k_gqa8"].with_(**over)
    q, k, v, out = _run(w, lam, tq, tk)
    _compare_heads(w, q, k, v, out, lam, [(b, h) for b in range(w.B) for h in range(w.Hq)])
    _check_counts(out)


@pytest.mark.parametrize("name", ["prefill_32k_gqa8", "prefill_128k_gqa8"])
def test_prefill_full_size_sampled(name):
    w = synth.WORKLOADS[name]
    q, k, v, _ = device_inputs(w)
    nqt = w.Sq // 128
    for lam in (0.0, 1e-3, 1e-2):
        out = bs.prefill(q, k, v, lam, causal=True, return_lse=True, return_mask=True,
                         return_visited=True)
        assert bs.check() == 0
        _compare_heads(w, q, k, v, out, lam, [(0, 0), (0, w.Hq - 1)], qtiles=[0, 37, nqt - 1])
        _check_counts(out)
        vis = out.visited_counts.cpu().numpy()
        assert np.all(vis == nqt * (nqt + 1) // 2)  # causal: sum of visible tiles per head
        if lam > 0:
            del out
    torch.cuda.synchronize()


def test_prefill_on_side_stream_and_reuse_out():
    w = synth.WORKLOADS["prefill_32k_gqa8"].with_(Hq=4, Hkv=1, Sq=1000, Skv=1000, window=128)
    q, k, v, _ = device_inputs(w)
    ref = bs.prefill(q, k, v, 1e-3).o.clone()
    s = torch.cuda.Stream()
    o = torch.empty_like(q)
    with torch.cuda.stream(s):
        bs.prefill(q, k, v, 1e-3, out=o)
    s.synchronize()
    assert torch.equal(o, ref)


def test_prefill_bounded_wait_reports_timeout():
    """A wait that nothing satisfies ends with a status code, not a hang or trap."""
    w = synth.WORKLOADS["prefill_32k_gqa8"].with_(B=1, Hq=2, Hkv=1, Sq=300, Skv=300, window=64)
    q, k, v, _ = device_inputs(w)
    bs.prefill(q, k, v, 1e-3, wait_limit_ms=20, inject_wait_timeout=True)
    assert bs.check() == 25
    assert bs.check() == 0  # cleared
    # the context is still usable and results are correct again
    q, k, v, out = _run(w, 1e-3)
    _compare_heads(w, q, k, v, out, 1e-3, [(0, h) for h in range(w.Hq)])


MEDIUM = [
    # larger shapes than SMALL, sampled: D=64 with every tile configuration, batch > 1,
    # non-causal, and Sq < Skv at a few thousand keys
    (dict(B=2, Hq=8, Hkv=2, Sq=4096, Skv=4096, D=64, window=256), 64, 64),
    (dict(B=2, Hq=8, Hkv=2, Sq=4096, Skv=4096, D=64, window=256), 128, 128),
    (dict(B=2, Hq=8, Hkv=2, Sq=4096, Skv=4096, D=64, window=256), 64, 128),
    (dict(B=2, Hq=8, Hkv=2, Sq=4096, Skv=4096, D=64, window=256), 128, 64),
    (dict(B=3, Hq=16, Hkv=4, Sq=3000, Skv=5000, D=128, window=512), 128, 128),
    (dict(B=1, Hq=8, Hkv=1, Sq=4000, Skv=4000, D=128, window=512, causal=False), 128, 128),
]


@pytest.mark.parametrize("lam", [1e-3, 1e-2])
@pytest.mark.parametrize("case", range(len(MEDIUM)))
def test_prefill_parity_medium_sampled(case, lam):
    over, tq, tk = MEDIUM[case]
    w = synth.WORKLOADS["prefill_32k_gqa8"].with_(**over)
    q, k, v, out = _run(w, lam, tq, tk)
    nqt = -(-w.Sq // tq)
    heads = [(0, 0), (w.B - 1, w.Hq - 1), (w.B // 2, w.Hq // 2)]
    _compare_heads(w, q, k, v, out, lam, heads, qtiles=[0, nqt // 3, nqt - 1])
    _check_counts(out)
