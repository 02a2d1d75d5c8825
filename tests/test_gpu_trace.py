"""Per-tile timing of the prefill loop from the test-only instrumented build.

libskipsm_trace.so is the library built with -DSKIPSM_TRACE=1: in one chosen CTA,
one lane of the softmax warp of TMEM quadrant 0 and one lane of the MMA warp stamp
clock64 at fixed points of every (key tile, Q tile) step (events listed in the
kernel source).  This test builds it if needed, runs one prefill through it, checks
that the stamps are ordered the way the pipeline orders them and that the kept
flags agree with the skip mask, and prints where a kept and a skipped tile spend
their cycles: the softmax's wait for S, the reduced load, the vote, the
exponentials and P store, the arrive, and the chain from the arrive through the MMA
warp's issue of the next Q.K^T to the next S.
"""

import ctypes
import os

import numpy as np
import pytest
import torch

import block_sparse_long_softmax_b300 as bs
from block_sparse_long_softmax_b300 import build as libbuild
import synth
from gpu_helpers import device_inputs

pytestmark = pytest.mark.gpu

EV = 16


def trace_library():
    path = libbuild.build(trace=True)
    lib = ctypes.CDLL(path)
    lib.skipsm_debug_prefill_trace.argtypes = [ctypes.c_void_p, ctypes.c_int]
    lib.skipsm_prefill_ex.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int] * 7 + \
        [ctypes.c_float, ctypes.c_void_p, ctypes.POINTER(bs.PrefillOpts), ctypes.c_void_p]
    lib.skipsm_prefill_ex.restype = ctypes.c_int
    lib.skipsm_check.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int)]
    return lib


def traced_prefill(lib, q, k, v, lam, cta):
    """Run one causal prefill (default tiles) with CTA `cta` traced; returns
    (stamps [nkt][2][EV] int64, skip_mask of the CTA's two Q tiles [2][nkt])."""
    B, Hq, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    nkt = -(-Skv // 128)
    buf = torch.zeros(nkt * 2 * EV, dtype=torch.int64, device=q.device)
    o = torch.empty_like(q)
    mask = torch.empty((B, Hq, -(-Sq // 128), nkt), dtype=torch.uint8, device=q.device)
    opts = bs.PrefillOpts(128, 128, 0.0, None, mask.data_ptr(), None, 0, 0, 0, 0.0, None, 0, None, 0, 0.0)
    lib.skipsm_debug_prefill_trace(buf.data_ptr(), cta)
    s = torch.cuda.current_stream().cuda_stream
    rc = lib.skipsm_prefill_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, Hq,
                               Hkv, Sq, Skv, D, 1, float(lam), None, ctypes.byref(opts), s)
    assert rc == 0
    st = ctypes.c_int(0)
    assert lib.skipsm_check(s, ctypes.byref(st)) == 0 and st.value == 0
    lib.skipsm_debug_prefill_trace(None, -1)
    # the CTA's (batch, head, query block): CTAs of one kv head are adjacent, GQA siblings
    # fastest, the last query blocks first
    G = Hq // Hkv
    nblk_q = -(-Sq // 256)
    gi, rest = cta % G, cta // G
    qblk = nblk_q - 1 - rest % nblk_q
    rest //= nblk_q
    hkv, b = rest % Hkv, rest // Hkv
    cm = mask[b, hkv * G + gi, 2 * qblk:2 * qblk + 2].cpu().numpy()
    return buf.view(nkt, 2, EV).cpu().numpy(), cm


def summarize(st, cm):
    """Median cycles per step, separately for tiles the CTA kept and skipped."""
    rows = []
    nkt = st.shape[0]
    for j in range(nkt - 1):
        for x in range(2):
            e = st[j, x]
            nxt = st[j + 1, x]
            if e[1] == 0 or nxt[1] == 0 or e[11] == 0:
                continue
            rows.append(dict(kept=int(e[6]), s_wait=e[1] - e[0], load=e[2] - e[1],
                             vote=e[3] - e[2], exp_store=e[4] - e[3], arrive=e[5] - e[4],
                             softmax=e[5] - e[1], mma_wake=e[9] - e[5],
                             mma_issue=e[11] - e[9], next_s=nxt[1] - e[11],
                             chain=nxt[1] - e[1]))
    out = {}
    for kept in (1, 0):
        sel = [r for r in rows if r["kept"] == kept]
        if sel:
            out["kept" if kept else "skipped"] = dict(
                n=len(sel), **{k: float(np.median([r[k] for r in sel])) for k in sel[0]
                               if k != "kept"})
    return out


@pytest.mark.parametrize("lam", [0.0, 1e-2])
def test_trace_stamps_are_ordered_and_match_the_mask(lam):
    w = synth.WORKLOADS["prefill_32k_gqa8"].with_(Hq=16, Hkv=2, Sq=8192, Skv=8192, window=1024)
    q, k, v, _ = device_inputs(w)
    lib = trace_library()
    st, cm = traced_prefill(lib, q, k, v, lam, cta=0)   # the last query block: every key tile
    nvis = int((cm[0] != 2).sum())
    assert nvis == w.Skv // 128 - 1 and int((cm[1] != 2).sum()) == w.Skv // 128
    for j in range(nvis):
        for x in range(2):
            e = st[j, x]
            assert 0 < e[0] <= e[1] <= e[2] <= e[3] <= e[4] <= e[5], (j, x, e[:6])
            assert e[8] <= e[9] <= e[10], (j, x, e[8:11])
            assert e[6] == (1 if cm[x, j] == 0 else 0), (j, x)   # this Q tile kept it
    for j in range(nvis - 1):
        for x in range(2):
            assert st[j, x, 9] >= st[j, x, 5] - 2000  # P is seen after (about) its arrive
            assert st[j, x, 11] >= st[j, x, 10]
    print(f"lambda={lam}: per-step median cycles", summarize(st, cm))


def decode_trace_library():
    lib = trace_library()
    lib.skipsm_debug_decode_trace.argtypes = [ctypes.c_void_p]
    lib.skipsm_decode_ex.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int] * 5 + \
        [ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
         ctypes.POINTER(bs.DecodeOpts), ctypes.c_void_p]
    lib.skipsm_decode_ex.restype = ctypes.c_int
    lib.skipsm_decode_num_splits.argtypes = [ctypes.c_int] * 4
    lib.skipsm_decode_workspace_size.argtypes = [ctypes.c_int] * 6
    lib.skipsm_decode_workspace_size.restype = ctypes.c_size_t
    return lib


def traced_decode(lib, q, k, v, lam):
    """One decode step with every split CTA's start and end time recorded: returns
    (times [B][Hkv][splits][2] ns, kept tiles per CTA [B][Hkv][splits], splits)."""
    B, Hq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    ns = lib.skipsm_decode_num_splits(B, Hkv, Skv, 0)
    ws = torch.empty(lib.skipsm_decode_workspace_size(B, Hq, Hkv, Skv, D, 0), dtype=torch.uint8,
                     device=q.device)
    o = torch.empty_like(q)
    nblk = -(-Skv // 64)
    mask = torch.empty((B, Hkv, nblk), dtype=torch.uint8, device=q.device)
    buf = torch.zeros(B * Hkv * ns * 2, dtype=torch.int64, device=q.device)
    opts = bs.DecodeOpts(0, 0.0, None, mask.data_ptr(), 0, 0, None, None)
    lib.skipsm_debug_decode_trace(buf.data_ptr())
    s = torch.cuda.current_stream().cuda_stream
    rc = lib.skipsm_decode_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, Hq, Hkv,
                              Skv, D, float(lam), None, ws.data_ptr(), ws.numel(), ctypes.byref(opts),
                              s)
    assert rc == 0
    st = ctypes.c_int(0)
    assert lib.skipsm_check(s, ctypes.byref(st)) == 0 and st.value == 0
    lib.skipsm_debug_decode_trace(None)
    per = -(-nblk // ns)
    m = mask.cpu().numpy()
    kept = np.zeros((B, Hkv, ns), dtype=np.int64)
    for sp in range(ns):
        kept[:, :, sp] = (m[:, :, sp * per:(sp + 1) * per] == 0).sum(axis=2)
    return buf.view(B, Hkv, ns, 2).cpu().numpy(), kept, ns


def tail_stats(times, slots):
    """Makespan, and the share of it during which fewer than half of the CTA slots are busy."""
    t = times.reshape(-1, 2)
    t0, t1 = t[:, 0].min(), t[:, 1].max()
    ev = sorted([(a, 1) for a in t[:, 0]] + [(b, -1) for b in t[:, 1]])
    active, last, low = 0, t0, 0
    for when, d in ev:
        if active < slots // 2:
            low += when - last
        active += d
        last = when
    dur = t[:, 1] - t[:, 0]
    return {"makespan_us": (t1 - t0) / 1e3, "share_below_half_busy": low / (t1 - t0),
            "cta_us_median": float(np.median(dur)) / 1e3, "cta_us_max": float(dur.max()) / 1e3}


@pytest.mark.parametrize("rho", [0.0, 0.8])
def test_decode_trace_covers_every_cta(rho):
    w = synth.WORKLOADS["decode_128k_gqa8"]
    q, k, v, _ = device_inputs(w)
    lam = 0.0 if rho == 0.0 else bs.calibrate_decode(q, k, v, rho)[0]
    lib = decode_trace_library()
    times, kept, ns = traced_decode(lib, q, k, v, lam)
    t = times.reshape(-1, 2)
    assert np.all(t[:, 0] > 0) and np.all(t[:, 1] >= t[:, 0])
    stats = tail_stats(times, 2 * 148)
    dur = (t[:, 1] - t[:, 0]).astype(np.float64)
    corr = float(np.corrcoef(dur, kept.reshape(-1))[0, 1]) if rho > 0 else 0.0
    print(f"decode 128K rho={rho} lambda={lam:.3e} splits={ns}: {stats}, "
          f"corr(CTA time, kept V tiles)={corr:.2f}")
