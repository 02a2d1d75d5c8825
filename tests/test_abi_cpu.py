"""The C-ABI library without a GPU: it loads, exports every declared symbol,
and rejects bad arguments on the host before touching CUDA."""

import ctypes
import os
import re
import subprocess

import pytest

import block_sparse_long_softmax_b300 as bs
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "skipsm.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(skipsm_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return bs.library()


def test_header_declares_the_boundary():
    fns = declared_functions()
    for f in ("skipsm_prefill", "skipsm_prefill_ex", "skipsm_decode", "skipsm_decode_ex",
              "skipsm_decode_workspace_size", "skipsm_decode_num_splits", "skipsm_check",
              "skipsm_last_error", "skipsm_version"):
        assert f in fns


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", bs.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (\w+)", out))
    for f in declared_functions():
        assert f in exported, f
        assert hasattr(lib, f)


def test_noalloc_scratch_fits_both_decode_workloads(lib):
    # the allocation-free decode keeps its split partials in a fixed 16 MiB array; with the
    # default split count both decode workloads (B=16 at 32K, B=8 at 128K; Hq=64, D=128) fit
    import synth
    for name in ("decode_32k_gqa8", "decode_128k_gqa8"):
        w = synth.WORKLOADS[name]
        need = lib.skipsm_decode_workspace_size(w.B, w.Hq, w.Hkv, w.Skv, w.D, 0)
        assert 0 < need <= 16 << 20, (name, need)


def test_version(lib):
    assert lib.skipsm_version() == 108


P = 0x10000  # a 16-byte aligned fake device address; validation never dereferences it


def _prefill(lib, q=P, k=P, v=P, o=P, B=1, Hq=2, Hkv=1, Sq=256, Skv=256, D=128, causal=1,
             lam=0.01, opts=None):
    return lib.skipsm_prefill_ex(q, k, v, o, B, Hq, Hkv, Sq, Skv, D, causal, lam, None,
                                 ctypes.byref(opts) if opts is not None else None, None)


def _decode(lib, q=P, k=P, v=P, o=P, B=1, Hq=8, Hkv=1, Skv=1024, D=128, lam=0.01, ws=P,
            wsb=1 << 30, opts=None):
    return lib.skipsm_decode_ex(q, k, v, o, B, Hq, Hkv, Skv, D, lam, None, ws, wsb,
                                ctypes.byref(opts) if opts is not None else None, None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=0), 1), (dict(o=0), 1), (dict(k=P + 8), 1), (dict(B=0), 1), (dict(Sq=0), 1),
    (dict(Hq=3, Hkv=2), 1), (dict(D=96), 2), (dict(D=256), 2), (dict(Sq=300, Skv=200), 1),
    (dict(lam=-0.1), 1), (dict(lam=1.5), 1), (dict(lam=float("nan")), 1),
    (dict(lam=float("inf")), 1),
])
def test_prefill_rejects(lib, kw, status):
    assert _prefill(lib, **kw) == status
    assert lib.skipsm_last_error()


@pytest.mark.parametrize("tq,tk", [(32, 128), (128, 256), (96, 64)])
def test_prefill_rejects_tiles(lib, tq, tk):
    assert _prefill(lib, opts=bs.PrefillOpts(tq, tk, 0.0, None, None, None, 0)) == 2


def test_prefill_rejects_bad_scale(lib):
    assert _prefill(lib, opts=bs.PrefillOpts(0, 0, -1.0, None, None, None, 0)) == 1


@pytest.mark.parametrize("mode", [-1, 2, 7])
def test_prefill_rejects_bad_exp_mode(lib, mode):
    assert _prefill(lib, opts=bs.PrefillOpts(0, 0, 0.0, None, None, None, 0, mode)) == 1
    assert "exp_mode" in lib.skipsm_last_error().decode()


@pytest.mark.parametrize("fmt,tk,D,descale,status", [
    (2, 0, 128, 0.0, 1), (-1, 0, 128, 0.0, 1), (1, 64, 128, 0.0, 2), (1, 0, 64, 0.0, 2),
    (0, 0, 128, -1.0, 1), (1, 0, 128, float("nan"), 1),
])
def test_prefill_rejects_bad_qk_format(lib, fmt, tk, D, descale, status):
    opts = bs.PrefillOpts(0, tk, 0.0, None, None, None, 0, 0, fmt, descale)
    assert _prefill(lib, D=D, opts=opts) == status


def test_binding_rejects_unknown_exp_mode():
    with pytest.raises(ValueError):
        bs._exp_mode("poly")
    assert bs._exp_mode("exact") == 0 and bs._exp_mode("pot") == 1


@pytest.mark.parametrize("kw,status", [
    (dict(q=0), 1), (dict(v=P + 2), 1), (dict(Hq=12, Hkv=1), 2), (dict(Hq=32, Hkv=2), 2),
    (dict(D=80), 2), (dict(lam=2.0), 1), (dict(Skv=0), 1), (dict(ws=0), 5), (dict(wsb=16), 5),
    (dict(ws=P + 16), 5),
])
def test_decode_rejects(lib, kw, status):
    assert _decode(lib, **kw) == status


def test_decode_rejects_negative_splits(lib):
    assert _decode(lib, opts=bs.DecodeOpts(-1, 0.0, None, None, 0, 0)) == 1


def test_valid_call_without_gpu_fails_cleanly(lib):
    # all arguments valid: the call reaches CUDA, which has no device here
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _prefill(lib) == 3
    assert _decode(lib) == 3


@pytest.mark.parametrize("B,Hkv,Skv,req", [
    (8, 8, 131072, 0), (16, 8, 32768, 0), (1, 1, 100, 0), (1, 1, 64, 0), (2, 4, 5000, 7),
    (1, 8, 131072, 64), (1, 1, 130, 16), (3, 2, 640, 4), (1, 1, 1, 0),
])
def test_split_geometry_matches_oracle(lib, B, Hkv, Skv, req):
    ns = bs.decode_num_splits(B, Hkv, Skv, req)
    assert ns >= 1
    ref_req = req if req else ns
    assert oracle.decode_split_geometry(Skv, 64, ref_req)[2] == ns
    if req == 0:
        # default: no more splits than tiles
        nblk = -(-Skv // 64)
        assert ns <= max(1, nblk)


@pytest.mark.parametrize("B,Hkv,Skv,want", [
    # 64 (b, kv head) items x 9 splits = 576 CTAs: two nearly full waves of 296
    (8, 8, 131072, 9),
    # 128 items x 9 = 1152 CTAs: four nearly full waves
    (16, 8, 32768, 9),
    # few items: as many splits as 16-tile splits allow, all in one wave
    (1, 1, 131072, 128),
    (1, 8, 32768, 32),
])
def test_default_splits_fill_whole_waves(lib, B, Hkv, Skv, want):
    ns = bs.decode_num_splits(B, Hkv, Skv, 0)
    assert ns == want
    nblk = -(-Skv // 64)
    assert -(-nblk // ns) >= 16


def test_workspace_size(lib):
    ns = bs.decode_num_splits(8, 8, 131072, 0)
    rows = 8 * 64 * ns
    al = lambda x: (x + 255) // 256 * 256  # noqa: E731
    assert bs.decode_workspace_size(8, 64, 8, 131072, 128, 0) == al(rows * 128 * 4) + al(rows * 4)
    assert bs.decode_workspace_size(8, 63, 8, 131072, 128, 0) == 0


def test_calibration_rejects_bad_arguments(lib):
    res = bs.Calibration()
    cal = lib.skipsm_prefill_calibrate
    # target outside [0, 1], bad iteration count, missing scratch or result: refused on the host
    assert cal(P, P, P, P, 1, 2, 1, 256, 256, 128, 1, 1.5, 0, P, None, ctypes.byref(res), None) == 1
    assert cal(P, P, P, P, 1, 2, 1, 256, 256, 128, 1, -0.1, 0, P, None, ctypes.byref(res), None) == 1
    assert cal(P, P, P, P, 1, 2, 1, 256, 256, 128, 1, 0.5, 65, P, None, ctypes.byref(res), None) == 1
    assert cal(P, P, P, P, 1, 2, 1, 256, 256, 128, 1, 0.5, 0, None, None, ctypes.byref(res), None) == 1
    assert cal(P, P, P, P, 1, 2, 1, 256, 256, 128, 1, 0.5, 0, P, None, None, None) == 1
    opts = bs.PrefillOpts(0, 0, 0.0, None, P, None, 0)  # a skip-mask output is not allowed
    assert cal(P, P, P, P, 1, 2, 1, 256, 256, 128, 1, 0.5, 0, P, ctypes.byref(opts),
               ctypes.byref(res), None) == 1
    dcal = lib.skipsm_decode_calibrate
    assert dcal(P, P, P, P, 1, 8, 1, 1024, 128, 2.0, 0, P, P, 1 << 20, None,
                ctypes.byref(res), None) == 1
    assert dcal(P, P, P, P, 1, 8, 3, 1024, 128, 0.5, 0, P, P, 1 << 20, None,
                ctypes.byref(res), None) == 1
