"""Python binding of libskipsm (Skip Softmax attention for B300, sm_103a).

Argument marshalling only: torch supplies device memory and the current
stream, every step of the attention runs in the library's CUDA kernels.  If
``libskipsm.so`` is missing or fails to load, every entry point raises — there
is no fallback.

    from block_sparse_long_softmax_b300 import prefill, decode
    out = prefill(q, k, v, lam=1e-3, causal=True)      # out.o, out.skip_counts
    out = decode(q1, k_cache, v_cache, lam=1e-3)
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

__all__ = ["prefill", "decode", "check", "decode_num_splits", "decode_workspace_size",
           "calibrate_prefill", "calibrate_decode", "library", "SkipsmError", "PrefillOut",
           "DecodeOut", "Calibration", "LIB_PATH"]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libskipsm.so")

STATUS = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "CUDA", 4: "TIMEOUT", 5: "WORKSPACE"}


class SkipsmError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"libskipsm {STATUS.get(status, status)}: {msg}")
        self.status = status


class PrefillOpts(ctypes.Structure):
    _fields_ = [("tile_q", ctypes.c_int), ("tile_k", ctypes.c_int),
                ("softmax_scale", ctypes.c_float), ("lse", ctypes.c_void_p),
                ("skip_mask", ctypes.c_void_p), ("visited_counts", ctypes.c_void_p),
                ("wait_limit_ms", ctypes.c_int), ("exp_mode", ctypes.c_int),
                ("qk_format", ctypes.c_int), ("qk_descale", ctypes.c_float),
                ("block_mask", ctypes.c_void_p), ("inject_wait_timeout", ctypes.c_int),
                ("status", ctypes.c_void_p), ("v_format", ctypes.c_int),
                ("v_descale", ctypes.c_float), ("v_load", ctypes.c_int),
                ("sync_check", ctypes.c_int)]


EXP_MODES = {"exact": 0, "pot": 1}


V_LOADS = {"default": 0, "ahead": 1, "after_vote": 2}


def _v_load(v_load) -> int:
    if v_load not in V_LOADS:
        raise ValueError(f"v_load must be one of {sorted(V_LOADS)}")
    return V_LOADS[v_load]


def _exp_mode(exp_mode) -> int:
    if exp_mode not in EXP_MODES:
        raise ValueError(f"exp_mode must be one of {sorted(EXP_MODES)}")
    return EXP_MODES[exp_mode]


class DecodeOpts(ctypes.Structure):
    _fields_ = [("num_splits", ctypes.c_int), ("softmax_scale", ctypes.c_float),
                ("lse", ctypes.c_void_p), ("skip_mask", ctypes.c_void_p),
                ("wait_limit_ms", ctypes.c_int), ("inject_wait_timeout", ctypes.c_int),
                ("block_mask", ctypes.c_void_p), ("status", ctypes.c_void_p),
                ("sync_check", ctypes.c_int)]


class Calibration(ctypes.Structure):
    _fields_ = [("lambda_", ctypes.c_float), ("skip_ratio", ctypes.c_float),
                ("launches", ctypes.c_int)]


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int


def library() -> ctypes.CDLL:
    """The loaded libskipsm (raises if the shared library is missing)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: run `python -m "
                              "block_sparse_long_softmax_b300.build` (needs nvcc)")
        lib = ctypes.CDLL(LIB_PATH)
        lib.skipsm_version.restype = _I
        lib.skipsm_last_error.restype = ctypes.c_char_p
        lib.skipsm_check.argtypes = [_P, ctypes.POINTER(_I)]
        lib.skipsm_check.restype = _I
        lib.skipsm_prefill.argtypes = [_P, _P, _P, _P] + [_I] * 7 + [ctypes.c_float, _P, _P]
        lib.skipsm_prefill.restype = _I
        lib.skipsm_prefill_ex.argtypes = [_P, _P, _P, _P] + [_I] * 7 + \
            [ctypes.c_float, _P, ctypes.POINTER(PrefillOpts), _P]
        lib.skipsm_prefill_ex.restype = _I
        lib.skipsm_decode_num_splits.argtypes = [_I] * 4
        lib.skipsm_decode_num_splits.restype = _I
        lib.skipsm_decode_workspace_size.argtypes = [_I] * 6
        lib.skipsm_decode_workspace_size.restype = ctypes.c_size_t
        lib.skipsm_decode.argtypes = [_P, _P, _P, _P] + [_I] * 5 + \
            [ctypes.c_float, _P, _P, ctypes.c_size_t, _P]
        lib.skipsm_decode.restype = _I
        lib.skipsm_decode_ex.argtypes = [_P, _P, _P, _P] + [_I] * 5 + \
            [ctypes.c_float, _P, _P, ctypes.c_size_t, ctypes.POINTER(DecodeOpts), _P]
        lib.skipsm_decode_ex.restype = _I
        lib.skipsm_prefill_calibrate.argtypes = [_P, _P, _P, _P] + [_I] * 7 + \
            [ctypes.c_float, _I, _P, ctypes.POINTER(PrefillOpts), ctypes.POINTER(Calibration), _P]
        lib.skipsm_prefill_calibrate.restype = _I
        lib.skipsm_decode_calibrate.argtypes = [_P, _P, _P, _P] + [_I] * 5 + \
            [ctypes.c_float, _I, _P, _P, ctypes.c_size_t, ctypes.POINTER(DecodeOpts),
             ctypes.POINTER(Calibration), _P]
        lib.skipsm_decode_calibrate.restype = _I
        _lib = lib
    return _lib


def _raise(st: int):
    if st != 0:
        raise SkipsmError(st, library().skipsm_last_error().decode())


def _stream(stream) -> int:
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check_tensor(name, t, ndim, fp8=False):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    want = torch.float8_e4m3fn if fp8 else torch.bfloat16
    if t.dtype != want or t.dim() != ndim or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous {want} tensor with {ndim} dims")


def _status_ptr(status):
    """Device address of a caller's per-call status word (None = the shared word)."""
    import torch
    if status is None:
        return None
    if (not isinstance(status, torch.Tensor) or not status.is_cuda or status.dtype != torch.int32
            or status.numel() != 1):
        raise TypeError("status must be a one-element int32 CUDA tensor")
    return status.data_ptr()


def check(stream=None) -> int:
    """Synchronise `stream`, read and clear the device status word (0 = clean)."""
    st = ctypes.c_int(0)
    rc = library().skipsm_check(_P(_stream(stream)), ctypes.byref(st))
    if rc not in (0, 4):
        _raise(rc)
    return st.value


@dataclass
class PrefillOut:
    o: "torch.Tensor"
    skip_counts: "torch.Tensor"
    lse: Optional["torch.Tensor"] = None
    skip_mask: Optional["torch.Tensor"] = None
    visited_counts: Optional["torch.Tensor"] = None
    tile_q: int = 0
    tile_k: int = 0


def prefill(q, k, v, lam: float, causal: bool = True, *, tile_q: int = 0, tile_k: int = 0,
            softmax_scale: float = 0.0, return_lse: bool = False, return_mask: bool = False,
            return_visited: bool = False, out=None, skip_counts=None, stream=None,
            wait_limit_ms: int = 0, exp_mode: str = "exact",
            qk_descale: float = 0.0, block_mask=None,
            inject_wait_timeout: bool = False, status=None,
            v_descale: float = 0.0, v_load: str = "default",
            sync_check: bool = False) -> PrefillOut:
    """Skip Softmax prefill: q [B][Hq][Sq][D], k/v [B][Hkv][Skv][D] CUDA tensors.

    q and k are bf16, or both float8_e4m3fn (the FP8/BF16 mixed-precision path, D = 128:
    Q.K^T in e4m3, scaled by qk_descale); v is bf16 [B][Hkv][Skv][D], or, with e4m3 q and
    k, float8_e4m3fn transposed to [B][Hkv][D][Skv] (P.V in e4m3 as well; the output is
    multiplied by v_descale).  v_load: "default", "ahead" (every V tile before the vote) or
    "after_vote" (only the V tiles of kept key tiles).  exp_mode "exact" uses exponentials on
    kept tiles, "pot" Rowmax-PoT powers of two.  block_mask: optional uint8/bool CUDA
    tensor [B][Hq][ceil(Sq/tile_q)][ceil(Skv/tile_k)] of the pairs to visit.
    status: optional int32 CUDA tensor of one element that receives this call's
    device status (a timed-out wait's site) instead of the library's shared word.
    sync_check: wait for the stream and raise if one of this call's kernel waits timed out.
    """
    import torch
    lib = library()
    fp8 = q.dtype == torch.float8_e4m3fn
    v8 = fp8 and v.dtype == torch.float8_e4m3fn
    _check_tensor("q", q, 4, fp8), _check_tensor("k", k, 4, fp8), _check_tensor("v", v, 4, v8)
    B, Hq, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    if v8 and tuple(v.shape) != (B, Hkv, D, Skv):
        raise TypeError(f"e4m3 v must be transposed: shape {(B, Hkv, D, Skv)}")
    tq = tile_q or (64 if D == 64 else 128)
    tk = tile_k or (64 if D == 64 else 128)
    o = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device) if out is None else out
    cnt = torch.empty(Hq, dtype=torch.int64, device=q.device) if skip_counts is None else skip_counts
    lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device) if return_lse else None
    nqt, nkt = -(-Sq // tq), -(-Skv // tk)
    mask = torch.empty((B, Hq, nqt, nkt), dtype=torch.uint8, device=q.device) if return_mask else None
    vis = torch.empty(Hq, dtype=torch.int64, device=q.device) if return_visited else None
    ptr = lambda t: _P(t.data_ptr()) if t is not None else _P(0)  # noqa: E731
    if block_mask is not None and (
            not isinstance(block_mask, torch.Tensor) or not block_mask.is_cuda
            or block_mask.dtype not in (torch.uint8, torch.bool)
            or tuple(block_mask.shape) != (B, Hq, nqt, nkt) or not block_mask.is_contiguous()):
        raise TypeError(f"block_mask must be a contiguous uint8/bool CUDA tensor "
                        f"of shape {(B, Hq, nqt, nkt)}")
    opts = PrefillOpts(tq, tk, float(softmax_scale), ptr(lse).value, ptr(mask).value,
                       ptr(vis).value, int(wait_limit_ms), _exp_mode(exp_mode), 1 if fp8 else 0,
                       float(qk_descale), ptr(block_mask).value,
                       1 if inject_wait_timeout else 0, _status_ptr(status), 1 if v8 else 0,
                       float(v_descale), _v_load(v_load), 1 if sync_check else 0)
    _raise(lib.skipsm_prefill_ex(ptr(q), ptr(k), ptr(v), ptr(o), B, Hq, Hkv, Sq, Skv, D,
                                 1 if causal else 0, float(lam), ptr(cnt), ctypes.byref(opts),
                                 _P(_stream(stream))))
    return PrefillOut(o, cnt, lse, mask, vis, tq, tk)


def decode_num_splits(B: int, Hkv: int, Skv: int, requested: int = 0) -> int:
    return library().skipsm_decode_num_splits(B, Hkv, Skv, requested)


def decode_workspace_size(B, Hq, Hkv, Skv, D, num_splits=0) -> int:
    return library().skipsm_decode_workspace_size(B, Hq, Hkv, Skv, D, num_splits)


@dataclass
class DecodeOut:
    o: "torch.Tensor"
    skip_counts: "torch.Tensor"
    num_splits: int
    lse: Optional["torch.Tensor"] = None
    skip_mask: Optional["torch.Tensor"] = None


def decode(q, k, v, lam: float, *, num_splits: int = 0, softmax_scale: float = 0.0,
           return_lse: bool = False, return_mask: bool = False, workspace=None, out=None,
           skip_counts=None, stream=None, wait_limit_ms: int = 0,
           inject_wait_timeout: bool = False, block_mask=None, status=None,
           sync_check: bool = False) -> DecodeOut:
    """Skip Softmax decode: q [B][Hq][D], k/v [B][Hkv][Skv][D] bf16 CUDA tensors.

    block_mask: optional uint8/bool CUDA tensor [B][Hkv][ceil(Skv/64)] of the key tiles
    to visit (nonzero = visit).  status, sync_check: as for prefill.
    """
    import torch
    lib = library()
    _check_tensor("q", q, 3), _check_tensor("k", k, 4), _check_tensor("v", v, 4)
    B, Hq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    ns = lib.skipsm_decode_num_splits(B, Hkv, Skv, num_splits)
    wsb = lib.skipsm_decode_workspace_size(B, Hq, Hkv, Skv, D, num_splits)
    ws = torch.empty(wsb, dtype=torch.uint8, device=q.device) if workspace is None else workspace
    o = torch.empty_like(q) if out is None else out
    cnt = torch.empty(Hq, dtype=torch.int64, device=q.device) if skip_counts is None else skip_counts
    lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device) if return_lse else None
    nblk = -(-Skv // 64)
    mask = torch.empty((B, Hkv, nblk), dtype=torch.uint8, device=q.device) if return_mask else None
    ptr = lambda t: _P(t.data_ptr()) if t is not None else _P(0)  # noqa: E731
    if block_mask is not None:
        if (not isinstance(block_mask, torch.Tensor) or not block_mask.is_cuda
                or block_mask.dtype not in (torch.uint8, torch.bool)
                or tuple(block_mask.shape) != (B, Hkv, nblk) or not block_mask.is_contiguous()):
            raise TypeError(f"block_mask must be a contiguous uint8/bool CUDA tensor "
                            f"of shape {(B, Hkv, nblk)}")
    opts = DecodeOpts(int(num_splits), float(softmax_scale), ptr(lse).value, ptr(mask).value,
                      int(wait_limit_ms), 1 if inject_wait_timeout else 0, ptr(block_mask).value,
                      _status_ptr(status), 1 if sync_check else 0)
    _raise(lib.skipsm_decode_ex(ptr(q), ptr(k), ptr(v), ptr(o), B, Hq, Hkv, Skv, D, float(lam),
                                ptr(cnt), ptr(ws), ws.numel() * ws.element_size(),
                                ctypes.byref(opts), _P(_stream(stream))))
    return DecodeOut(o, cnt, ns, lse, mask)


def calibrate_prefill(q, k, v, target_skip_ratio: float, causal: bool = True, *, tile_q: int = 0,
                      tile_k: int = 0, max_iters: int = 0, out=None, stream=None,
                      exp_mode: str = "exact"):
    """lambda whose measured prefill tile skip ratio is closest to the target.

    Returns (lambda, skip_ratio, launches).  Runs the kernel max_iters times (default 14).
    """
    import torch
    lib = library()
    _check_tensor("q", q, 4), _check_tensor("k", k, 4), _check_tensor("v", v, 4)
    B, Hq, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    o = torch.empty_like(q) if out is None else out
    counts = torch.empty(2 * Hq, dtype=torch.int64, device=q.device)
    opts = PrefillOpts(tile_q, tile_k, 0.0, None, None, None, 0, _exp_mode(exp_mode))
    res = Calibration()
    _raise(lib.skipsm_prefill_calibrate(_P(q.data_ptr()), _P(k.data_ptr()), _P(v.data_ptr()),
                                        _P(o.data_ptr()), B, Hq, Hkv, Sq, Skv, D,
                                        1 if causal else 0, float(target_skip_ratio),
                                        int(max_iters), _P(counts.data_ptr()), ctypes.byref(opts),
                                        ctypes.byref(res), _P(_stream(stream))))
    return res.lambda_, res.skip_ratio, res.launches


def calibrate_decode(q, k, v, target_skip_ratio: float, *, num_splits: int = 0,
                     max_iters: int = 0, workspace=None, out=None, stream=None):
    """lambda whose measured decode tile skip ratio is closest to the target.

    Returns (lambda, skip_ratio, launches).
    """
    import torch
    lib = library()
    _check_tensor("q", q, 3), _check_tensor("k", k, 4), _check_tensor("v", v, 4)
    B, Hq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    wsb = lib.skipsm_decode_workspace_size(B, Hq, Hkv, Skv, D, num_splits)
    ws = torch.empty(wsb, dtype=torch.uint8, device=q.device) if workspace is None else workspace
    o = torch.empty_like(q) if out is None else out
    counts = torch.empty(Hq, dtype=torch.int64, device=q.device)
    opts = DecodeOpts(int(num_splits), 0.0, None, None, 0, 0)
    res = Calibration()
    _raise(lib.skipsm_decode_calibrate(_P(q.data_ptr()), _P(k.data_ptr()), _P(v.data_ptr()),
                                       _P(o.data_ptr()), B, Hq, Hkv, Skv, D,
                                       float(target_skip_ratio), int(max_iters),
                                       _P(counts.data_ptr()), _P(ws.data_ptr()),
                                       ws.numel() * ws.element_size(), ctypes.byref(opts),
                                       ctypes.byref(res), _P(_stream(stream))))
    return res.lambda_, res.skip_ratio, res.launches
