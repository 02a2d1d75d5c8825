"""Device twin of the planted-structure generator (CUDA, bit-identical to numpy).

Builds ``synth/libplanted.so`` on first use (or via ``build()``) and fills
torch bf16 CUDA tensors in place.  Used by the benchmark and the GPU tests to
create large inputs directly in HBM.
"""

from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

from .planted import PlantTables, Workload, make_tables, stream_key

HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(HERE, "libplanted.so")
SRC = os.path.join(HERE, "planted_dev.cu")
_lib = None


def build() -> str:
    if os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-Xcompiler", "-fPIC", "-shared", "-fmad=false", SRC, "-o", LIB + ".tmp"],
                   check=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


def _load():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        _lib.planted_fill.restype = ctypes.c_int
        _lib.planted_fill.argtypes = [ctypes.c_void_p, ctypes.c_ulonglong] + [ctypes.c_int] * 15 + \
            [ctypes.c_void_p] * 4
    return _lib


class DeviceTables:
    """The planted tables of a workload, resident on the GPU."""

    def __init__(self, w: Workload, t: PlantTables = None, device="cuda"):
        import torch
        t = make_tables(w) if t is None else t
        self.host = t
        self.qu = torch.from_numpy(t.qu.copy()).to(device)
        self.ku = torch.from_numpy(t.ku.copy()).to(device)
        nw = t.qv.shape[1]
        self.nw = nw
        self.qv = torch.from_numpy(t.qv.reshape(-1).copy() if nw else t.qu.reshape(-1).copy()).to(device)
        self.kv = torch.from_numpy(t.kv.reshape(-1).copy() if nw else t.ku.reshape(-1).copy()).to(device)
        self.rblk = torch.from_numpy(t.rblk.reshape(-1).copy()).to(device)
        self.nrb = t.rblk.shape[2]


def fill(w: Workload, dt: DeviceTables, tensor: str, out, stream=None) -> None:
    """Fill `out` (torch bf16 CUDA tensor, contiguous) with Q, K or V of workload w."""
    import torch
    assert out.dtype == torch.bfloat16 and out.is_cuda and out.is_contiguous()
    tid = {"q": 1, "k": 2, "v": 3}[tensor]
    if tensor == "q":
        H, S = w.Hq, (1 if w.kind == "decode" else w.Sq)
    else:
        H, S = w.Hkv, w.Skv
    assert out.numel() == w.B * H * S * w.D
    tu = dt.qu if tensor == "q" else dt.ku
    tv = dt.qv if tensor == "q" else dt.kv
    s = torch.cuda.current_stream().cuda_stream if stream is None else stream
    rc = _load().planted_fill(out.data_ptr(), stream_key(w.seed, tensor), tid, w.B, H, S, w.D, w.G,
                              w.Hkv, w.Sq, w.Skv, w.window, w.sink, w.rblock, dt.nrb, dt.nw,
                              1 if w.kind == "decode" else 0, tu.data_ptr(), tv.data_ptr(),
                              dt.rblk.data_ptr(), s)
    if rc != 0:
        raise RuntimeError(f"planted_fill failed (cuda error {rc})")


def make_inputs(w: Workload, device="cuda"):
    """(q, k, v, tables) as bf16 CUDA tensors generated on the device."""
    import torch
    dt = DeviceTables(w, device=device)
    qshape = (w.B, w.Hq, w.D) if w.kind == "decode" else (w.B, w.Hq, w.Sq, w.D)
    q = torch.empty(qshape, dtype=torch.bfloat16, device=device)
    k = torch.empty((w.B, w.Hkv, w.Skv, w.D), dtype=torch.bfloat16, device=device)
    v = torch.empty_like(k)
    fill(w, dt, "q", q)
    fill(w, dt, "k", k)
    fill(w, dt, "v", v)
    return q, k, v, dt
