"""Out-of-bounds writes: every output of a C ABI call sits between guard bands.

Each output buffer (and the decode workspace) is carved from a larger device allocation
whose bytes are all set to a sentinel first.  After the call the guard bands on both
sides must still hold the sentinel everywhere, and the buffers the header declares as
fully written (o, lse, skip_mask, the counts) must hold no sentinel value any more.
Shapes are ragged (partial query and key tiles, Sq < Skv, odd split counts) so that the
kernels' tail handling is what gets checked.
"""

import ctypes

import numpy as np
import pytest
import torch

import block_sparse_long_softmax_b300 as bs
import synth
from synth import device as sdev

pytestmark = pytest.mark.gpu

P = ctypes.c_void_p
GUARD = 4096          # bytes on each side; keeps the 256-byte alignment of the buffer
SENTINEL = 0xA5


class Guarded:
    """A typed view of `nbytes` device bytes with sentinel-filled guard bands around it."""

    def __init__(self, shape, dtype):
        itemsize = torch.empty((), dtype=dtype).element_size()
        n = int(np.prod(shape)) * itemsize
        self.nbytes = n
        self.raw = torch.full((GUARD + n + GUARD,), SENTINEL, dtype=torch.uint8, device="cuda")
        self.t = self.raw[GUARD:GUARD + n].view(dtype).view(shape)

    def ptr(self):
        return P(self.t.data_ptr())

    def guards_intact(self):
        g = torch.cat([self.raw[:GUARD], self.raw[GUARD + self.nbytes:]])
        return bool((g == SENTINEL).all().item())

    def fully_written(self):
        """No element still has every byte equal to the sentinel."""
        body = self.raw[GUARD:GUARD + self.nbytes]
        item = self.t.element_size()
        per_elem = (body == SENTINEL).view(-1, item).all(dim=1)
        return not bool(per_elem.any().item())


def _stream():
    return P(torch.cuda.current_stream().cuda_stream)


PREFILL = [
    # (workload overrides, tile_q, tile_k, exp_mode, block mask density)
    (dict(B=1, Hq=4, Hkv=2, Sq=700, Skv=700, D=128, window=128), 128, 128, 0, None),
    (dict(B=1, Hq=4, Hkv=2, Sq=700, Skv=700, D=128, window=128), 64, 64, 0, None),
    (dict(B=2, Hq=2, Hkv=1, Sq=520, Skv=520, D=64, window=64), 64, 64, 0, None),
    (dict(B=1, Hq=2, Hkv=2, Sq=200, Skv=777, D=128, window=128), 128, 128, 1, None),
    (dict(B=1, Hq=2, Hkv=1, Sq=300, Skv=520, D=128, window=128, causal=False), 128, 128, 0, 0.5),
    (dict(B=1, Hq=4, Hkv=2, Sq=700, Skv=700, D=128, window=128), 64, 128, 0, 0.6),
]


@pytest.mark.parametrize("case", range(len(PREFILL)))
def test_prefill_writes_stay_in_bounds(case):
    over, tq, tk, exp_mode, density = PREFILL[case]
    w = synth.WORKLOADS["prefill_32k_gqa8"].with_(**over)
    q, k, v, _ = sdev.make_inputs(w)
    B, Hq, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    nqt, nkt = -(-Sq // tq), -(-Skv // tk)
    o = Guarded((B, Hq, Sq, D), torch.bfloat16)
    lse = Guarded((B, Hq, Sq), torch.float32)
    mask = Guarded((B, Hq, nqt, nkt), torch.uint8)
    vis = Guarded((Hq,), torch.int64)
    cnt = Guarded((Hq,), torch.int64)
    bm = None
    if density is not None:
        g = torch.Generator(device="cpu").manual_seed(case)
        bm = (torch.rand((B, Hq, nqt, nkt), generator=g) < density).to(torch.uint8).cuda()
    lib = bs.library()
    opts = bs.PrefillOpts(tq, tk, 0.0, lse.t.data_ptr(), mask.t.data_ptr(), vis.t.data_ptr(),
                          0, exp_mode, 0, 0.0, bm.data_ptr() if bm is not None else None, 0)
    rc = lib.skipsm_prefill_ex(P(q.data_ptr()), P(k.data_ptr()), P(v.data_ptr()), o.ptr(), B, Hq,
                               Hkv, Sq, Skv, D, 1 if w.causal else 0, 1e-3, cnt.ptr(),
                               ctypes.byref(opts), _stream())
    assert rc == 0, lib.skipsm_last_error()
    torch.cuda.synchronize()
    assert bs.check() == 0
    for name, buf in (("o", o), ("lse", lse), ("skip_mask", mask), ("visited", vis),
                      ("skip_counts", cnt)):
        assert buf.guards_intact(), f"{name}: write outside its buffer"
        assert buf.fully_written(), f"{name}: elements left unwritten"


DECODE = [
    # (workload overrides, splits, block mask density)
    (dict(B=2, Hq=16, Hkv=2, Skv=4096 + 37, D=128, window=256), 0, None),
    (dict(B=2, Hq=16, Hkv=2, Skv=4096 + 37, D=128, window=256), 5, None),
    (dict(B=1, Hq=8, Hkv=8, Skv=1000, D=64, window=128), 3, None),
    (dict(B=1, Hq=8, Hkv=1, Skv=65, D=128, window=16), 2, 0.5),
    (dict(B=3, Hq=8, Hkv=2, Skv=2500, D=128, window=128), 7, 0.3),
]


@pytest.mark.parametrize("case", range(len(DECODE)))
def test_decode_writes_stay_in_bounds(case):
    over, splits, density = DECODE[case]
    w = synth.WORKLOADS["decode_32k_gqa8"].with_(**over)
    q, k, v, _ = sdev.make_inputs(w)
    B, Hq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    nblk = -(-Skv // 64)
    lib = bs.library()
    wsb = lib.skipsm_decode_workspace_size(B, Hq, Hkv, Skv, D, splits)
    assert wsb > 0
    o = Guarded((B, Hq, D), torch.bfloat16)
    lse = Guarded((B, Hq), torch.float32)
    mask = Guarded((B, Hkv, nblk), torch.uint8)
    cnt = Guarded((Hq,), torch.int64)
    ws = Guarded((wsb,), torch.uint8)
    bm = None
    if density is not None:
        g = torch.Generator(device="cpu").manual_seed(100 + case)
        bm = (torch.rand((B, Hkv, nblk), generator=g) < density).to(torch.uint8).cuda()
    opts = bs.DecodeOpts(splits, 0.0, lse.t.data_ptr(), mask.t.data_ptr(), 0, 0,
                         bm.data_ptr() if bm is not None else None)
    rc = lib.skipsm_decode_ex(P(q.data_ptr()), P(k.data_ptr()), P(v.data_ptr()), o.ptr(), B, Hq,
                              Hkv, Skv, D, 1e-3, cnt.ptr(), ws.ptr(), wsb, ctypes.byref(opts),
                              _stream())
    assert rc == 0, lib.skipsm_last_error()
    torch.cuda.synchronize()
    assert bs.check() == 0
    for name, buf in (("o", o), ("lse", lse), ("skip_mask", mask), ("skip_counts", cnt),
                      ("workspace", ws)):
        assert buf.guards_intact(), f"{name}: write outside its buffer"
    for name, buf in (("o", o), ("lse", lse), ("skip_mask", mask), ("skip_counts", cnt)):
        assert buf.fully_written(), f"{name}: elements left unwritten"
