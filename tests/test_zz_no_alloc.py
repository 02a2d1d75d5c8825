"""skipsm_decode_noalloc: the decode step for callers that cannot allocate device
memory (it keeps its split partials in a fixed array owned by the library).

Collected last on purpose.  Each check compares the allocation-free call with
the ordinary skipsm_decode (caller-provided workspace) on the same inputs.
"""

import ctypes

import numpy as np
import pytest
import torch

import block_sparse_long_softmax_b300 as bs
import synth
from synth import device as sdev

pytestmark = pytest.mark.gpu

ATOL = RTOL = 1e-2
SCRATCH = 16 << 20
P, I = ctypes.c_void_p, ctypes.c_int


def _noalloc():
    f = bs.library().skipsm_decode_noalloc
    f.argtypes = [P, P, P, P] + [I] * 5 + [ctypes.c_float, P, P]
    f.restype = I
    return f


def _call(q, k, v, lam):
    B, Hq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    o = torch.full_like(q, float("nan"))
    cnt = torch.full((Hq,), -1, dtype=torch.int64, device=q.device)
    rc = _noalloc()(P(q.data_ptr()), P(k.data_ptr()), P(v.data_ptr()), P(o.data_ptr()), B, Hq,
                    Hkv, Skv, D, lam, P(cnt.data_ptr()),
                    P(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, bs.library().skipsm_last_error()
    return o, cnt


def test_noalloc_matches_decode_on_two_calls_in_a_row():
    cases = [
        (synth.WORKLOADS["decode_32k_gqa8"].with_(B=4, Skv=8192, window=512), 1e-3),
        (synth.WORKLOADS["decode_32k_gqa8"].with_(B=1, Hq=8, Hkv=2, Skv=3001, D=64,
                                                   window=256, seed=3), 1e-2),
    ]
    for w, lam in cases:  # the second call reuses scratch the first one filled
        q, k, v, _ = sdev.make_inputs(w)
        assert bs.decode_workspace_size(w.B, w.Hq, w.Hkv, w.Skv, w.D) <= SCRATCH
        o, cnt = _call(q, k, v, lam)
        ref = bs.decode(q, k, v, lam)
        torch.cuda.synchronize()
        assert bs.check() == 0
        assert torch.isfinite(o.float()).all()
        assert torch.allclose(o.float(), ref.o.float(), atol=ATOL, rtol=RTOL)
        assert torch.equal(cnt, ref.skip_counts)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # 512 sequences x 64 heads x 1 split x (128 + 1) floats > 16 MiB
    B, Hq, Hkv, Skv, D = 512, 64, 8, 256, 128
    assert bs.decode_workspace_size(B, Hq, Hkv, Skv, D) > SCRATCH
    fake = P(0x10000)  # never dereferenced: the call is refused before any launch
    rc = _noalloc()(fake, fake, fake, fake, B, Hq, Hkv, Skv, D, 1e-3, None, None)
    assert rc == 5
    assert b"workspace" in bs.library().skipsm_last_error()
