"""The CUDA input generator is bit-identical to the numpy one."""

import numpy as np
import pytest
import torch

import synth
from synth import planted as P
from gpu_helpers import device_inputs

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("w", [
    synth.WORKLOADS["prefill_1k_d64"].with_(B=2, Hq=4, Hkv=2, Sq=300, Skv=500, window=64),
    synth.WORKLOADS["decode_32k_gqa8"].with_(B=2, Skv=3000, window=256),
    synth.WORKLOADS["prefill_32k_gqa8"].with_(Hq=16, Hkv=2, Sq=1000, Skv=1000, window=256),
])
def test_device_generator_bit_exact(w):
    q, k, v, dt = device_inputs(w)
    t, qh, kh, vh = synth.gen_all(w)
    assert np.array_equal(_bits(q), qh)
    assert np.array_equal(_bits(k), kh)
    assert np.array_equal(_bits(v), vh)


def test_device_generator_full_size_rows():
    w = synth.WORKLOADS["decode_128k_gqa8"]
    q, k, v, dt = device_inputs(w)
    t = dt.host
    assert np.array_equal(_bits(q[7, 63:64]), P.gen_q_rows(w, t, 7, 63))
    assert np.array_equal(_bits(k[7, 7, 131000:131072]), P.gen_k_rows(w, t, 7, 7, 131000, 131072))
    assert np.array_equal(_bits(v[3, 2, :50]), P.gen_v_rows(w, 3, 2, 0, 50))
