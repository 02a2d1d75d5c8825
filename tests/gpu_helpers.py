"""Shared helpers of the GPU parity tests (inputs, host copies, comparisons)."""

import numpy as np
import pytest
import torch

import synth
from synth import device as sdev

ATOL = 1e-2
RTOL = 1e-2
MARGIN = 1e-3  # nats: masks must agree on every tile decided by more than this

needs_gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


def to_f64(t: torch.Tensor) -> np.ndarray:
    """bf16 CUDA tensor -> exact fp64 numpy array."""
    bits = t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return synth.bf16_bits_to_f64(bits)


def device_inputs(w):
    q, k, v, dt = sdev.make_inputs(w)
    torch.cuda.synchronize()
    return q, k, v, dt


def assert_close(o_gpu: np.ndarray, o_ref: np.ndarray, what="output"):
    err = np.abs(o_gpu - o_ref)
    bound = ATOL + RTOL * np.abs(o_ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} elements out of tolerance, "
                           f"max err {err.max():.3e}")


def assert_masks(mask_gpu: np.ndarray, mask_ref: np.ndarray, margin: np.ndarray, what="mask"):
    sure = margin > MARGIN
    diff = (mask_gpu != mask_ref) & sure
    assert not diff.any(), f"{what}: {diff.sum()} confident tiles disagree"
    return int(((mask_gpu != mask_ref) & ~sure).sum())
