"""Per-call device status words (the `status` option of the _ex calls).

By default a timed-out wait is recorded in the library's one status word per
device, which every caller shares and skipsm_check clears.  A caller that passes
its own word gets its calls' failures there instead, and the shared word stays
clean.  The failure is made the way the other failure-detection tests make it: one
wait per CTA on a barrier nothing arrives at, with a 20 ms bound, so the kernel
winds down and returns; nothing traps or faults.
"""

import pytest
import torch

import block_sparse_long_softmax_b300 as bs
import synth
from gpu_helpers import device_inputs

pytestmark = pytest.mark.gpu


def test_prefill_timeout_goes_to_the_callers_word():
    w = synth.WORKLOADS["prefill_32k_gqa8"].with_(B=1, Hq=2, Hkv=1, Sq=300, Skv=300, window=64)
    q, k, v, _ = device_inputs(w)
    st = torch.zeros(1, dtype=torch.int32, device=q.device)
    bs.prefill(q, k, v, 1e-3, wait_limit_ms=20, inject_wait_timeout=True, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 25
    assert bs.check() == 0          # the shared word saw nothing
    # a clean call leaves the caller's word at zero, and is correct
    st.zero_()
    out = bs.prefill(q, k, v, 1e-3, status=st)
    ref = bs.prefill(q, k, v, 1e-3)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and bs.check() == 0
    assert torch.equal(out.o, ref.o)


def test_decode_timeout_goes_to_the_callers_word():
    w = synth.WORKLOADS["decode_32k_gqa8"].with_(B=1, Hq=8, Hkv=1, Skv=1024, window=128)
    q, k, v, _ = device_inputs(w)
    st = torch.zeros(1, dtype=torch.int32, device=q.device)
    bs.decode(q, k, v, 1e-3, num_splits=1, wait_limit_ms=20, inject_wait_timeout=True, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 7
    assert bs.check() == 0
    st.zero_()
    out = bs.decode(q, k, v, 1e-3, status=st)
    ref = bs.decode(q, k, v, 1e-3)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and bs.check() == 0
    assert torch.equal(out.o, ref.o)


def test_status_must_be_an_int32_device_word():
    w = synth.WORKLOADS["decode_32k_gqa8"].with_(B=1, Hq=8, Hkv=1, Skv=256, window=64)
    q, k, v, _ = device_inputs(w)
    with pytest.raises(TypeError):
        bs.decode(q, k, v, 1e-3, status=torch.zeros(1, dtype=torch.int64, device=q.device))


@pytest.mark.parametrize("own_word", [False, True])
def test_sync_check_reports_the_timeout(own_word):
    """sync_check: the call waits for the stream and returns SKIPSM_ERR_TIMEOUT (4) when one of
    its waits ran out; the shared word is read and cleared, a caller's own word is left set."""
    w = synth.WORKLOADS["prefill_32k_gqa8"].with_(B=1, Hq=2, Hkv=1, Sq=300, Skv=300, window=64)
    q, k, v, _ = device_inputs(w)
    st = torch.zeros(1, dtype=torch.int32, device=q.device) if own_word else None
    with pytest.raises(bs.SkipsmError) as e:
        bs.prefill(q, k, v, 1e-3, wait_limit_ms=20, inject_wait_timeout=True, status=st,
                   sync_check=True)
    assert e.value.status == 4 and "site 25" in str(e.value)
    assert bs.check() == 0            # cleared by the call, or never set
    if own_word:
        assert int(st.item()) == 25
    # a clean call with sync_check returns normally and is correct
    out = bs.prefill(q, k, v, 1e-3, sync_check=True)
    ref = bs.prefill(q, k, v, 1e-3)
    torch.cuda.synchronize()
    assert torch.equal(out.o, ref.o)


def test_decode_sync_check():
    w = synth.WORKLOADS["decode_32k_gqa8"].with_(B=1, Hq=8, Hkv=1, Skv=1024, window=128)
    q, k, v, _ = device_inputs(w)
    with pytest.raises(bs.SkipsmError) as e:
        bs.decode(q, k, v, 1e-3, num_splits=1, wait_limit_ms=20, inject_wait_timeout=True,
                  sync_check=True)
    assert e.value.status == 4 and "site 7" in str(e.value)
    assert bs.check() == 0
    out = bs.decode(q, k, v, 1e-3, sync_check=True)
    ref = bs.decode(q, k, v, 1e-3)
    torch.cuda.synchronize()
    assert torch.equal(out.o, ref.o)
