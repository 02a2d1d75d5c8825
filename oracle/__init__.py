"""fp64 CPU oracle of the Skip Softmax attention path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline``
and reference legs of ``bench.py`` use it.  It shares no code with the CUDA
library; the only common dependency is the seeded input generator ``synth``.

Parity is pinned for every function here (see ``tests/test_oracle_pins.py``):
dense attention from a library routine at lambda = 0, an independent
closed-form skip mask, a closed-form output over the kept keys, monotonicity
in lambda, the analytic error bound, and hand-derived worked examples.  The
optional Rowmax-PoT weights are pinned in ``tests/test_oracle_pot.py`` (worked
examples, reduction to dense softmax for integer exponents, a bound against
dense softmax, planted mistakes); the optional FP8 P.V weights in ``tests/test_oracle_fp8_pv.py`` (e4m3 rounding
against worked values and torch's cast, a hand-worked example, reduction to the
exact oracle when every scaled weight is an e4m3 value, a bound against it, planted
mistakes); the optional decode block mask in
``tests/test_oracle_blockmask.py`` (SDPA over the selected keys, invariance to
unselected keys, worked examples, planted mistakes).
"""

from .skipsm_oracle import (  # noqa: F401
    PrefillResult,
    DecodeResult,
    prefill,
    prefill_qtile,
    decode,
    decode_group,
    decode_split_geometry,
    dense_attention,
    skipped_mass,
    e4m3_round,
    FP8_AMBIGUOUS_BAND,
)
