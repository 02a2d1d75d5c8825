"""Seeded synthetic attention inputs with planted structure.

This module is the only code shared by the oracle side and the CUDA side.  It
synthesises inputs; it holds none of the attention arithmetic.  The numpy
generator (`planted`) and the CUDA generator (`device`, a separate shared
library) produce bit-identical bf16 tensors from the same `Workload`.
"""

from .planted import (  # noqa: F401
    Workload,
    PlantTables,
    make_tables,
    gen_q,
    gen_k,
    gen_v,
    gen_all,
    bf16_bits_to_f64,
    bf16_bits_to_f32,
    f32_to_bf16_bits,
    e4m3_round,
    normal_bits,
    WORKLOADS,
)
