"""CPU oracle of the sparse-decode KV offload step (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg may use
this package; the library path never imports it.
"""
from .oracle import (  # noqa: F401
    OK, EINVAL, ENOMEM, ERANGE, ECAPACITY, PAD_PAYLOAD, DIM, OracleUnit, StepResult, build,
    compile_source,
    lib, score, step_many, threads, f32_to_f16, f16_to_f32, fwht128, quant_rotated, quant128,
    score_i8, attend_rows,
)
