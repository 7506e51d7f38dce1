"""Plain CPU oracle for the streamed NF4-LoRA hot path (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or calls it, and the two share no
code: the oracle is plain C (``oracle.c``) compiled with gcc, double
accumulation, straight loops over the definitions.

``build()`` compiles ``liboracle.so`` next to this file; the functions below
are ctypes wrappers that take and return numpy arrays.
"""
from .binding import (  # noqa: F401
    nf4_levels,
    build,
    lib,
    num_threads,
    f32_to_bf16,
    bf16_to_f64,
    f64_to_bf16,
    quantize_nf4,
    dequant_nf4,
    philox4x32_10,
    keep_threshold,
    dropout_mask,
    lora_fwd,
    lora_bwd,
    StackCfg,
    stack_fwd_bwd,
    adam_step,
    rmsnorm_bf16,
    silu_mul_bf16,
    repeat_kv,
    rmsnorm_f64,
    rmsnorm_bwd,
    silu_mul_f64,
    silu_mul_bwd,
    repeat_kv_bwd,
    attention_fwd,
    attention_bwd,
    LIN_NAMES,
)
