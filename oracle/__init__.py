"""NVFP4 CPU oracle -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` leg of
``bench.py`` may import this package. The product package never imports it,
and the two share no code: the C file ``nvfp4_oracle.c`` is written from the
format definitions on the "nvfp4-gemma4" page (section 2) and the storage
layout on the "nvfp4-difusion" page (section 2); see its header for the
readings taken where the pages are silent.
"""
from .oracle import (  # noqa: F401
    build,
    lib_path,
    num_threads,
    e2m1_value,
    e4m3_value,
    e4m3_rne_satfinite,
    e2m1_rne_satfinite,
    bf16_from_double,
    global_scale,
    quantize,
    SCALE_ABSMAX,
    SCALE_FOUR_OVER_SIX,
    SCALE_MSE,
    dequantize,
    gemm,
    gemm_rows,
    lora_rows,
    round_bf16,
    linear_lora_rows,
    symmetric_quantize,
)
