"""Seeded synthetic inputs for the DFlash2 draft + select + verify step.

This package holds no arithmetic of the method itself: it only draws seeded
random numbers (weights, feature taps, context K/V, noise) in the layouts the
C ABI and the oracle both consume.  Both the CUDA path (through its Python
binding) and the CPU oracle take their inputs from here.
"""
from .configs import Geometry, Workload, TOY, FULL, WORKLOADS, workload  # noqa: F401
from .gen import (  # noqa: F401
    bf16_bits_from_f32, f32_from_bf16_bits, quantize_q8g64, make_weights,
    make_request_inputs, make_target_noise, tap_rows, kv_rows, make_selector_inputs,
    make_verify_inputs, WEIGHT_NAMES_GLOBAL,
    WEIGHT_NAMES_LAYER, MATRIX_NAMES,
)
