"""Seeded synthetic inputs shared by the tests, the bench and the oracle runs.

This package holds only input generation (random draws and the bf16 rounding
of the drawn values); it contains none of the MXFP4 method's arithmetic.
"""
from .synth import (CONFIGS, WorkloadConfig, bf16_bits, bf16_bits_to_f32, config_inputs,
                    normal_bf16, outlier_channels_bf16, silu_gate_bf16, student_t3_bf16)

__all__ = ["CONFIGS", "WorkloadConfig", "bf16_bits", "bf16_bits_to_f32", "config_inputs",
           "normal_bf16", "outlier_channels_bf16", "silu_gate_bf16", "student_t3_bf16"]
