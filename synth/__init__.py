"""Seeded synthetic inputs shared by the oracle and the CUDA path.

This package only draws numbers: a counter-based SplitMix64 stream (Steele, Lea
and Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014; the
64-bit finaliser constants are the published ones) and the value mappings that
turn 16-bit fields of each draw into the workloads' value distributions. It
holds none of the decode path's arithmetic (no scoring, selection, cache rule,
dequantisation or attention).

Every tensor element is addressed by (stream key, field index), so any row of
any history or any step's queries can be regenerated alone, on the host with
numpy (``synth.rng``) or on the GPU (``synth.gpu``), and both give identical
bytes.
"""
from .rng import (  # noqa: F401
    stream_key, fields16, uniform_int_fields, normal_fields_f32,
    f32_to_bf16_bits, bf16_bits_to_f32,
)
from .workloads import WORKLOADS, Workload, UnitInputs  # noqa: F401
