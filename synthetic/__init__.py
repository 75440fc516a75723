"""Seeded synthetic operands for the GEMM workloads.

This package is the one piece shared by the oracle side and the CUDA side: it
draws numbers and encodes them as bf16 / E4M3 codes.  It holds none of the
GEMM's arithmetic.

Generator: a counter-based SplitMix64 (Steele, Lea & Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014).  Every value is a pure function
of (seed, operand stream, linear index), so any slice of an operand can be
regenerated on its own and the draws do not depend on thread count or chunking.

  key      = mix64(seed * GOLDEN + stream + 1)
  x(index) = mix64(key + (index + 1) * GOLDEN)
  uniform01 = (x >> 11) * 2^-53                         in [0, 1)
  normal    = sqrt(-2 ln u1) * cos(2 pi u2)  with u1 = ((x(2i) >> 11) + 1) * 2^-53,
                                                  u2 = uniform01(x(2i + 1))

Streams: A = 0, B = 1, sa = 2, sb = 3.
"""
from .rng import (STREAM_A, STREAM_B, STREAM_SA, STREAM_SB, normal, uniform,  # noqa: F401
                  integers, splitmix64_stream)
from .encode import to_bf16_codes, to_e4m3_codes  # noqa: F401
from .workloads import (GemmCase, make_case, make_workload_case, WORKLOADS, workload_shapes,  # noqa: F401
                        RAGGED_SWEEP, LLAMA_SHAPES, SQUARE_SHAPES, FP8_SHAPES)
