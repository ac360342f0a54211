"""Seeded synthetic workloads shared by the oracle tests, the GPU tests and the bench.

Holds only input generation (no part of the Engram computation)."""
from .configs import ALL, BY_NAME, Workload, TINY_F32, PREFILL_BF16, DECODE_BF16, INT8_HOST, MULTIBRANCH_N4  # noqa: F401
from .gen import (LayerInputs, layer_inputs, token_stream, projection_map, hash_multipliers,  # noqa: F401
                  first_primes_from, splitmix64, f32_to_bf16_bits, bf16_bits_to_f32)
