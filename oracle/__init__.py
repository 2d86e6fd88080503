"""ORACLE -- test infrastructure, not part of the library.

A plain, slow, obviously checkable CPU implementation of one DFlash speculative-decode step over
Q4_1 weights: products in C (dfl_oracle.c, double precision, ascending reduction order), the rest in
double-precision numpy one row at a time. Only tests/, the smoke check and the benchmark's
CPU-baseline and reference legs may import it. It shares no code with the CUDA path; the only
module both sides use is the seeded input generator `gen`, which holds none of the step's arithmetic.
"""
from . import _native
from ._native import (bf16r, bf16_decode, half_decode, linear_bf16, linear_q41, q41_dequant, sample, set_threads, threads,
                      uniform)
from .model import (Draft, Target, attend, keep_positions, kv_widths, ple_tail, positions_held, rmsnorm, rope, silu,
                    swiglu)
from .spec import Pair, Run, Sampler, accept_length, plain_decode, serve_single_turn, spec_decode


def build() -> str:
    """Compile the oracle's C numerics (building the checker does not run it)."""
    return _native.build()
