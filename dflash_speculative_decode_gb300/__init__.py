"""DFlash speculative decode over Q4_1 weights on one GB300 (sm_103a).

The step (draft block -> batched verify -> accept -> commit_verify_rows) runs in libdfl.so, a CUDA
library with a C ABI (include/dfl.h). This package holds its build script, the ctypes binding with the
ABI's names (`_abi`), and the decode loops a caller drives (`decode`).
"""
from ._abi import (DFL_KEEP_ACCEPTED, DFL_OPT_GRAPHS, DFL_OPT_KEEP_LOGITS, DflError, Engine, config_from_pair,
                   dfl_config, lib)
from .decode import Generation, PrefixCache, plain_decode, serve_single_turn, spec_decode

__all__ = ["Engine", "DflError", "config_from_pair", "dfl_config", "lib", "plain_decode", "spec_decode", "Generation", "PrefixCache", "serve_single_turn",
           "DFL_KEEP_ACCEPTED", "DFL_OPT_KEEP_LOGITS", "DFL_OPT_GRAPHS"]
