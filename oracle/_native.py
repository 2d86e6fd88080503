"""ctypes access to the oracle's C numerics (dfl_oracle.c). Test infrastructure only."""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dfl_oracle.c")
_SO = os.path.join(_HERE, "libdfl_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle's C file with the host compiler (no machine-specific flags)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                               "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
        f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
        u16p = np.ctypeslib.ndpointer(np.uint16, flags="C_CONTIGUOUS")
        u8p = np.ctypeslib.ndpointer(np.uint8, flags="C_CONTIGUOUS")
        L.orc_bf16_round.argtypes = [f32p, f32p, ctypes.c_long]
        L.orc_bf16_decode.argtypes = [u16p, f32p, ctypes.c_long]
        L.orc_half_decode.argtypes = [u16p, f64p, ctypes.c_long]
        L.orc_q41_dequant.argtypes = [u8p, ctypes.c_long, f64p]
        L.orc_linear_q41.argtypes = [f32p, ctypes.c_int, ctypes.c_int, u8p, ctypes.c_int, f32p]
        L.orc_linear_bf16.argtypes = [f32p, ctypes.c_int, ctypes.c_int, u16p, ctypes.c_int, f32p]
        L.orc_uniform.argtypes = [ctypes.c_uint64, ctypes.c_int64]
        L.orc_uniform.restype = ctypes.c_double
        L.orc_sample.argtypes = [f32p, ctypes.c_int, ctypes.c_double, ctypes.c_double,
                                 ctypes.POINTER(ctypes.c_double)]
        L.orc_sample.restype = ctypes.c_int
        L.orc_set_threads.argtypes = [ctypes.c_int]
        L.orc_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def bf16r(x) -> np.ndarray:
    """Round to the nearest bf16 value (ties to even); returned as float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty_like(x)
    lib().orc_bf16_round(x.reshape(-1), y.reshape(-1), x.size)
    return y


def bf16_decode(b) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    y = np.empty(b.shape, np.float32)
    lib().orc_bf16_decode(b.reshape(-1), y.reshape(-1), b.size)
    return y


def half_decode(h) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    y = np.empty(h.shape, np.float64)
    lib().orc_half_decode(h.reshape(-1), y.reshape(-1), h.size)
    return y


def q41_dequant(blocks) -> np.ndarray:
    """uint8 [..., 20] Q4_1 blocks -> float64 [..., 32] weights d*q + m."""
    b = np.ascontiguousarray(blocks, dtype=np.uint8)
    nb = b.size // 20
    w = np.empty(nb * 32, np.float64)
    lib().orc_q41_dequant(b.reshape(-1), nb, w)
    return w.reshape(b.shape[:-1] + (32,))


def linear_q41(x, W) -> np.ndarray:
    """x float32 [R][K] (bf16-valued) times Q4_1 W uint8 [N][K/32][20] -> float32 [R][N]."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    R, K = x.shape
    N = W.shape[0]
    assert W.shape == (N, K // 32, 20)
    y = np.empty((R, N), np.float32)
    lib().orc_linear_q41(x, R, K, np.ascontiguousarray(W), N, y)
    return y


def linear_bf16(x, W) -> np.ndarray:
    """x float32 [R][K] times bf16 W uint16 [N][K] -> float32 [R][N]."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    R, K = x.shape
    N = W.shape[0]
    assert W.shape == (N, K)
    y = np.empty((R, N), np.float32)
    lib().orc_linear_bf16(x, R, K, np.ascontiguousarray(W), N, y)
    return y


def set_threads(n: int) -> None:
    """Threads the products use (OpenMP over output columns; every result is the same for any count)."""
    lib().orc_set_threads(int(n))


def threads() -> int:
    return int(lib().orc_threads())


def uniform(seed: int, pos: int) -> float:
    return lib().orc_uniform(ctypes.c_uint64(seed & 0xFFFFFFFFFFFFFFFF), int(pos))


def sample(logits, T: float, u: float):
    """(token, relative distance of u*sum(p) to the chosen interval's nearer edge)."""
    l = np.ascontiguousarray(logits, dtype=np.float32)
    g = ctypes.c_double(0.0)
    j = lib().orc_sample(l, l.size, float(T), float(u), ctypes.byref(g))
    return int(j), float(g.value)
