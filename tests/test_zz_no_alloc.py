"""The product with library-owned scratch (dfl_q41_gemm_noalloc) against dfl_q41_gemm.

Collected after the parity files (file name), so it also runs after them in the same process; it
passes alone in a fresh process as well. Two calls in a row check that the shared static scratch is left in a
usable state (arrival counters back at zero) by each call.
"""
import ctypes

import numpy as np
import pytest

import gen
import oracle

pytestmark = pytest.mark.gpu


def _setup(torch, K, N, M, seed):
    from dflash_speculative_decode_gb300 import _abi, build
    build.build()
    L = _abi.lib()
    dev = torch.device("cuda:0")
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    W = gen.make_tensor(gen.TensorSpec("noalloc", "q41", (N, K), 0.02), seed=seed)
    src = torch.from_numpy(W.reshape(-1)).to(dev)
    img = torch.empty(L.dfl_q41_image_bytes(K, N), dtype=torch.uint8, device=dev)
    assert L.dfl_q41_pack(ctypes.c_void_p(src.data_ptr()), K, N, ctypes.c_void_p(img.data_ptr()), st) == 0
    x = torch.from_numpy(oracle.bf16_decode(gen.activations(M, K, seed=seed + 1))).to(dev)
    act = torch.empty(L.dfl_act_bytes(M, K), dtype=torch.uint8, device=dev)
    assert L.dfl_act_pack(ctypes.c_void_p(x.data_ptr()), M, K, ctypes.c_void_p(act.data_ptr()), st) == 0
    return L, st, img, act


@pytest.mark.parametrize("K,N,M", [(2560, 10240, 8), (256, 384, 5), (1280, 96, 13)])
def test_noalloc_matches_caller_scratch(K, N, M):
    torch = pytest.importorskip("torch")
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    L, st, img, act = _setup(torch, K, N, M, seed=K + N + M)
    dev = torch.device("cuda:0")
    sb = L.dfl_q41_gemm_scratch_bytes(K, N, M)
    assert 0 < sb <= L.dfl_q41_gemm_noalloc_max_scratch()
    scratch = torch.zeros(max(sb, 256), dtype=torch.uint8, device=dev)
    y_ref = torch.empty((M, N), dtype=torch.float32, device=dev)
    assert L.dfl_q41_gemm(ctypes.c_void_p(img.data_ptr()), K, N, ctypes.c_void_p(act.data_ptr()), M,
                          ctypes.c_void_p(y_ref.data_ptr()), ctypes.c_void_p(scratch.data_ptr()), sb, st) == 0
    outs = []
    for _ in range(2):   # two calls in a row on the shared static scratch
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
        assert L.dfl_q41_gemm_noalloc(ctypes.c_void_p(img.data_ptr()), K, N, ctypes.c_void_p(act.data_ptr()), M,
                                      ctypes.c_void_p(y.data_ptr()), st) == 0
        outs.append(y)
    torch.cuda.synchronize()
    ref = y_ref.cpu().numpy().astype(np.float64)
    scale = np.abs(ref).max() + 1e-30
    for y in outs:
        got = y.cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all()
        # same kernel and split: the results agree to rounding (they are in fact identical)
        assert np.abs(got - ref).max() <= 1e-6 * scale


def test_noalloc_rejects_sizes_beyond_its_scratch():
    torch = pytest.importorskip("torch")
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from dflash_speculative_decode_gb300 import _abi, build
    build.build()
    L = _abi.lib()
    cap = L.dfl_q41_gemm_noalloc_max_scratch()
    # a shape whose scratch exceeds the array: wide N with a deep split of K
    K, N = 65536, 65536
    assert L.dfl_q41_gemm_scratch_bytes(K, N, 16) > cap
    dummy = torch.empty(256, dtype=torch.uint8, device="cuda:0")
    p = ctypes.c_void_p(dummy.data_ptr())
    rc = L.dfl_q41_gemm_noalloc(p, K, N, p, 16, p, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == _abi.DFL_E_CAPACITY
