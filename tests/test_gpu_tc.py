"""The Q4_1 product at many rows on the tcgen05 tensor cores (dfl_q41_gemm_tc) against the oracle."""
import ctypes

import numpy as np
import pytest

import gen
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from dflash_speculative_decode_gb300 import build
    build.build()
    return torch


def _tc(torch, W, x, K, N):
    """Pack W (container layout [N][K/32][20]), run the tcgen05 product on fp32 rows x [M][K]."""
    from dflash_speculative_decode_gb300 import _abi
    L = _abi.lib()
    M = x.shape[0]
    dev = torch.device("cuda:0")
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    src = torch.from_numpy(W.reshape(-1)).to(dev)
    img = torch.empty(L.dfl_q41_image_bytes(K, N), dtype=torch.uint8, device=dev)
    assert L.dfl_q41_pack(ctypes.c_void_p(src.data_ptr()), K, N, ctypes.c_void_p(img.data_ptr()), st) == 0
    xd = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(dev)
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
    sb = L.dfl_q41_gemm_tc_scratch_bytes(K, N, M)
    assert sb > 0
    scratch = torch.zeros(sb + 1024, dtype=torch.uint8, device=dev)
    base = (scratch.data_ptr() + 1023) // 1024 * 1024
    rc = L.dfl_q41_gemm_tc(ctypes.c_void_p(img.data_ptr()), K, N, ctypes.c_void_p(xd.data_ptr()), M,
                           ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(base), sb, st)
    assert rc == 0
    assert L.dfl_q41_gemm_status(ctypes.c_void_p(base), st) == 0
    torch.cuda.synchronize()
    return y.cpu().numpy()


def _bound(x, W):
    """hi/lo splits of x and w (2^-17 each, and the dropped lo*lo term) plus fp32 accumulation over K."""
    xd = np.abs(x.astype(np.float64))
    wd = np.abs(oracle.q41_dequant(W).reshape(W.shape[0], -1))
    K = x.shape[1]
    return (xd @ wd.T) * (2.0 ** -15 + (K + 64) * 2.0 ** -23) + 1e-6


def _case(K, N, M, seed):
    rng = np.random.default_rng(seed)
    W = gen.pack_q41((rng.standard_normal((N, K)) * 0.02).astype(np.float32))
    x = rng.standard_normal((M, K)).astype(np.float32)
    return W, x


@pytest.mark.parametrize("K,N,M", [(64, 128, 128), (256, 256, 128), (96, 160, 200), (640, 384, 256),
                                   (2560, 512, 384), (1280, 1056, 130), (32, 32, 1), (320, 2592, 129)])
def test_tc_gemm_matches_oracle(torch_cuda, K, N, M):
    """Tiles of 128 x 128 with ragged edges in every dimension (K not a multiple of 64, N not a multiple
    of 128, M not a multiple of 128), against the oracle's fp64 product."""
    W, x = _case(K, N, M, K * 13 + N * 7 + M)
    y = _tc(torch_cuda, W, x, K, N)
    ref = oracle.linear_q41(x, W).astype(np.float64)
    assert np.isfinite(y).all()
    err = np.abs(y - ref)
    assert np.all(err <= _bound(x, W)), f"max err {err.max():.3g}"


def test_tc_gemm_rows_independent_of_batch(torch_cuda):
    """A row's result does not depend on how many rows the call carries or which tile holds it."""
    K, N = 1024, 384
    W, x = _case(K, N, 300, 3)
    full = _tc(torch_cuda, W, x, K, N)
    for M in (1, 128, 129, 200):
        np.testing.assert_array_equal(_tc(torch_cuda, W, x[:M], K, N), full[:M])


def test_tc_gemm_one_hot(torch_cuda):
    """x = e_k returns the dequantised weights of input k to the split's precision (2^-16 relative)."""
    K, N = 512, 256
    W, _ = _case(K, N, 1, 4)
    ks = np.array([0, 1, 31, 32, 63, 64, 200, 511, 7, 100, 300, 450, 17, 33, 65, 255])
    x = np.zeros((len(ks), K), np.float32)
    x[np.arange(len(ks)), ks] = 1.0
    y = _tc(torch_cuda, W, x, K, N)
    deq = oracle.q41_dequant(W).reshape(N, K)
    for m, k in enumerate(ks):
        np.testing.assert_allclose(y[m], deq[:, k], rtol=2.0 ** -16, atol=1e-9)


@pytest.mark.parametrize("K,N,M", [(2560, 10240, 512), (10240, 2560, 256), (5376, 8192, 1024)])
def test_tc_gemm_full_size_sampled_columns(torch_cuda, K, N, M):
    """Prompt-ingest shapes of the E4B and 27B-class layers: sampled output columns against the oracle."""
    rng = np.random.default_rng(K + N + M)
    W = gen.make_tensor(gen.TensorSpec("sweep", "q41", (N, K), 0.02), seed=5)
    x = rng.standard_normal((M, K)).astype(np.float32)
    y = _tc(torch_cuda, W, x, K, N)
    cols = np.unique(np.concatenate([rng.integers(0, N, 24), [0, 127, 128, N - 1]]))
    rows = np.unique(np.concatenate([rng.integers(0, M, 24), [0, 127, 128, M - 1]]))
    Wc = W[cols]
    ref = oracle.linear_q41(x[rows], Wc).astype(np.float64)
    assert np.all(np.abs(y[np.ix_(rows, cols)] - ref) <= _bound(x[rows], Wc))


def test_tc_gemm_agrees_with_skinny_product(torch_cuda):
    """On bf16-valued rows both products approximate the same exact sum: within both bounds."""
    from test_gpu_parity import _gemm
    K, N = 1280, 512
    rng = np.random.default_rng(6)
    W = gen.pack_q41((rng.standard_normal((N, K)) * 0.02).astype(np.float32))
    xb = gen.bf16_bits(rng.standard_normal((16, K)).astype(np.float32))
    xf = oracle.bf16_decode(xb)
    small, _ = _gemm(torch_cuda, W, xb, K, N)
    big = np.concatenate([_tc(torch_cuda, W, np.tile(xf, (8, 1)), K, N)[:16]])
    assert np.all(np.abs(small - big) <= 2 * _bound(xf, W))
