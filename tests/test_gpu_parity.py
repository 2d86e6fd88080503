"""GPU parity: the CUDA path, called through the C ABI, against the oracle on the same seeded inputs."""
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


# ---------------------------------------------------------------------------------------------------
# the Q4_1 product on its own
# ---------------------------------------------------------------------------------------------------
def _gemm(torch, W, x_bits, K, N):
    """Pack W, pack the (bf16-valued) activations into the operand format, run the product."""
    from dflash_speculative_decode_gb300 import _abi
    L = _abi.lib()
    M = x_bits.shape[0]
    dev = torch.device("cuda:0")
    src = torch.from_numpy(W.reshape(-1)).to(dev)
    img = torch.empty(L.dfl_q41_image_bytes(K, N), dtype=torch.uint8, device=dev)
    st = torch.cuda.current_stream().cuda_stream
    assert L.dfl_q41_pack(ctypes.c_void_p(src.data_ptr()), K, N, ctypes.c_void_p(img.data_ptr()), ctypes.c_void_p(st)) == 0
    x = torch.from_numpy(oracle.bf16_decode(x_bits)).to(dev)
    act = torch.empty(L.dfl_act_bytes(M, K), dtype=torch.uint8, device=dev)
    assert L.dfl_act_pack(ctypes.c_void_p(x.data_ptr()), M, K, ctypes.c_void_p(act.data_ptr()), ctypes.c_void_p(st)) == 0
    y = torch.empty((M, N), dtype=torch.float32, device=dev)
    sb = L.dfl_q41_gemm_scratch_bytes(K, N, M)
    scratch = torch.zeros(max(sb, 256), dtype=torch.uint8, device=dev)
    rc = L.dfl_q41_gemm(ctypes.c_void_p(img.data_ptr()), K, N, ctypes.c_void_p(act.data_ptr()), M,
                        ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(scratch.data_ptr()), sb, ctypes.c_void_p(st))
    assert rc == 0
    torch.cuda.synchronize()
    return y.cpu().numpy(), (img, scratch)


def _bound(x, W):
    """|y_gpu - y_exact| bound: fp32 accumulation over K terms of |x w| plus the split into blocks."""
    xd = np.abs(oracle.bf16_decode(x).astype(np.float64))
    wd = np.abs(oracle.q41_dequant(W).reshape(W.shape[0], -1))
    return (xd @ wd.T) * (x.shape[1] + 64) * 2.0 ** -24 + 1e-6


@pytest.mark.parametrize("K,N,M", [(64, 32, 1), (256, 384, 8), (256, 512, 5), (512, 256, 16), (32, 256, 3),
                                   (2560, 256, 8), (256, 2560, 8), (1280, 96, 13)])
def test_q41_gemm_matches_oracle(torch_cuda, K, N, M):
    rng = np.random.default_rng(K * 7 + N + M)
    W = gen.pack_q41((rng.standard_normal((N, K)) * 0.02).astype(np.float32))
    x = gen.bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    y, _ = _gemm(torch_cuda, W, x, K, N)
    ref = oracle.linear_q41(oracle.bf16_decode(x), W).astype(np.float64)
    assert np.all(np.abs(y - ref) <= _bound(x, W))


def test_q41_gemm_one_hot_exact(torch_cuda):
    """x = e_k returns the dequantised weight row k exactly (d*q*1 + m*1 has no rounding)."""
    K, N = 512, 256
    rng = np.random.default_rng(1)
    W = gen.pack_q41((rng.standard_normal((N, K)) * 0.02).astype(np.float32))
    ks = [0, 1, 31, 32, 63, 64, 200, 511, 7, 100, 300, 450, 17, 33, 65, 255]
    x = np.zeros((16, K), np.float32)
    for m, k in enumerate(ks):
        x[m, k] = 1.0
    y, _ = _gemm(torch_cuda, W, gen.bf16_bits(x), K, N)
    deq = oracle.q41_dequant(W).reshape(N, K)
    for m, k in enumerate(ks):
        np.testing.assert_array_equal(y[m], deq[:, k].astype(np.float32))


def test_q41_gemm_rows_independent_of_batch(torch_cuda):
    """Row m of an M-row product equals the same row computed alone, bit for bit (M = 1..16)."""
    K, N = 2560, 512
    rng = np.random.default_rng(2)
    W = gen.pack_q41((rng.standard_normal((N, K)) * 0.02).astype(np.float32))
    x = gen.bf16_bits(rng.standard_normal((16, K)).astype(np.float32))
    full, _ = _gemm(torch_cuda, W, x, K, N)
    for M in (1, 2, 4, 8, 11, 16):
        part, _ = _gemm(torch_cuda, W, x[:M], K, N)
        np.testing.assert_array_equal(part, full[:M])


@pytest.mark.parametrize("K,N", [(2560, 10240), (10240, 2560), (2560, 4096), (20480, 2560)])
def test_q41_gemm_full_size_sampled_columns(torch_cuda, K, N):
    """The isolated product sweep's full shapes: sampled output columns against the oracle."""
    rng = np.random.default_rng(K + N)
    W = gen.make_tensor(gen.TensorSpec("sweep", "q41", (N, K), 0.02), seed=5)
    x = gen.bf16_bits(rng.standard_normal((8, K)).astype(np.float32))
    y, _ = _gemm(torch_cuda, W, x, K, N)
    cols = np.unique(np.concatenate([rng.integers(0, N, 48), [0, 15, 16, 31, 32, N - 1]]))
    ref = oracle.linear_q41(oracle.bf16_decode(x), W[cols]).astype(np.float64)
    assert np.all(np.abs(y[:, cols] - ref) <= _bound(x, W[cols]))


# ---------------------------------------------------------------------------------------------------
# the whole step
# ---------------------------------------------------------------------------------------------------
@pytest.fixture(scope="module", params=["tiny", "tiny-shared"])
def pair(request, torch_cuda):
    pc = gen.PAIRS[request.param]()
    return pc, gen.generate(pc)


@pytest.mark.parametrize("p", [0.3, 0.0])
def test_spec_decode_lockstep_greedy(pair, p):
    from gpu_harness import lockstep
    pc, W = pair
    res, plain = lockstep(pc, W, gen.prompt(pc.target.vocab, 32), 32, p=p)
    if res.near_ties == 0:
        assert res.tokens == [int(t) for t in plain.tokens]
    assert res.max_rel_l1 < 1e-4          # far inside the 1e-3 bar: no cascade of rounding differences


def test_spec_decode_lockstep_sampled(pair):
    """Sampled verify: every target token equals the oracle's draw (a differing draw is allowed only when
    u * sum(p) lies within 1e-5 * sum(p) of an interval edge, asserted in the harness)."""
    from gpu_harness import lockstep
    pc, W = pair
    res, plain = lockstep(pc, W, gen.prompt(pc.target.vocab, 32), 32, p=0.3, temperature=0.8, seed=3)
    if res.near_ties == 0:
        assert res.tokens == [int(t) for t in plain.tokens]


@pytest.mark.parametrize("temperature,cluster", [(None, 16), (0.8, 16), (None, 8), (None, 4)])
def test_spec_decode_long_context(pair, temperature, cluster):
    """A 2000-token prompt: the sliding rings wrap many times over, full layers read dozens of key
    blocks, and the draft catches up on the whole context. Lockstep with the oracle as above, with
    attention clusters of up to 16, 8 and 4 CTAs."""
    import dataclasses
    from dflash_speculative_decode_gb300._abi import DFL_OPT_ATTN_CLUSTER
    from gpu_harness import engine, lockstep
    pc, W = pair
    pc = dataclasses.replace(pc, max_ctx=2304)
    eng = engine(pc, W)
    eng.dfl_set_option(DFL_OPT_ATTN_CLUSTER, cluster)
    res, plain = lockstep(pc, W, gen.prompt(pc.target.vocab, 2000, request=7), 24, p=0.3,
                          temperature=temperature, seed=11, eng=eng)
    if res.near_ties == 0:
        assert res.tokens == [int(t) for t in plain.tokens]
    assert res.max_rel_l1 < 1e-3


def test_gpu_batched_equals_sequential(pair):
    """k rows in one pass give bit-identical logits to k one-row passes on the GPU."""
    from dflash_speculative_decode_gb300 import DFL_OPT_KEEP_LOGITS
    from gpu_harness import engine
    pc, W = pair
    prompt = gen.prompt(pc.target.vocab, 20)
    rows = [int(t) for t in gen.prompt(pc.target.vocab, 8, request=5)]
    a = engine(pc, W)
    a.dfl_set_option(DFL_OPT_KEEP_LOGITS, 1)
    a.dfl_prefill(prompt)
    a.dfl_verify_block(rows)
    la = a.dfl_read_logits(0, 8)
    a.dfl_commit_verify_rows(8)
    b = engine(pc, W)
    b.dfl_set_option(DFL_OPT_KEEP_LOGITS, 1)
    b.dfl_prefill(prompt)
    lb = []
    for r in rows:
        b.dfl_verify_block([r])
        lb.append(b.dfl_read_logits(0, 1)[0])
        b.dfl_commit_verify_rows(1)
    np.testing.assert_array_equal(la, np.stack(lb))
    sa, sb = a.dfl_snapshot(), b.dfl_snapshot()
    assert (sa.cpu().numpy() == sb.cpu().numpy()).all()


def test_gpu_rollback_equals_forward_over_accepted_rows(pair):
    from dflash_speculative_decode_gb300 import DFL_OPT_KEEP_LOGITS
    from gpu_harness import engine
    pc, W = pair
    prompt = gen.prompt(pc.target.vocab, 20)
    rows = [int(t) for t in gen.prompt(pc.target.vocab, 8, request=6)]
    nxt = [int(t) for t in gen.prompt(pc.target.vocab, 4, request=7)]
    a = engine(pc, W)
    a.dfl_set_option(DFL_OPT_KEEP_LOGITS, 1)
    a.dfl_prefill(prompt)
    a.dfl_verify_block(rows)
    a.dfl_commit_verify_rows(3)
    assert a.dfl_positions_held() == 23
    a.dfl_verify_block(nxt)
    la = a.dfl_read_logits(0, 4)
    b = engine(pc, W)
    b.dfl_set_option(DFL_OPT_KEEP_LOGITS, 1)
    b.dfl_prefill(prompt)
    b.dfl_verify_block(rows[:3])
    b.dfl_commit_verify_rows(3)
    b.dfl_verify_block(nxt)
    np.testing.assert_array_equal(la, b.dfl_read_logits(0, 4))


def test_gpu_kv_widths_and_commit_arithmetic(pair):
    from dflash_speculative_decode_gb300 import DflError
    from gpu_harness import engine
    pc, W = pair
    eng = engine(pc, W)
    assert list(eng.dfl_kv_widths()) == oracle.kv_widths(pc.target)
    eng.dfl_prefill(gen.prompt(pc.target.vocab, 3))
    assert eng.dfl_positions_held() == 3
    eng.dfl_verify_block([1, 2, 3, 4])
    assert eng.dfl_positions_held() == 3
    with pytest.raises(DflError):
        eng.dfl_verify_block([1])              # pending
    with pytest.raises(DflError):
        eng.dfl_snapshot()                     # pending
    with pytest.raises(DflError):
        eng.dfl_commit_verify_rows(5)          # keep > k
    assert eng.dfl_positions_held() == 3
    eng.dfl_commit_verify_rows(2)
    assert eng.dfl_positions_held() == 5
    with pytest.raises(DflError):
        eng.dfl_commit_verify_rows(1)          # nothing pending
    with pytest.raises(DflError):
        eng.dfl_verify_block([pc.target.vocab])  # token out of range
    with pytest.raises(DflError):
        eng.dfl_verify_block(list(range(17)))  # k > 16
    assert eng.dfl_positions_held() == 5


def test_gpu_snapshot_restore_replays(pair):
    """Snapshot after a prefix; decode; restore; the same decode gives the same tokens and logits."""
    from dflash_speculative_decode_gb300 import DFL_OPT_KEEP_LOGITS, spec_decode
    from gpu_harness import engine
    pc, W = pair
    eng = engine(pc, W)
    eng.dfl_set_option(DFL_OPT_KEEP_LOGITS, 1)
    t0 = eng.dfl_prefill(gen.prompt(pc.target.vocab, 24))
    snap = eng.dfl_snapshot()
    assert snap.numel() == eng.dfl_snapshot_bytes()
    runs = []
    for _ in range(2):
        eng.dfl_restore(snap)
        assert eng.dfl_positions_held() == 24
        toks = [t0]
        for _ in range(4):
            dp = eng.dfl_draft_block(toks[-1])
            tt, a = eng.dfl_verify_block([toks[-1]] + list(map(int, dp)))
            eng.dfl_commit_verify_rows(a + 1)
            toks += list(map(int, dp[:a])) + [int(tt[a])]
        runs.append((toks, eng.dfl_read_logits(0, pc.draft.block)))
    assert runs[0][0] == runs[1][0]
    np.testing.assert_array_equal(runs[0][1], runs[1][1])


def test_gpu_shared_layers_have_no_plane():
    """tiny-shared: KV-shared layers report width 0 and the snapshot holds only owner planes."""
    from gpu_harness import engine
    pc = gen.tiny_shared_pair()
    W = gen.generate(pc)
    eng = engine(pc, W)
    w = list(eng.dfl_kv_widths())
    assert w[4] == 0 and w[5] == 0 and w[2] == 256 and w[3] == 128
    eng.dfl_prefill(gen.prompt(pc.target.vocab, 10))
    b10 = eng.dfl_snapshot_bytes()
    eng.dfl_verify_block([1, 2])
    eng.dfl_commit_verify_rows(2)
    b12 = eng.dfl_snapshot_bytes()
    # per new position: the full owner layer's K and V (2 heads x 64 floats) plus, until the next draft
    # block makes them context, the position's taps (3 taps x 256 floats); sliding planes are rings of
    # fixed size and shared layers hold nothing
    assert b12 - b10 == 2 * (2 * 2 * 64 * 4) + 2 * (3 * 256 * 4)


def test_bounded_wait_timeout_reports_and_recovers():
    """The error path of the bounded waits, without a fault: with DFL_OPT_TEST_STALL the products' copy
    warps issue nothing, the first product's waits give up after about a second, later products of the
    pass skip their copies, and the verify returns DFL_E_TIMEOUT with positions held unchanged. With the
    option off again the same verify gives the logits of a context that never failed."""
    from dflash_speculative_decode_gb300 import DFL_OPT_KEEP_LOGITS, DflError
    from dflash_speculative_decode_gb300._abi import DFL_E_TIMEOUT, DFL_OPT_TEST_STALL
    from gpu_harness import engine
    pc = gen.tiny_pair()
    W = gen.generate(pc)
    prompt = gen.prompt(pc.target.vocab, 20)
    rows = [int(t) for t in gen.prompt(pc.target.vocab, 8, request=6)]
    a = engine(pc, W)
    a.dfl_set_option(DFL_OPT_KEEP_LOGITS, 1)
    a.dfl_prefill(prompt)
    a.dfl_set_option(DFL_OPT_TEST_STALL, 1)
    with pytest.raises(DflError) as ei:
        a.dfl_verify_block(rows)
    assert ei.value.code == DFL_E_TIMEOUT
    assert a.dfl_positions_held() == 20
    with pytest.raises(DflError):
        a.dfl_commit_verify_rows(1)            # nothing is pending after the failed verify
    a.dfl_set_option(DFL_OPT_TEST_STALL, 0)
    tt_a, acc_a = a.dfl_verify_block(rows)
    la = a.dfl_read_logits(0, 8)
    b = engine(pc, W)
    b.dfl_set_option(DFL_OPT_KEEP_LOGITS, 1)
    b.dfl_prefill(prompt)
    tt_b, acc_b = b.dfl_verify_block(rows)
    np.testing.assert_array_equal(la, b.dfl_read_logits(0, 8))
    assert list(tt_a) == list(tt_b) and acc_a == acc_b
    # the draft's context after a failed draft block is rebuilt: proposals as on the clean context
    a.dfl_commit_verify_rows(3)
    b.dfl_commit_verify_rows(3)
    a.dfl_set_option(DFL_OPT_TEST_STALL, 1)
    with pytest.raises(DflError) as ei:
        a.dfl_draft_block(int(tt_a[2]))
    assert ei.value.code == DFL_E_TIMEOUT
    a.dfl_set_option(DFL_OPT_TEST_STALL, 0)
    assert list(a.dfl_draft_block(int(tt_a[2]))) == list(b.dfl_draft_block(int(tt_b[2])))


def test_standalone_product_status(torch_cuda):
    """dfl_q41_gemm_status reads the scratch's error word: DFL_OK after products that completed."""
    from dflash_speculative_decode_gb300 import _abi
    K, N = 256, 384
    rng = np.random.default_rng(3)
    W = gen.pack_q41((rng.standard_normal((N, K)) * 0.02).astype(np.float32))
    x = gen.bf16_bits(rng.standard_normal((4, K)).astype(np.float32))
    _, (img, scratch) = _gemm(torch_cuda, W, x, K, N)
    st = ctypes.c_void_p(torch_cuda.cuda.current_stream().cuda_stream)
    assert _abi.lib().dfl_q41_gemm_status(ctypes.c_void_p(scratch.data_ptr()), st) == _abi.DFL_OK


@pytest.mark.parametrize("K,N,M", [(256, 2048, 7), (2560, 4096, 8), (512, 1024, 16), (2560, 262144, 8)])
def test_bf16_head_argmax_matches_oracle(torch_cuda, K, N, M):
    """The standalone head: logits within the fp32 bound of the exact products, and the first-maximum
    argmax equal to the oracle's (or at a near-tie of the oracle's logits)."""
    from dflash_speculative_decode_gb300 import _abi
    from gpu_harness import NEAR_TIE
    torch = torch_cuda
    L = _abi.lib()
    rng = np.random.default_rng(K + N + M)
    Wb = gen.bf16_bits((rng.standard_normal((N, K)) * (2.0 / K ** 0.5)).astype(np.float32))
    x = gen.bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    dev = torch.device("cuda:0")
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    src = torch.from_numpy(Wb.reshape(-1).view(np.int16)).to(dev)
    img = torch.empty(L.dfl_bf16_image_bytes(K, N), dtype=torch.uint8, device=dev)
    assert L.dfl_bf16_pack(ctypes.c_void_p(src.data_ptr()), K, N, ctypes.c_void_p(img.data_ptr()), st) == 0
    xf = torch.from_numpy(oracle.bf16_decode(x)).to(dev)
    act = torch.empty(L.dfl_act_bytes(M, K), dtype=torch.uint8, device=dev)
    assert L.dfl_act_pack(ctypes.c_void_p(xf.data_ptr()), M, K, ctypes.c_void_p(act.data_ptr()), st) == 0
    sb = L.dfl_bf16_head_scratch_bytes(K, N, M)
    scratch = torch.zeros(sb, dtype=torch.uint8, device=dev)
    am = torch.full((M,), -1, dtype=torch.int32, device=dev)
    lg = torch.empty((M, N), dtype=torch.float32, device=dev)
    for _ in range(2):   # the scratch is reusable
        assert L.dfl_bf16_head_argmax(ctypes.c_void_p(img.data_ptr()), K, N, ctypes.c_void_p(act.data_ptr()), M,
                                      ctypes.c_void_p(am.data_ptr()), ctypes.c_void_p(lg.data_ptr()),
                                      ctypes.c_void_p(scratch.data_ptr()), sb, st) == 0
    torch.cuda.synchronize()
    ref = oracle.linear_bf16(oracle.bf16_decode(x), Wb).astype(np.float64)
    absdot = oracle.linear_bf16(np.abs(oracle.bf16_decode(x)), Wb & np.uint16(0x7FFF)).astype(np.float64)
    bound = absdot * (K + 64) * 2.0 ** -24 + 1e-6
    got = lg.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= bound)
    for m, i in enumerate(am.cpu().numpy()):
        j = int(np.argmax(ref[m]))
        assert i == j or ref[m, j] - ref[m, i] < NEAR_TIE


def test_spec_decode_lockstep_fused_steps(pair):
    """The same lockstep with the row and q/k steps run on the products' last CTAs (DFL_OPT_FUSE_STEPS)."""
    from dflash_speculative_decode_gb300._abi import DFL_OPT_FUSE_STEPS
    from gpu_harness import engine, lockstep
    pc, W = pair
    eng = engine(pc, W)
    eng.dfl_set_option(DFL_OPT_FUSE_STEPS, 1)
    res, plain = lockstep(pc, W, gen.prompt(pc.target.vocab, 32), 32, p=0.3, eng=eng)
    if res.near_ties == 0:
        assert res.tokens == [int(t) for t in plain.tokens]
    assert res.max_rel_l1 < 1e-4


def test_ple_split_and_one_launch():
    """The per-layer-embedding tail as one cluster launch (default) and as two products
    (DFL_OPT_PLE_SPLIT): both in lockstep with the oracle, and their verify logits within the logit
    tolerance of each other; 16-row passes take the one-launch path too (a 20-row prefill)."""
    from dflash_speculative_decode_gb300 import DFL_OPT_KEEP_LOGITS
    from dflash_speculative_decode_gb300._abi import DFL_OPT_PLE_SPLIT
    from gpu_harness import check_logits, engine, lockstep
    pc = gen.tiny_shared_pair()
    W = gen.generate(pc)
    eng = engine(pc, W)
    eng.dfl_set_option(DFL_OPT_PLE_SPLIT, 1)
    res, plain = lockstep(pc, W, gen.prompt(pc.target.vocab, 20), 24, p=0.3, eng=eng)
    if res.near_ties == 0:
        assert res.tokens == [int(t) for t in plain.tokens]
    prompt = gen.prompt(pc.target.vocab, 20, request=4)
    rows = [int(v) for v in gen.prompt(pc.target.vocab, 8, request=5)]
    out = []
    for split in (0, 1):
        e = engine(pc, W)
        e.dfl_set_option(DFL_OPT_KEEP_LOGITS, 1)
        e.dfl_set_option(DFL_OPT_PLE_SPLIT, split)
        t = e.dfl_prefill(prompt)
        e.dfl_verify_block([t] + rows[1:])
        out.append((t, e.dfl_read_logits(0, 8)))
    check_logits(out[0][1], out[1][1], "one launch vs two products")


def test_single_turn_serving_matches_oracle():
    """Single-turn serving on tiny-shared (KV-shared layers with empty planes, PLE, two KV widths): a
    prefix cache of two slots, requests P1:A, P2:B, P1:A, P1:B with a stop token, each against the
    oracle restoring the same pinned prefix; positions held exclude the stop token's row."""
    from dflash_speculative_decode_gb300 import PrefixCache, serve_single_turn
    from gpu_harness import engine
    pc = gen.tiny_shared_pair()
    W = gen.generate(pc)
    V = pc.target.vocab
    pre = {1: list(gen.prompt(V, 24, request=30)), 2: list(gen.prompt(V, 40, request=33))}
    req = {"A": list(gen.prompt(V, 12, request=31)), "B": list(gen.prompt(V, 12, request=32))}
    eng = engine(pc, W)
    cache = PrefixCache(eng, slots=2)
    pairs = {}
    for p in pre:
        pair = oracle.Pair(pc, W)
        pair.prefill(pre[p], oracle.Sampler())
        pairs[p] = (pair, pair.snapshot())
    full = oracle.serve_single_turn(pairs[1][0], pairs[1][1], req["B"], 20, oracle.Sampler()).tokens
    stop = int(full[7])
    seen = {}
    for p, name, st in ((1, "A", None), (2, "B", None), (1, "A", None), (1, "B", stop)):
        got = serve_single_turn(eng, cache, pre[p], req[name], 20, stop_token=st)
        ref = oracle.serve_single_turn(pairs[p][0], pairs[p][1], req[name], 20, oracle.Sampler(), stop=st)
        assert got.tokens == [int(t) for t in ref.tokens], (p, name)
        assert eng.dfl_positions_held() == pairs[p][0].target.n
        seen.setdefault((p, name), got.tokens)
        assert got.tokens == seen[(p, name)]
    assert len(got.tokens) == [int(t) for t in full].index(stop) + 1


@pytest.mark.parametrize("temperature", [None, 0.8])
def test_pinned_prefix_requests_a_b_a_lockstep(temperature):
    """tiny-shared (shared layers' planes empty, window 16 so the rings wrap within the prefix): the prefix
    snapshot restored on both sides before each of requests A, B, A, then every pass of the request in
    lockstep with the oracle (draft and verify logits, tokens, accepted lengths, positions held)."""
    from gpu_harness import engine, lockstep
    pc = gen.tiny_shared_pair()
    W = gen.generate(pc)
    V = pc.target.vocab
    prefix = gen.prompt(V, 48, request=40)
    eng = engine(pc, W)
    eng.dfl_prefill(prefix)
    snap_g = eng.dfl_snapshot()
    op = oracle.Pair(pc, W)
    op.prefill(prefix, oracle.Sampler())
    op.sync_draft()
    snap_o = op.snapshot()
    req = {"A": gen.prompt(V, 12, request=41), "B": gen.prompt(V, 12, request=42)}
    out = []
    for name in "ABA":
        eng.dfl_restore(snap_g)
        op.restore(snap_o)
        res, plain = lockstep(pc, W, req[name], 20, p=0.3, temperature=temperature, seed=9, eng=eng, op=op)
        if res.near_ties == 0:
            assert res.tokens == [int(t) for t in plain.tokens]
        out.append(res.tokens)
    assert out[0] == out[2]
