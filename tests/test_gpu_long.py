"""GPU parity at long context on an E4B-shaped cut: 12 target layers of the E4B shapes (hidden 2560, 12
query heads of 256, sliding window 512 with one KV head, full layers with two, layers 8-11 KV-shared
(three sliding layers reading layer 7's plane, the full layer 11 reading layer 5's), double-wide MLPs on
the shared layers, PLE 256) and the full 5-layer E4B draft (window 1024), vocabulary cut to 32768 so the
oracle finishes. One prefix of 1100 tokens, prefilled once on each side: the sliding rings (W + 15 = 527
slots) have wrapped twice, the full layers read 35 key blocks spread over clusters of 16 CTAs.

On top of that prefix: greedy speculative decode in lockstep with the oracle; the KV planes and the taps
compared with the oracle's directly; and long-context sampled serving in miniature: sampled decode (T = 0.8) of requests A,
B, A, each after restoring the pinned prefix snapshot on both sides (FastFlowLM PR #899
"gemma4e-dflash-flash", "Changes": a pinned prefix must not be overwritten by a request; the bug showed
on a sequence A, B, A, B, A)."""
import dataclasses
import os

import numpy as np
import pytest

import gen
import oracle

pytestmark = pytest.mark.gpu

PREFIX = 1100


@pytest.fixture(scope="module")
def cut():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from dflash_speculative_decode_gb300 import build
    from gpu_harness import engine
    build.build()
    V = 32768
    t = gen.e4b_target(n_layers=12, first_shared=8, vocab=V)
    d = dataclasses.replace(gen.e4b_draft(vocab=V), taps=(1, 3, 5, 8, 11))
    pc = gen.PairConfig(t, d, max_ctx=PREFIX + 160)
    W = gen.generate(pc, workers=min(16, os.cpu_count() or 1))
    prompt = gen.prompt(V, PREFIX, request=11)
    op = oracle.Pair(pc, W)
    op.prefill(prompt, oracle.Sampler(), chunk=64)
    op.sync_draft()
    eng = engine(pc, W)
    eng.dfl_prefill(prompt)
    return pc, W, op, op.snapshot(), eng, eng.dfl_snapshot()


def _restore(cut):
    pc, W, op, snap_o, eng, snap_g = cut
    op.restore(snap_o)
    eng.dfl_restore(snap_g)
    assert eng.dfl_positions_held() == op.target.n == PREFIX
    return pc, W, op, eng


def test_cut_shapes(cut):
    pc = cut[0]
    w = oracle.kv_widths(pc.target)
    assert w[:8] == [512, 512, 512, 512, 512, 1024, 512, 512] and w[8:] == [0, 0, 0, 0]
    assert pc.target.kv_owner[8:] == (7, 7, 7, 5)
    assert list(cut[4].dfl_kv_widths()) == w


def test_cut_kv_planes_and_taps_direct(cut):
    """Key and value rows of every owner layer, and the taps, against the oracle's after the prefix:
    sliding rows through the ring slot p mod 527, full rows by position."""
    pc, W, op, eng = _restore(cut)
    t = pc.target
    hd = t.head_dim
    cap_s = t.window + 15
    for l in range(t.n_layers):
        if not t.is_owner(l):
            continue
        nkv = t.kv_heads[l]
        full = t.layer_type[l] == gen.FULL
        slots = PREFIX if full else cap_s          # a read may stop short of the plane's end
        Kg = eng.dfl_debug_read(f"k{l}", (slots, nkv * hd), np.float32)
        Vg = eng.dfl_debug_read(f"v{l}", (slots, nkv * hd), np.float32)
        plane = op.target.planes[l].reshape(-1, 2 * nkv * hd)
        positions = [0, 1, 511, 588, 1054, PREFIX - 1] if full else [PREFIX - t.window, 800, 1054, PREFIX - 1]
        for pos in positions:
            s = pos if full else pos % cap_s
            for got, ref, what in ((Kg[s], plane[pos, :nkv * hd], "K"), (Vg[s], plane[pos, nkv * hd:], "V")):
                err = np.abs(got.astype(np.float64) - ref).sum() / np.abs(ref.astype(np.float64)).sum()
                assert err < 1e-4, f"layer {l} {what} position {pos}: rel-L1 {err:.3g}"
    for pos0 in (0, 700, PREFIX - 8):
        got = eng.dfl_read_taps(pos0, 8)
        ref = op.target.taps[pos0:pos0 + 8]
        err = np.abs(got.astype(np.float64) - ref).sum() / np.abs(ref.astype(np.float64)).sum()
        assert err < 1e-4, f"taps at {pos0}: rel-L1 {err:.3g}"


def test_cut_long_context_greedy_lockstep(cut):
    """Greedy speculative decode after the 1100-token prefix (an 8-token request, 24 tokens): draft and
    verify logits, tokens, accepted lengths and positions held against the oracle every pass."""
    from gpu_harness import lockstep
    pc, W, op, eng = _restore(cut)
    res, plain = lockstep(pc, W, gen.prompt(pc.target.vocab, 8, request=12), 24, p=0.3, eng=eng, op=op)
    if res.near_ties == 0:
        assert res.tokens == [int(v) for v in plain.tokens]
    assert res.max_rel_l1 < 1e-3 and res.passes >= 3
    assert min(res.accepted) < 7          # a partial accept (rollback) on every layer width


def test_cut_pinned_prefix_requests_a_b_a_sampled(cut):
    """Long-context sampled serving in miniature: the prefix snapshot restored before each of requests A, B, A; sampled
    verify at T = 0.8 with planted drafts (p = 0.3); every pass against the oracle restored the same
    way. A's two runs give the same tokens."""
    from gpu_harness import lockstep
    pc, W = cut[0], cut[1]
    V = pc.target.vocab
    req = {"A": gen.prompt(V, 24, request=21), "B": gen.prompt(V, 24, request=22)}
    out = []
    for name in ("A", "B", "A"):
        _, _, op, eng = _restore(cut)
        res, plain = lockstep(pc, W, req[name], 16, p=0.3, temperature=0.8, seed=5, eng=eng, op=op)
        if res.near_ties == 0:
            assert res.tokens == [int(v) for v in plain.tokens]
        assert res.max_rel_l1 < 1e-3
        out.append(res.tokens)
    assert out[0] == out[2]
