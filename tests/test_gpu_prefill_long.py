"""Long prefill passes (prefill_rows > 0: up to that many prompt rows per pass, products on the tcgen05
tensor cores, attention in tiles of 16 rows) against the oracle: the first token after the prompt, and
then speculative decode pass by pass, whose draft and verify logits see the planes and taps the long
pass wrote."""
import os

import numpy as np
import pytest

import gen

pytestmark = pytest.mark.gpu


def _engine(pc, W, prefill_rows):
    from dflash_speculative_decode_gb300 import Engine, build, config_from_pair
    build.build()
    eng = Engine(config_from_pair(pc, prefill_rows=prefill_rows))
    eng.load(W)
    return eng


@pytest.fixture(scope="module", params=["tiny", "tiny-shared"])
def pair(request):
    import torch
    assert torch.cuda.is_available()
    pc = gen.PAIRS[request.param]()
    return pc, gen.generate(pc)


@pytest.mark.parametrize("prefill_rows,plen", [(128, 200), (256, 230), (128, 128)])
def test_long_prefill_lockstep(pair, prefill_rows, plen):
    """One long pass (then chunks of 16 for the rest), greedy speculative decode after it."""
    from gpu_harness import lockstep
    pc, W = pair
    eng = _engine(pc, W, prefill_rows)
    res, plain = lockstep(pc, W, gen.prompt(pc.target.vocab, plen, request=plen), 16, p=0.3, eng=eng)
    if res.near_ties == 0:
        assert res.tokens == [int(t) for t in plain.tokens]
    assert res.max_rel_l1 < 1e-3


def test_long_prefill_sampled(pair):
    from gpu_harness import lockstep
    pc, W = pair
    eng = _engine(pc, W, 128)
    res, plain = lockstep(pc, W, gen.prompt(pc.target.vocab, 150, request=3), 12, p=0.3, temperature=0.8,
                          seed=7, eng=eng)
    if res.near_ties == 0:
        assert res.tokens == [int(t) for t in plain.tokens]


def test_long_prefill_matches_chunked_prefill(pair):
    """The same prompt through long passes and through 16-row passes: the same next token (up to a
    near-tie) and verify logits within the logit tolerance of each other."""
    from gpu_harness import check_logits
    from dflash_speculative_decode_gb300 import DFL_OPT_KEEP_LOGITS
    pc, W = pair
    prompt = gen.prompt(pc.target.vocab, 180, request=11)
    rows = [int(v) for v in gen.prompt(pc.target.vocab, 8, request=12)]
    out = []
    for pf in (0, 128):
        eng = _engine(pc, W, pf)
        eng.dfl_set_option(DFL_OPT_KEEP_LOGITS, 1)
        t = eng.dfl_prefill(prompt)
        eng.dfl_verify_block([t] + rows[1:])
        out.append((t, eng.dfl_read_logits(0, 8), eng.dfl_positions_held()))
        eng.close()
    assert out[0][2] == out[1][2] == len(prompt)
    check_logits(out[1][1], out[0][1], "long vs chunked prefill")


@pytest.mark.parametrize("cut", ["e4b", "27b"])
def test_long_prefill_full_shapes(cut):
    """Full per-layer shapes (six E4B layers with PLE; two 27B-class layers): a 260-token prompt in one
    long pass of 256 rows and a chunk of 4, then greedy speculative decode against the oracle."""
    import dataclasses
    import torch
    from gpu_harness import lockstep
    assert torch.cuda.is_available()
    if cut == "e4b":
        t = gen.e4b_target(n_layers=6, first_shared=6, vocab=32768)
        d = dataclasses.replace(gen.e4b_draft(vocab=32768), taps=(1, 3, 5))
        pc = gen.PairConfig(t, d, max_ctx=512)
    else:
        pc = gen.b27_cut(max_ctx=512, n_layers=2)
    W = gen.generate(pc, workers=min(16, os.cpu_count() or 1))
    eng = _engine(pc, W, 256)
    res, plain = lockstep(pc, W, gen.prompt(pc.target.vocab, 260, request=5), 8, p=0.3, eng=eng)
    if res.near_ties == 0:
        assert res.tokens == [int(t) for t in plain.tokens]
    assert res.max_rel_l1 < 1e-3


@pytest.mark.parametrize("temperature", [None, 0.8])
def test_long_passes_after_restored_prefix(pair, temperature):
    """Long passes that start past position 0, as single-turn serving runs them: a 40-token prefix on
    both sides, pinned by snapshot; another request's 150-token prompt over it on the GPU (one long pass
    at position 40); the prefix restored on both sides; then a 300-token prompt in two long passes of
    128 rows (at positions 40 and 168) and 16-row passes for the rest, and speculative decode in
    lockstep with the oracle."""
    import dataclasses
    import oracle
    from gpu_harness import lockstep
    pc0, W = pair
    pc = dataclasses.replace(pc0, max_ctx=512)
    V = pc.target.vocab
    eng = _engine(pc, W, 128)
    op = oracle.Pair(pc, W)
    prefix = gen.prompt(V, 40, request=21)
    eng.dfl_prefill(prefix, temperature, 5)
    op.prefill(prefix, oracle.Sampler(temperature, 5))
    snap_g, snap_o = eng.dfl_snapshot(), op.snapshot()
    eng.dfl_prefill(gen.prompt(V, 150, request=22), temperature, 5)
    assert eng.dfl_positions_held() == 190
    eng.dfl_restore(snap_g)
    op.restore(snap_o)
    res, plain = lockstep(pc, W, gen.prompt(V, 300, request=23), 12, p=0.3, temperature=temperature, seed=5,
                          eng=eng, op=op)
    if res.near_ties == 0:
        assert res.tokens == [int(t) for t in plain.tokens]
    assert res.max_rel_l1 < 1e-3
