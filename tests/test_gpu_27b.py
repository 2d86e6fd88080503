"""GPU parity at the 27B-class pair's per-layer shapes (hidden 5376, 32/16 heads of 128, FFN 21504,
window 1024; the 5-layer draft at width 5376 with FFN 10752 and a 5 x 5376 fc) against the oracle, on a
six-layer cut of the target with vocab 32768: greedy and sampled speculative decode at block 8 (seven
proposals verified in one pass), pass by pass."""
import os

import numpy as np
import pytest

import gen
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def b27():
    import torch
    assert torch.cuda.is_available()
    from dflash_speculative_decode_gb300 import build
    build.build()
    pc = gen.b27_cut(max_ctx=256)
    W = gen.generate(pc, workers=min(16, os.cpu_count() or 1))
    return pc, W


def test_27b_shapes_lockstep_greedy(b27):
    from gpu_harness import lockstep
    pc, W = b27
    res, plain = lockstep(pc, W, gen.prompt(pc.target.vocab, 12), 16, p=0.3)
    if res.near_ties == 0:
        assert res.tokens == [int(t) for t in plain.tokens]
    assert res.max_rel_l1 < 1e-3
    print(f"27B-class greedy: {res.passes} passes, accepted {res.accepted}, rel-L1 {res.max_rel_l1:.3g}")


def test_27b_shapes_lockstep_sampled(b27):
    """Sampling at temperature 0.8: target tokens from the same seeded uniform as the oracle's, so the
    emitted tokens follow the target's distribution and match the oracle's draw."""
    from gpu_harness import lockstep
    pc, W = b27
    res, plain = lockstep(pc, W, gen.prompt(pc.target.vocab, 12, request=4), 16, p=0.3, temperature=0.8,
                          seed=5)
    if res.near_ties == 0:
        assert res.tokens == [int(t) for t in plain.tokens]
    assert res.max_rel_l1 < 1e-3


def test_27b_prefill_head_last_row_only(b27):
    """A prefill longer than one chunk (40 rows: chunks of 16, 16, 8): the next token and the last row's
    logits equal the oracle's, and the held context matches a verify of the next rows."""
    from gpu_harness import check_logits, engine
    from dflash_speculative_decode_gb300 import DFL_OPT_KEEP_LOGITS
    pc, W = b27
    prompt = gen.prompt(pc.target.vocab, 40, request=6)
    eng = engine(pc, W)
    eng.dfl_set_option(DFL_OPT_KEEP_LOGITS, 1)
    t_g = eng.dfl_prefill(prompt)
    lg_g = eng.dfl_read_logits(0, 1)
    op = oracle.Pair(pc, W, with_draft=False)
    lg_o = op.target.forward(prompt, head_rows=1)
    op.target.commit(len(prompt))
    t_o, _ = oracle.Sampler().pick(lg_o[-1], op.target.n)
    assert t_g == t_o or oracle.model.top2_gap(lg_o[-1]) < 1e-3
    check_logits(lg_g, lg_o[-1:], "27B-class prefill last-row logits")
    rows = [t_o] + [int(v) for v in gen.prompt(pc.target.vocab, 7, request=8)]
    eng.dfl_verify_block(rows)
    check_logits(eng.dfl_read_logits(0, 8), op.target.forward(rows), "27B-class verify after prefill")
    eng.close()
