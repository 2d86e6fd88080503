"""GPU parity at the E4B pair's full shapes (42 target layers with KV sharing, PLE and double-wide MLPs;
5-layer draft; vocab 262144) against the oracle, at a context short enough for the oracle."""
import os

import numpy as np
import pytest

import gen
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def e4b():
    import torch
    assert torch.cuda.is_available()
    from dflash_speculative_decode_gb300 import DFL_OPT_KEEP_LOGITS, Engine, build, config_from_pair
    build.build()
    pc = gen.e4b_pair(max_ctx=256)
    W = gen.generate(pc, workers=min(16, os.cpu_count() or 1))
    eng = Engine(config_from_pair(pc))
    eng.load(W)
    eng.dfl_set_option(DFL_OPT_KEEP_LOGITS, 1)
    return pc, W, eng


def test_e4b_draft_and_verify_logits(e4b):
    from gpu_harness import NEAR_TIE, check_logits
    pc, W, eng = e4b
    prompt = gen.prompt(pc.target.vocab, 6)
    pair = oracle.Pair(pc, W)
    t_o, _ = pair.prefill(prompt, oracle.Sampler())
    t_g = eng.dfl_prefill(prompt)
    assert t_g == t_o
    pair.sync_draft()
    dp_o, dl_o = pair.draft.block(t_o, W["emb"], W["head"])
    dp_g = eng.dfl_draft_block(t_g)
    check_logits(eng.dfl_read_logits(1, 7), dl_o, "E4B draft logits")
    for i in range(7):
        assert dp_g[i] == dp_o[i] or oracle.model.top2_gap(dl_o[i]) < NEAR_TIE
    rows = [t_o] + [int(v) for v in gen.prompt(pc.target.vocab, 7, request=9)]
    tt_o, cl, lg_o = pair.verify(rows, oracle.Sampler())
    tt_g, a_g = eng.dfl_verify_block(rows)
    r, m = check_logits(eng.dfl_read_logits(0, 8), lg_o, "E4B verify logits")
    for i in range(8):
        assert tt_g[i] == tt_o[i] or cl[i] < NEAR_TIE
    assert a_g == oracle.accept_length(rows[1:], tt_o[:-1])
    assert list(eng.dfl_kv_widths()) == oracle.kv_widths(pc.target)
    print(f"E4B verify logits rel-L1 {r:.3g} max-abs {m:.3g}")


def test_e4b_commit_and_next_pass(e4b):
    """After a partial accept, the next verify equals a fresh context that saw only the kept rows."""
    from gpu_harness import check_logits
    pc, W, eng = e4b
    eng.dfl_commit_verify_rows(3)
    nxt = [int(v) for v in gen.prompt(pc.target.vocab, 8, request=10)]
    eng.dfl_verify_block(nxt)
    la = eng.dfl_read_logits(0, 8)
    held = eng.dfl_positions_held()
    assert held == 6 + 3
    prompt = gen.prompt(pc.target.vocab, 6)
    pair2 = oracle.Pair(pc, W, with_draft=False)
    t_first, _ = pair2.prefill(prompt, oracle.Sampler())
    kept = [t_first] + [int(v) for v in gen.prompt(pc.target.vocab, 7, request=9)][:2]
    pair2.target.forward(kept)
    pair2.target.commit(3)
    lb = pair2.target.forward(nxt)
    check_logits(la, lb, "E4B next pass after commit(3)")


def test_e4b_draft_alone_contexts(e4b):
    """The E4B draft on its own (5 layers, 32/8 heads of 128, window 1024, shared head of 262144)
    over context rows made from N(0, 1) taps, at contexts of 30, 1024 and 4096 rows (the last wraps the
    1024-slot context ring four times): draft logits and proposals against the oracle's draft."""
    import torch
    from gpu_harness import NEAR_TIE, check_logits
    from dflash_speculative_decode_gb300 import DFL_OPT_KEEP_LOGITS, Engine, config_from_pair
    import dataclasses
    pc0, W, _ = e4b
    pc = dataclasses.replace(pc0, max_ctx=4096 + 64)
    eng = Engine(config_from_pair(pc))
    eng.load(W)
    eng.dfl_set_option(DFL_OPT_KEEP_LOGITS, 1)
    taps = gen.fc_taps(4096, len(pc.draft.taps) * pc.target.hidden)
    d = oracle.Draft(pc.draft, W, pc.target)
    have = 0
    for ctx, tok in ((30, 17), (1024, 4242), (4096, 262000)):
        eng.dfl_draft_append_taps(torch.from_numpy(taps[have:ctx]).cuda())
        d.append_ctx(taps[have:ctx])
        have = ctx
        assert eng.dfl_positions_held() == ctx == d.n_ctx
        dp_g = eng.dfl_draft_block(tok)
        dp_o, dl_o = d.block(tok, W["emb"], W["head"])
        r, m = check_logits(eng.dfl_read_logits(1, 7), dl_o, f"draft alone at context {ctx}")
        for i in range(7):
            assert dp_g[i] == dp_o[i] or oracle.model.top2_gap(dl_o[i]) < NEAR_TIE
        print(f"draft alone, context {ctx}: rel-L1 {r:.3g}, max-abs {m:.3g}")
    eng.close()
