"""Oracle properties the pages state for the whole step (1bit engine PR "Gemma4 verifies a draft in one
batched pass", "Proof"; model card "Nemotron-3.5-Bolt-E4B-DFlash-NPU2", "How it is used"), with the
mutants that must fail them. CPU only."""
import numpy as np
import pytest

import gen
import oracle
from oracle import model as om


@pytest.fixture(scope="module", params=["tiny", "tiny-shared"])
def pair_w(request):
    pc = gen.PAIRS[request.param]()
    return pc, gen.generate(pc)


def _prefilled(pc, W, P=20, mutant=None):
    pair = oracle.Pair(pc, W, width_mutant=mutant)
    pair.prefill(gen.prompt(pc.target.vocab, P), oracle.Sampler())
    return pair


def test_batched_equals_sequential(pair_w):
    """P3: k rows in one layer-by-layer pass give bit-identical logits and planes to k one-row passes."""
    pc, W = pair_w
    rows = [int(t) for t in gen.prompt(pc.target.vocab, 6, request=5)]
    a = _prefilled(pc, W)
    la = a.target.forward(rows)
    a.target.commit(len(rows))
    b = _prefilled(pc, W)
    lb = []
    for r in rows:
        lb.append(b.target.forward([r])[0])
        b.target.commit(1)
    np.testing.assert_array_equal(la, np.stack(lb))
    for l in a.target.planes:
        np.testing.assert_array_equal(a.target.planes[l], b.target.planes[l])
    np.testing.assert_array_equal(a.target.taps, b.target.taps)


def test_rollback_equals_forward_over_accepted_rows(pair_w):
    """P5: after a verify of 8 rows and commit(3), the next pass equals a pair that only ever saw the
    3 accepted rows."""
    pc, W = pair_w
    rows = [int(t) for t in gen.prompt(pc.target.vocab, 8, request=6)]
    nxt = [int(t) for t in gen.prompt(pc.target.vocab, 4, request=7)]
    a = _prefilled(pc, W)
    a.target.forward(rows)
    a.target.commit(3)
    assert a.target.positions_held() == 23
    la = a.target.forward(nxt)
    b = _prefilled(pc, W)
    b.target.forward(rows[:3])
    b.target.commit(3)
    lb = b.target.forward(nxt)
    np.testing.assert_array_equal(la, lb)


def test_width_mutant_fails_rollback():
    """The pages' mutant (one KV width for every layer) must break rollback on a two-width model."""
    pc = gen.tiny_shared_pair()
    W = gen.generate(pc)
    rows = [int(t) for t in gen.prompt(pc.target.vocab, 8, request=6)]
    b = _prefilled(pc, W)
    b.target.forward(rows[:3])
    b.target.commit(3)
    a2 = _prefilled(pc, W, mutant=128)             # the sliding width; full layers are 256 wide
    a2.target.forward(rows)
    a2.target.commit(3)
    # the count agrees with itself, but the full layer's plane kept only half of its positions
    assert a2.target.positions_held() == 23
    assert len(a2.target.planes[2]) // 256 < 23
    assert not np.array_equal(a2.target.forward([5])[0], b.target.forward([5])[0])


def test_shared_planes_stay_empty():
    """P6: KV-shared layers hold no plane through verify, rollback, snapshot and restore; the held count
    ignores them; owners grow by exactly their width per row."""
    pc = gen.tiny_shared_pair()
    W = gen.generate(pc)
    pair = _prefilled(pc, W, P=10)
    tg = pair.target
    shared = [l for l in range(pc.target.n_layers) if not pc.target.is_owner(l)]
    assert shared == [4, 5]
    widths = oracle.kv_widths(pc.target)
    assert [widths[l] for l in shared] == [0, 0]
    snap = pair.snapshot()
    tg.forward([1, 2, 3, 4, 5])
    for l in tg.planes:
        assert len(tg.planes[l]) == 15 * widths[l]
    tg.commit(2)
    assert all(tg.plane(l) is None for l in shared) and tg.positions_held() == 12
    pair.restore(snap)
    assert all(tg.plane(l) is None for l in shared) and tg.positions_held() == 10


def test_shared_layer_reads_owner_plane():
    """Changing the owner's stored keys changes a shared layer's output; the shared layer appends none."""
    pc = gen.tiny_shared_pair()
    W = gen.generate(pc)
    a = _prefilled(pc, W, P=10)
    b = _prefilled(pc, W, P=10)
    b.target.planes[3] = b.target.planes[3] * np.float32(0.5)     # layer 4 reads layer 3's plane
    assert not np.array_equal(a.target.forward([7])[0], b.target.forward([7])[0])


def test_snapshot_restore_replays_identically(pair_w):
    pc, W = pair_w
    pair = _prefilled(pc, W)
    s = pair.snapshot()
    l1 = pair.target.forward([3, 4, 5])
    pair.target.commit(3)
    pair.sync_draft()
    pair.restore(s)
    assert pair.target.positions_held() == 20 and pair.draft.n_ctx == 20
    l2 = pair.target.forward([3, 4, 5])
    np.testing.assert_array_equal(l1, l2)


def _greedy_stream(pc, W, prompt, n_gen, sampler):
    run = oracle.plain_decode(oracle.Pair(pc, W), prompt, n_gen, sampler)
    G = np.zeros(pc.max_ctx, np.int32)
    G[len(prompt):len(prompt) + len(run.tokens)] = run.tokens
    return run, G


@pytest.mark.parametrize("p", [0.0, 0.3, 1.0])
def test_greedy_spec_equals_plain(pair_w, p):
    """P7: greedy speculative output is token-identical to plain greedy decode (planted drafts at
    corruption p; p = 0 accepts every proposal)."""
    pc, W = pair_w
    prompt = gen.prompt(pc.target.vocab, 32)
    plain, G = _greedy_stream(pc, W, prompt, 32, oracle.Sampler())
    cor = gen.corruption(p, pc.target.vocab, pc.max_ctx)
    run = oracle.spec_decode(oracle.Pair(pc, W), prompt, 32, oracle.Sampler(),
                             propose=lambda n, dp: cor.propose(G, np.arange(n + 1, n + 8)))
    assert [int(t) for t in run.tokens] == [int(t) for t in plain.tokens]
    if p == 0.0:
        assert all(s.accepted == 7 for s in run.steps[:-1])
    for s in run.steps[:-1]:
        assert len(s.emitted) == s.accepted + 1


def test_greedy_spec_with_draft_proposals_equals_plain(pair_w):
    pc, W = pair_w
    prompt = gen.prompt(pc.target.vocab, 32)
    plain, _ = _greedy_stream(pc, W, prompt, 24, oracle.Sampler())
    run = oracle.spec_decode(oracle.Pair(pc, W), prompt, 24, oracle.Sampler())
    assert [int(t) for t in run.tokens] == [int(t) for t in plain.tokens]


def test_sampled_spec_equals_plain_sampled(pair_w):
    """With per-position uniforms the sampled speculative output equals plain sampled decode."""
    pc, W = pair_w
    prompt = gen.prompt(pc.target.vocab, 32)
    s = oracle.Sampler(0.8, 3)
    plain, G = _greedy_stream(pc, W, prompt, 32, s)
    cor = gen.corruption(0.3, pc.target.vocab, pc.max_ctx)
    run = oracle.spec_decode(oracle.Pair(pc, W), prompt, 32, s,
                             propose=lambda n, dp: cor.propose(G, np.arange(n + 1, n + 8)))
    assert [int(t) for t in run.tokens] == [int(t) for t in plain.tokens]
    assert sum(st.accepted for st in run.steps) > 0


def test_draft_context_window_and_bidirectional_block():
    """The draft's block sees only the context rows inside its window (relative to the block start)."""
    pc = gen.tiny_shared_pair()            # draft window 24
    W = gen.generate(pc)
    pair = _prefilled(pc, W, P=40)
    d = pair.draft
    _, l0 = d.block(5, W["emb"], W["head"])
    snap = d.snapshot()
    d.ctx_k = [a.copy() for a in d.ctx_k]
    d.ctx_v = [a.copy() for a in d.ctx_v]
    for a in d.ctx_k + d.ctx_v:
        a[: 40 - 24] = 0.0                 # outside the window: no effect
    _, l1 = d.block(5, W["emb"], W["head"])
    np.testing.assert_array_equal(l0, l1)
    for a in d.ctx_v:
        a[40 - 24] = 0.0                   # first key inside the window: effect
    _, l2 = d.block(5, W["emb"], W["head"])
    assert not np.array_equal(l0, l2)
    d.restore(snap)
