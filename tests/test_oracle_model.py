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


def _check_shared_planes_empty(pair):
    """The empty-plane checks: shared layers hold no plane through verify, rollback, snapshot and
    restore; owners grow by exactly their width per row; the held count ignores shared layers."""
    pc = pair.pc
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


def test_shared_planes_stay_empty():
    """P6 on tiny-shared (layers 4 and 5 read the planes of layers 3 and 2)."""
    pc = gen.tiny_shared_pair()
    W = gen.generate(pc)
    _check_shared_planes_empty(_prefilled(pc, W, P=10))


def test_shared_append_mutant_fails_empty_plane_check():
    """A KV-shared layer that appends (its owner's rows, to a plane of its own) must fail P6."""
    pc = gen.tiny_shared_pair()
    W = gen.generate(pc)
    pair = oracle.Pair(pc, W, shared_appends=True)
    pair.prefill(gen.prompt(pc.target.vocab, 10), oracle.Sampler())
    # the logits are those of the correct model: only the bookkeeping differs, so only P6 sees it
    ok = _prefilled(pc, W, P=10)
    np.testing.assert_array_equal(pair.target.forward([7])[0], ok.target.forward([7])[0])
    pair.target.commit(0)
    with pytest.raises(AssertionError):
        _check_shared_planes_empty(pair)


def _rollback_logits(pc, W, P, **opts):
    """(verify 8 rows, commit 3, next 4 rows) on a pair with the given storage options."""
    rows = [int(t) for t in gen.prompt(pc.target.vocab, 8, request=6)]
    nxt = [int(t) for t in gen.prompt(pc.target.vocab, 4, request=7)]
    a = oracle.Pair(pc, W, **opts)
    a.prefill(gen.prompt(pc.target.vocab, P), oracle.Sampler(), chunk=16)   # passes of at most 16 rows
    a.target.forward(rows)
    a.target.commit(3)
    return a.target.forward(nxt)


def test_ring_capacity_reading():
    """P5 with ring storage: a sliding ring of W + 15 slots (what the device arena holds) gives the
    logits of linear storage exactly at a context where the ring has wrapped; a ring of exactly W slots
    fails (the pass overwrites keys its own first rows and the rows kept after the rollback need)."""
    pc = gen.tiny_pair()                       # window 64, passes of up to 16 rows
    W = gen.generate(pc)
    P, Wn = 150, pc.target.window              # 150 + 11 positions: the rings wrap twice
    lin = _rollback_logits(pc, W, P)
    np.testing.assert_array_equal(_rollback_logits(pc, W, P, ring_capacity=Wn + 15), lin)
    bad = _rollback_logits(pc, W, P, ring_capacity=Wn)
    assert np.abs(bad.astype(np.float64) - lin).max() > 1e-3


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


# ---- the draft's context path and block (model card "Nemotron-3.5-Bolt-E4B-DFlash-NPU2", spec table:
# fc fuses the zero-based outputs of the tapped target layers; block of [token, mask, ...]) ----------
def test_taps_are_layer_outputs_in_ascending_order():
    """Tap slice i of a row is the residual stream after target layer taps[i] (PLE and lambda included)."""
    pc = gen.tiny_shared_pair()                # taps (1, 3, 5)
    W = gen.generate(pc)
    tg = om.Target(pc.target, W, tap_layers=pc.draft.taps)
    tg.record = {}
    tg.forward(gen.prompt(pc.target.vocab, 5))
    H = pc.target.hidden
    for i, l in enumerate(pc.draft.taps):
        np.testing.assert_array_equal(tg.taps[:, i * H:(i + 1) * H], tg.record[l]["x"])


def test_fc_orientation_one_nonzero_entry():
    """fc [hidden out][taps*hidden in] with one nonzero entry (output 3, input H + 40): every context
    row is nonzero only at element 3 and follows element 40 of tap 1 alone (a transposed fc or another
    concatenation order would move or lose it)."""
    pc = gen.tiny_shared_pair()
    W = dict(gen.generate(pc))
    H, T = pc.target.hidden, len(pc.draft.taps)
    fc = np.zeros((H, T * H), np.float32)
    fc[3, H + 40] = 1.0
    W["d.fc"] = gen.bf16_bits(fc)
    d = om.Draft(pc.draft, W, pc.target)
    taps = np.random.default_rng(14).standard_normal((4, T * H)).astype(np.float32)
    c = d.context_rows(taps)
    assert (np.count_nonzero(c, axis=1) == 1).all() and (c[:, 3] != 0).all()
    t2 = taps.copy()
    t2[:, 40] *= -3.0                          # element 40 of tap 0: no effect
    t2[:, 2 * H + 40] *= -3.0                  # element 40 of tap 2: no effect
    t2[:, H + 3] *= -3.0                       # element 3 of tap 1: no effect
    np.testing.assert_array_equal(d.context_rows(t2), c)
    t3 = taps.copy()
    t3[:, H + 40] *= -1.0                      # element 40 of tap 1: the sign follows it
    np.testing.assert_array_equal(d.context_rows(t3), -c)


def test_draft_context_keys_rotated_at_their_positions():
    """Context row j's key is rotated at absolute position j: the same taps row made context at
    positions 0 and 1 gives k_1 = rope(k_0, 1) exactly (rope at position 0 is the identity)."""
    pc = gen.tiny_shared_pair()
    W = gen.generate(pc)
    d = om.Draft(pc.draft, W, pc.target)
    row = np.random.default_rng(15).standard_normal((1, len(pc.draft.taps) * pc.target.hidden)).astype(np.float32)
    d.append_ctx(np.concatenate([row, row]))
    hd = pc.draft.head_dim
    for l in range(pc.draft.n_layers):
        for g in range(pc.draft.n_kv_heads):
            k0 = d.ctx_k[l][0, g * hd:(g + 1) * hd]
            np.testing.assert_array_equal(d.ctx_k[l][1, g * hd:(g + 1) * hd], oracle.rope(k0, 1, pc.draft.rope_base))
        np.testing.assert_array_equal(d.ctx_v[l][0], d.ctx_v[l][1])   # values are not rotated


def test_draft_block_is_bidirectional():
    """Row 0 of the block (the last token) sees the mask rows after it: its hidden state changes with
    the mask token. A causal block would leave row 0 unchanged."""
    import dataclasses
    pc = gen.tiny_shared_pair()
    W = gen.generate(pc)
    pair = _prefilled(pc, W, P=30)
    d0 = pair.draft
    d0.block(5, W["emb"], W["head"])
    h0 = d0.last_hidden.copy()
    d1 = om.Draft(dataclasses.replace(pc.draft, mask_token=pc.draft.mask_token - 1), W, pc.target)
    d1.restore(d0.snapshot())
    d1.block(5, W["emb"], W["head"])
    assert np.abs(d1.last_hidden[0].astype(np.float64) - h0[0]).max() > 1e-4


def test_draft_block_rotary_relative_positions():
    """The block's rows sit at positions n..n+B-1 and context keys at their own positions: shifting the
    whole context by 4 positions (with the window hiding the extra rows) leaves the proposals and, up
    to rounding of the rotations, the logits unchanged; rows rotated at fixed positions would not."""
    pc = gen.tiny_shared_pair()                # draft window 24
    W = gen.generate(pc)
    T = np.random.default_rng(16).standard_normal((40, len(pc.draft.taps) * pc.target.hidden)).astype(np.float32)
    a = om.Draft(pc.draft, W, pc.target)
    a.append_ctx(T)
    pa, la = a.block(9, W["emb"], W["head"])
    b = om.Draft(pc.draft, W, pc.target)
    b.append_ctx(np.concatenate([np.zeros((4, T.shape[1]), np.float32), T]))
    pb, lb = b.block(9, W["emb"], W["head"])
    assert list(pa) == list(pb)
    np.testing.assert_allclose(lb, la, rtol=0, atol=2e-4)
    # the same 24 visible rows one position further from the block (a row dropped at the window's far
    # end, a zero row added next to the block) change the logits: relative positions matter
    c = om.Draft(pc.draft, W, pc.target)
    c.append_ctx(np.concatenate([T[:39], np.zeros((1, T.shape[1]), np.float32)]))
    _, lc = c.block(9, W["emb"], W["head"])
    assert np.abs(lc.astype(np.float64) - la).max() > 1e-3


def test_ple_model_with_silent_tail_equals_ple_free_model():
    """lambda = 1 and a zero PLE projection give exactly the same logits as the model without PLE."""
    import dataclasses
    pc = gen.tiny_shared_pair()
    W = dict(gen.generate(pc))
    t = pc.target
    for l in range(t.n_layers):
        W[f"t{l}.wple_p"] = gen.pack_q41(np.zeros((t.hidden, t.ple_dim), np.float32))
        W[f"t{l}.lambda"] = gen.bf16_bits(np.ones(1, np.float32))
    t0 = dataclasses.replace(t, ple_dim=0)
    toks = gen.prompt(t.vocab, 6)
    la = om.Target(t, W).forward(toks)
    lb = om.Target(t0, W).forward(toks)
    np.testing.assert_array_equal(la, lb)


# ---- single-turn serving on a pinned prefix (FastFlowLM PR #899 "gemma4e-dflash-flash", "What" and
# "Changes": system prompt pinned and reused; no re-checkpoint after prefill; no KV row for the stop token)
def _pinned(pc, W, prefix):
    pair = oracle.Pair(pc, W)
    pair.prefill(prefix, oracle.Sampler())
    return pair, pair.snapshot()


def test_single_turn_requests_repeat_exactly():
    """Requests A, B, A, B, A on one pinned prefix: every A gives the same tokens, every B too, and each
    equals a fresh context that prefilled prefix + request. A server that re-checkpoints after each
    request's prefill (the pages' bug) restores into a stale context and answers A differently."""
    pc = gen.tiny_shared_pair()
    W = gen.generate(pc)
    V = pc.target.vocab
    prefix = list(gen.prompt(V, 24, request=30))
    req = {"A": list(gen.prompt(V, 12, request=31)), "B": list(gen.prompt(V, 12, request=32))}
    pair, pin = _pinned(pc, W, prefix)
    out = {"A": [], "B": []}
    for name in "ABABA":
        out[name].append(oracle.serve_single_turn(pair, pin, req[name], 16, oracle.Sampler()).tokens)
    for name in "AB":
        assert all(o == out[name][0] for o in out[name])
        fresh = oracle.plain_decode(oracle.Pair(pc, W), prefix + req[name], 16, oracle.Sampler())
        assert [int(t) for t in out[name][0]] == [int(t) for t in fresh.tokens]
    # the mutant: the pin is overwritten by each request's prefill
    bad, pin2 = _pinned(pc, W, prefix)
    for name in "AB":                      # each request's prefill taken as the new pin
        bad.restore(pin2)
        bad.prefill(req[name], oracle.Sampler())
        pin2 = bad.snapshot()
    bad_a = oracle.serve_single_turn(bad, pin2, req["A"], 16, oracle.Sampler()).tokens
    assert bad_a != out["A"][0]


def test_single_turn_stop_token_has_no_row():
    """The stop token is emitted and ends the request; no row of the context holds it: positions held
    = prefix + prompt + tokens before the stop token."""
    pc = gen.tiny_shared_pair()
    W = gen.generate(pc)
    V = pc.target.vocab
    prefix = list(gen.prompt(V, 24, request=30))
    prompt = list(gen.prompt(V, 12, request=31))
    pair, pin = _pinned(pc, W, prefix)
    full = oracle.serve_single_turn(pair, pin, prompt, 20, oracle.Sampler()).tokens
    stop = int(full[9])
    j = [int(t) for t in full].index(stop)
    run = oracle.serve_single_turn(pair, pin, prompt, 20, oracle.Sampler(), stop=stop)
    assert [int(t) for t in run.tokens] == [int(t) for t in full[: j + 1]]
    assert pair.target.positions_held() == len(prefix) + len(prompt) + j
