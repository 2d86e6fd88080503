"""The decode loops of `decode.py` (plain, speculative, single-turn serving over a prefix cache) on the
CPU. They drive a stand-in engine that keeps the C ABI's host-side contract: positions held, one pending
verify, the commit of the accepted rows within a budget and up to a stop token, and device snapshots
(here the oracle's) restored any number of times. The model arithmetic behind it is the oracle pair, so
every loop can be compared with the oracle's own loop over the same requests (model card
"Nemotron-3.5-Bolt-E4B-DFlash-NPU2", "How it is used"; FastFlowLM PR #899 "gemma4e-dflash-flash",
"What" and "Changes")."""
import numpy as np
import pytest

import gen
import oracle
from dflash_speculative_decode_gb300 import decode


class _Cfg:
    def __init__(self, block):
        self.block = block


class OracleEngine:
    """The calls `decode.py` makes, with the ABI's state rules, over an oracle pair (a test double)."""

    def __init__(self, pc, W):
        self.pc, self.W = pc, W
        self.pair = oracle.Pair(pc, W)
        self.cfg = _Cfg(pc.draft.block)
        self.pending = None          # (k, accepted, target tokens) of the verify awaiting its commit
        self.prefill_calls = 0

    def dfl_positions_held(self):
        return self.pair.target.n

    def dfl_prefill(self, tokens, temperature=None, seed=0):
        assert self.pending is None, "DFL_E_STATE: a verify is pending"
        self.prefill_calls += 1
        tok, _ = self.pair.prefill(list(tokens), oracle.Sampler(temperature, seed))
        return int(tok)

    def dfl_draft_block(self, last_tok, want=True):
        assert self.pending is None, "DFL_E_STATE: a verify is pending"
        self.pair.sync_draft()
        dp, _ = self.pair.draft.block(int(last_tok), self.W["emb"], self.W["head"])
        return np.asarray(dp, np.int32) if want else None

    def dfl_verify_block(self, rows, k=None, temperature=None, seed=0):
        assert self.pending is None, "DFL_E_STATE: a verify is pending"
        rows = [int(v) for v in rows]
        tt, _, _ = self.pair.verify(rows, oracle.Sampler(temperature, seed))
        a = oracle.accept_length(rows[1:], list(tt[:-1]))
        self.pending = (len(rows), a, [int(v) for v in tt])
        return np.asarray(tt, np.int32), a

    def dfl_commit_verify_rows(self, keep):
        k, _, _ = self.pending
        assert 0 <= keep <= k, "DFL_E_INVALID_ARG: keep must be 0..k"
        self.pair.target.commit(keep)
        self.pending = None

    def dfl_commit_accepted(self, max_keep, stop_token=-1):
        k, a, tt = self.pending
        keep = min(a + 1, k, max_keep)
        stopped = False
        if stop_token >= 0:
            for i in range(keep):
                if tt[i] == stop_token:
                    keep, stopped = i + 1, True
                    break
        self.dfl_commit_verify_rows(keep)
        return keep if stop_token < 0 else (keep, stopped)

    def dfl_snapshot(self):
        assert self.pending is None, "DFL_E_STATE: snapshot needs the committed state"
        return self.pair.snapshot()

    def dfl_restore(self, snap):
        assert self.pending is None, "DFL_E_STATE: restore needs the committed state"
        self.pair.restore(snap)


@pytest.fixture(scope="module")
def tiny():
    pc = gen.tiny_pair()
    return pc, gen.generate(pc)


def _planted(pc, W, prompt, n_gen, p, temperature=None, seed=3):
    """Proposals planted from the oracle's plain decode of the request (corruption p, keyed by position)."""
    ref = oracle.plain_decode(oracle.Pair(pc, W), prompt, n_gen, oracle.Sampler(temperature, seed))
    G = np.zeros(pc.max_ctx + 32, np.int32)
    G[len(prompt):len(prompt) + len(ref.tokens)] = ref.tokens
    cor = gen.corruption(p, pc.target.vocab, pc.max_ctx + 32)
    return ref, (lambda n, dp: cor.propose(G, np.arange(n + 1, n + pc.draft.block)))


@pytest.mark.parametrize("temperature", [None, 0.8])
def test_spec_decode_matches_the_oracle_loop(tiny, temperature):
    """Tokens, accepted lengths and positions held of decode.spec_decode equal those of the oracle's
    speculative loop, and both equal the plain decode of the same request (greedy or sampled)."""
    pc, W = tiny
    prompt = gen.prompt(pc.target.vocab, 24, request=51)
    ref, propose = _planted(pc, W, prompt, 30, 0.3, temperature)
    eng = OracleEngine(pc, W)
    got = decode.spec_decode(eng, prompt, 30, temperature=temperature, seed=3, propose=propose)
    want = oracle.spec_decode(oracle.Pair(pc, W), prompt, 30, oracle.Sampler(temperature, 3), propose=propose)
    assert got.tokens == [int(t) for t in want.tokens] == [int(t) for t in ref.tokens]
    assert got.accepted == [s.accepted for s in want.steps]
    assert got.held == [s.n for s in want.steps]
    assert eng.dfl_positions_held() == len(prompt) + len(got.tokens) - 1
    assert got.passes < len(got.tokens) - 1          # some proposals were accepted


def test_spec_decode_stops_at_the_budget(tiny):
    """A pass that accepts more than the budget allows commits only the budget's rows."""
    pc, W = tiny
    prompt = gen.prompt(pc.target.vocab, 20, request=52)
    _, propose = _planted(pc, W, prompt, 40, 0.0)    # every proposal right: 8 tokens per pass
    for n_gen in (1, 2, 9, 13):
        eng = OracleEngine(pc, W)
        got = decode.spec_decode(eng, prompt, n_gen, propose=propose)
        assert len(got.tokens) == n_gen
        assert eng.dfl_positions_held() == len(prompt) + n_gen - 1


def test_plain_decode_matches_the_oracle(tiny):
    pc, W = tiny
    prompt = gen.prompt(pc.target.vocab, 16, request=53)
    got = decode.plain_decode(OracleEngine(pc, W), prompt, 12)
    want = oracle.plain_decode(oracle.Pair(pc, W), prompt, 12, oracle.Sampler())
    assert got.tokens == [int(t) for t in want.tokens]
    assert got.accepted == [0] * 11


def test_prefix_cache_pins_and_evicts_least_recently_used(tiny):
    """Two slots over prefixes P1, P2, P1, P3, P2: P1's second request reuses its pin; P3 evicts P2
    (least recently used), so P2's second request prefills it again. Every request's tokens equal the
    oracle's single-turn request over its own pinned prefix, and P1's two requests agree."""
    pc, W = tiny
    V = pc.target.vocab
    pre = {f"P{i}": [int(v) for v in gen.prompt(V, 20 + 4 * i, request=60 + i)] for i in (1, 2, 3)}
    prompt = [int(v) for v in gen.prompt(V, 6, request=64)]
    eng = OracleEngine(pc, W)
    cache = decode.PrefixCache(eng, slots=2)
    calls, out = [], []
    for name in ("P1", "P2", "P1", "P3", "P2"):
        before = eng.prefill_calls
        g = decode.serve_single_turn(eng, cache, pre[name], prompt, 14)
        calls.append(eng.prefill_calls - before)      # 2 on a miss (prefix, prompt), 1 on a hit
        out.append(g.tokens)
        pin = oracle.Pair(pc, W)
        pin.prefill(pre[name], oracle.Sampler())
        want = oracle.serve_single_turn(pin, pin.snapshot(), prompt, 14, oracle.Sampler())
        assert g.tokens == [int(t) for t in want.tokens], name
        assert eng.dfl_positions_held() == len(pre[name]) + len(prompt) + len(g.tokens) - 1
    assert calls == [2, 2, 1, 2, 2]
    assert out[0] == out[2]
    assert list(cache.pins) == [tuple(pre["P3"]), tuple(pre["P2"])]
    with pytest.raises(ValueError):
        decode.PrefixCache(eng, slots=0)


def test_single_turn_stop_token_has_no_row(tiny):
    """With every planted proposal right (8 tokens per pass), a stop token in the middle of an accepted
    run ends the request there: it is the last token emitted, that pass commits only the rows up to it,
    and the context holds the prefix, the prompt and every emitted token but the stop token."""
    pc, W = tiny
    V = pc.target.vocab
    prefix = [int(v) for v in gen.prompt(V, 24, request=70)]
    prompt = [int(v) for v in gen.prompt(V, 5, request=71)]
    _, propose = _planted(pc, W, prefix + prompt, 40, 0.0)
    eng = OracleEngine(pc, W)
    cache = decode.PrefixCache(eng)
    full = decode.serve_single_turn(eng, cache, prefix, prompt, 20, propose=propose)
    assert full.accepted[0] == pc.draft.block - 1
    stop = full.tokens[11]                            # inside the second pass's run of 8
    first = full.tokens.index(stop)                   # its first occurrence ends the request
    got = decode.serve_single_turn(eng, cache, prefix, prompt, 20, stop_token=stop, propose=propose)
    assert got.tokens == full.tokens[:first + 1]
    assert eng.dfl_positions_held() == len(prefix) + len(prompt) + first
    pin = oracle.Pair(pc, W)
    pin.prefill(prefix, oracle.Sampler())
    want = oracle.serve_single_turn(pin, pin.snapshot(), prompt, 20, oracle.Sampler(), stop=stop, propose=propose)
    assert got.tokens == [int(t) for t in want.tokens]
