"""Decode loops over the C ABI: prefill, then draft -> verify -> accept -> commit until a token budget.

Acceptance (model card "Nemotron-3.5-Bolt-E4B-DFlash-NPU2", "How it is used"): each pass proposes up to
block-1 tokens, the target checks them together, and the longest agreeing prefix plus one token of the
target's own is kept; the next pass starts that many positions later (1bit engine PR "a Gemma4 pack
stops re-reading its weights every token; tools/dflash_acceptance", item 2).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Callable, List, Optional

import numpy as np


@dataclass
class Generation:
    tokens: List[int]                                   # generated tokens (the first from prefill)
    accepted: List[int] = field(default_factory=list)   # accepted proposals per pass
    held: List[int] = field(default_factory=list)       # positions held before each pass
    proposals: List[list] = field(default_factory=list)  # the draft's own proposals per pass
    targets: List[list] = field(default_factory=list)    # the target's tokens per pass

    @property
    def passes(self) -> int:
        return len(self.accepted)


def plain_decode(eng, prompt, n_gen: int, temperature=None, seed=0) -> Generation:
    """Token-by-token decode: verify one row, commit it."""
    t = eng.dfl_prefill(prompt, temperature, seed)
    g = Generation(tokens=[t])
    while len(g.tokens) < n_gen:
        g.held.append(eng.dfl_positions_held())
        tt, a = eng.dfl_verify_block([g.tokens[-1]], temperature=temperature, seed=seed)
        eng.dfl_commit_verify_rows(1)
        g.accepted.append(0)
        g.targets.append(list(map(int, tt)))
        g.tokens.append(int(tt[0]))
    return g


def spec_decode(eng, prompt, n_gen: int, temperature=None, seed=0,
                propose: Optional[Callable[[int, np.ndarray], np.ndarray]] = None) -> Generation:
    """Speculative decode. `propose(held, draft_proposals)` may replace the draft's proposals for
    positions held+1..held+block-1 (planted drafts); the draft block still runs every pass."""
    B = eng.cfg.block
    t = eng.dfl_prefill(prompt, temperature, seed)
    g = Generation(tokens=[t])
    while len(g.tokens) < n_gen:
        n = eng.dfl_positions_held()
        last = g.tokens[-1]
        dp = eng.dfl_draft_block(last)
        props = np.asarray(propose(n, dp) if propose else dp, np.int32)[: B - 1]
        rows = np.concatenate([[last], props]).astype(np.int32)
        tt, a = eng.dfl_verify_block(rows, temperature=temperature, seed=seed)
        kept = eng.dfl_commit_accepted(n_gen - len(g.tokens))   # accepted + 1, within the budget
        emit = [int(v) for v in tt[:kept]]                     # the verify's tokens of the kept rows
        g.held.append(n)
        g.accepted.append(a)
        g.proposals.append(list(map(int, dp)))
        g.targets.append(list(map(int, tt)))
        g.tokens += emit
    return g


class PrefixCache:
    """Pinned prefixes for single-turn serving: each is prefilled once into a context that starts empty,
    and its committed state is kept as a device snapshot (dfl_snapshot). At most `slots` prefixes are kept;
    the least recently used one is dropped first. Requests only ever restore a pin: nothing checkpoints
    over it (FastFlowLM PR #899 "gemma4e-dflash-flash", "Changes": a re-checkpoint after prefill overwrote
    the pinned system prefix, so repeated requests gave different answers)."""

    def __init__(self, eng, slots: int = 1):
        if slots < 1:
            raise ValueError("slots must be >= 1")
        self.eng, self.slots = eng, slots
        self.empty = eng.dfl_snapshot()          # the context as created: no positions held
        self.pins = {}                           # prefix tokens -> snapshot, in use order

    def pin(self, prefix, temperature=None, seed=0):
        key = tuple(int(t) for t in prefix)
        if key in self.pins:
            snap = self.pins.pop(key)
        else:
            if len(self.pins) >= self.slots:
                self.pins.pop(next(iter(self.pins)))
            self.eng.dfl_restore(self.empty)
            self.eng.dfl_prefill(list(key), temperature, seed)
            snap = self.eng.dfl_snapshot()
        self.pins[key] = snap
        return snap


def serve_single_turn(eng, cache: PrefixCache, prefix, prompt, n_gen: int, stop_token=None, temperature=None,
                      seed=0, propose: Optional[Callable[[int, np.ndarray], np.ndarray]] = None) -> Generation:
    """One single-turn request: restore the pinned prefix, prefill the prompt, then speculative decode
    until n_gen tokens or the stop token. The stop token is emitted but never fed back: no row of the
    context holds it (dfl_commit_accepted with the stop token), and the request leaves no checkpoint."""
    B = eng.cfg.block
    stop = -1 if stop_token is None else int(stop_token)
    eng.dfl_restore(cache.pin(prefix, temperature, seed))
    t = eng.dfl_prefill(prompt, temperature, seed)
    g = Generation(tokens=[t])
    if t == stop:
        return g
    while len(g.tokens) < n_gen:
        n = eng.dfl_positions_held()
        last = g.tokens[-1]
        dp = eng.dfl_draft_block(last)
        props = np.asarray(propose(n, dp) if propose else dp, np.int32)[: B - 1]
        rows = np.concatenate([[last], props]).astype(np.int32)
        tt, a = eng.dfl_verify_block(rows, temperature=temperature, seed=seed)
        kept, stopped = eng.dfl_commit_accepted(n_gen - len(g.tokens), stop) if stop >= 0 else \
            (eng.dfl_commit_accepted(n_gen - len(g.tokens)), False)
        g.held.append(n)
        g.accepted.append(a)
        g.proposals.append(list(map(int, dp)))
        g.targets.append(list(map(int, tt)))
        g.tokens += [int(v) for v in tt[:kept]]
        if stopped:
            break
    return g
