"""Oracle speculative loop: prefill, plain decode, and the draft -> verify -> accept -> commit walk.
TEST INFRASTRUCTURE ONLY (see oracle/model.py).

Acceptance (model card "Nemotron-3.5-Bolt-E4B-DFlash-NPU2", "How it is used"; acceptance tool of the
1bit engine PR "a Gemma4 pack stops re-reading its weights every token", item 2): the verify's row i
(i = 0..k-1) gives the target's token t_i for position n+i+1; proposal d_i (position n+i) is accepted
while d_i == t_{i-1}; a pass that accepted a emits d_1..d_a and t_a and keeps a + 1 rows, so the next
pass starts a + 1 positions later. Greedy takes the first maximum; with a temperature every position is
sampled (uniform keyed by the absolute position of the token drawn) and compared with the draft.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Callable, List, Optional

import numpy as np

from . import _native as nat
from .model import Draft, Target, argmax_first, top2_gap


@dataclass
class Sampler:
    """None-temperature means greedy."""
    temperature: Optional[float] = None
    seed: int = 3

    def pick(self, logits: np.ndarray, position: int):
        """(token for `position`, closeness to a decision boundary: top-2 logit gap for greedy,
        relative distance of u*sum(p) to the interval edge for sampling)."""
        if self.temperature is None:
            return argmax_first(logits), top2_gap(logits)
        u = nat.uniform(self.seed, position)
        return nat.sample(logits, self.temperature, u)


def accept_length(proposals, target_tokens) -> int:
    """Longest prefix with proposals[i] == target_tokens[i] (proposal i is for the position that target
    row i predicts)."""
    a = 0
    while a < len(proposals) and proposals[a] == target_tokens[a]:
        a += 1
    return a


@dataclass
class StepRecord:
    n: int                      # positions held before the pass
    rows: List[int]             # verify rows: last token, then proposals
    target: List[int]           # target token per row
    accepted: int
    emitted: List[int]
    closeness: List[float]
    draft_proposals: Optional[List[int]] = None


@dataclass
class Run:
    tokens: List[int]                          # generated tokens (first one from prefill)
    steps: List[StepRecord] = field(default_factory=list)
    prefill_closeness: float = 0.0


class Pair:
    """Target + draft with the draft's context kept up to date with committed rows."""

    def __init__(self, pc, W, width_mutant=None, with_draft=True, **target_options):
        self.pc = pc
        self.target = Target(pc.target, W, tap_layers=pc.draft.taps, width_mutant=width_mutant, **target_options)
        self.draft = Draft(pc.draft, W, pc.target) if with_draft else None
        self.W = W

    def sync_draft(self) -> None:
        if self.draft is not None and self.draft.n_ctx < self.target.n:
            self.draft.append_ctx(self.target.taps[self.draft.n_ctx:self.target.n])

    def prefill(self, prompt, sampler: Sampler, chunk: int = 0):
        """Run the prompt (in chunks of `chunk` rows, or all at once), commit it, return the first
        generated token and its closeness."""
        prompt = list(map(int, prompt))
        step = chunk or len(prompt)
        logits = None
        for i in range(0, len(prompt), step):
            rows = prompt[i:i + step]
            logits = self.target.forward(rows, head_rows=1)
            self.target.commit(len(rows))
        self.sync_draft()
        return sampler.pick(logits[-1], self.target.n)

    def snapshot(self):
        return (self.target.snapshot(), self.draft.snapshot() if self.draft else None)

    def restore(self, snap) -> None:
        self.target.restore(snap[0])
        if self.draft is not None:
            self.draft.restore(snap[1])

    def verify(self, rows, sampler: Sampler):
        n = self.target.n
        logits = self.target.forward(rows)
        picks = [sampler.pick(logits[i], n + i + 1) for i in range(len(rows))]
        return [p[0] for p in picks], [p[1] for p in picks], logits


def plain_decode(pair: Pair, prompt, n_gen: int, sampler: Sampler) -> Run:
    """Token-by-token decode: one row per pass."""
    t, close = pair.prefill(prompt, sampler)
    run = Run(tokens=[t], prefill_closeness=close)
    while len(run.tokens) < n_gen:
        n = pair.target.n
        tt, cl, _ = pair.verify([run.tokens[-1]], sampler)
        pair.target.commit(1)
        run.steps.append(StepRecord(n, [run.tokens[-1]], tt, 0, [tt[0]], cl))
        run.tokens.append(tt[0])
    pair.sync_draft()
    return run


def spec_decode(pair: Pair, prompt, n_gen: int, sampler: Sampler,
                propose: Optional[Callable[[int, List[int]], List[int]]] = None,
                run_draft: bool = True) -> Run:
    """Speculative decode. propose(n, draft_proposals) may replace the draft's proposals (planted
    drafts); it receives the positions-held count n (proposals are for positions n+1..n+B-1)."""
    B = pair.pc.draft.block
    t, close = pair.prefill(prompt, sampler)
    run = Run(tokens=[t], prefill_closeness=close)
    while len(run.tokens) < n_gen:
        n = pair.target.n
        last = run.tokens[-1]
        dprops = None
        if run_draft:
            pair.sync_draft()
            dp, _ = pair.draft.block(last, pair.W["emb"], pair.W["head"])
            dprops = [int(v) for v in dp]
        props = list(propose(n, dprops)) if propose else list(dprops)
        rows = [last] + props[: B - 1]
        tt, cl, _ = pair.verify(rows, sampler)
        a = accept_length(rows[1:], tt[:-1])
        emit = rows[1:1 + a] + [tt[a]]
        emit = emit[: n_gen - len(run.tokens)]
        pair.target.commit(len(emit))
        run.steps.append(StepRecord(n, rows, tt, a, emit, cl, dprops))
        run.tokens += emit
    pair.sync_draft()
    return run


def serve_single_turn(pair: Pair, pin, prompt, n_gen: int, sampler: Sampler, stop=None,
                      propose: Optional[Callable[[int, List[int]], List[int]]] = None) -> Run:
    """One single-turn request (FastFlowLM PR #899 "gemma4e-dflash-flash", "What" and "Changes"): restore
    the pinned prefix snapshot `pin`, prefill the prompt, speculative decode until n_gen tokens or the stop
    token. The stop token is emitted but never becomes a row of the context, and the request takes no
    checkpoint of its own."""
    B = pair.pc.draft.block
    pair.restore(pin)
    t, close = pair.prefill(prompt, sampler)
    run = Run(tokens=[t], prefill_closeness=close)
    if stop is not None and t == stop:
        return run
    while len(run.tokens) < n_gen:
        n = pair.target.n
        last = run.tokens[-1]
        pair.sync_draft()
        dp, _ = pair.draft.block(last, pair.W["emb"], pair.W["head"])
        dprops = [int(v) for v in dp]
        props = list(propose(n, dprops)) if propose else dprops
        rows = [last] + props[: B - 1]
        tt, cl, _ = pair.verify(rows, sampler)
        a = accept_length(rows[1:], tt[:-1])
        emit = (rows[1:1 + a] + [tt[a]])[: n_gen - len(run.tokens)]
        if stop is not None and stop in emit:
            emit = emit[: emit.index(stop) + 1]
        pair.target.commit(len(emit))
        run.steps.append(StepRecord(n, rows, tt, a, emit, cl, dprops))
        run.tokens += emit
        if stop is not None and emit[-1] == stop:
            break
    pair.sync_draft()
    return run
