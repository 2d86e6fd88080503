"""Helpers of the GPU parity tests: run the CUDA path through the C ABI and the oracle side by side."""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

import gen
import oracle
from dflash_speculative_decode_gb300 import DFL_OPT_KEEP_LOGITS, Engine, config_from_pair

LOGIT_REL_L1 = 1e-3      # tolerance on logits: sum|gpu - ref| / sum|ref|
LOGIT_MAX_ABS = 2e-2     # and max |gpu - ref|
NEAR_TIE = 1e-3          # greedy: top-2 logit gap below which a differing argmax is allowed
NEAR_TIE_SAMPLED = 1e-5  # sampled: relative distance of u*sum(p) to an interval edge (at least; see
                         # lockstep: widened to what the row's own logit error can move an edge)


def rel_l1(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.abs(a - b).sum() / max(np.abs(b).sum(), 1e-30))


def check_logits(got, ref, what=""):
    r = rel_l1(got, ref)
    m = float(np.abs(np.asarray(got, np.float64) - np.asarray(ref, np.float64)).max())
    assert r <= LOGIT_REL_L1 and m <= LOGIT_MAX_ABS, f"{what}: rel-L1 {r:.3g}, max-abs {m:.3g}"
    return r, m


def engine(pc, W) -> Engine:
    eng = Engine(config_from_pair(pc))
    eng.load(W)
    return eng


@dataclass
class Lockstep:
    passes: int = 0
    near_ties: int = 0          # mismatches on the verify side (target tokens), each at a near-tie
    draft_near_ties: int = 0    # mismatched draft proposals, each at a near-tie (proposals are planted)
    max_rel_l1: float = 0.0
    max_abs: float = 0.0
    tokens: list = field(default_factory=list)
    accepted: list = field(default_factory=list)


def lockstep(pc, W, prompt, n_gen, p=0.3, temperature=None, seed=3, eng=None, check_draft=True, op=None):
    """Speculative decode on the GPU and in the oracle, pass by pass, with planted drafts at
    corruption p (planted from the oracle's plain decode of the same request). Checks draft logits and
    proposals, verify logits, target tokens, accepted lengths and positions held. A differing token is
    allowed only at a near-tie; both sides then continue with the GPU's token.
    `prompt` is prefilled on top of whatever both sides already hold: a fresh pair, or (eng, op) in the
    same state (a restored prefix snapshot)."""
    eng = eng or engine(pc, W)
    eng.dfl_set_option(DFL_OPT_KEEP_LOGITS, 1)
    sm = oracle.Sampler(temperature, seed)
    op = op or oracle.Pair(pc, W)
    n0 = op.target.n
    assert eng.dfl_positions_held() == n0
    snap = op.snapshot()
    plain = oracle.plain_decode(op, prompt, n_gen, sm)
    op.restore(snap)
    G = np.zeros(pc.max_ctx + 32, np.int32)
    G[n0 + len(prompt):n0 + len(prompt) + len(plain.tokens)] = plain.tokens
    cor = gen.corruption(p, pc.target.vocab, pc.max_ctx + 32)
    B = pc.draft.block
    res = Lockstep()
    t_o, close = op.prefill(prompt, sm)
    t_g = eng.dfl_prefill(prompt, temperature, seed)
    lim = NEAR_TIE if temperature is None else NEAR_TIE_SAMPLED
    if t_g != t_o:
        assert close < lim, f"prefill token {t_g} != {t_o} (closeness {close})"
        res.near_ties += 1
    tokens = [t_g]
    while len(tokens) < n_gen:
        n = op.target.n
        assert eng.dfl_positions_held() == n
        last = tokens[-1]
        if check_draft:
            op.sync_draft()
            dp_o, dl_o = op.draft.block(last, W["emb"], W["head"])
            dp_g = eng.dfl_draft_block(last)
            dl_g = eng.dfl_read_logits(1, B - 1)
            r, m = check_logits(dl_g, dl_o, f"draft logits at n={n}")
            res.max_rel_l1, res.max_abs = max(res.max_rel_l1, r), max(res.max_abs, m)
            for i in range(B - 1):
                if dp_g[i] != dp_o[i]:
                    assert oracle.model.top2_gap(dl_o[i]) < NEAR_TIE, f"draft proposal {i} at n={n}"
                    res.draft_near_ties += 1
        props = cor.propose(G, np.arange(n + 1, n + B))
        rows = [last] + [int(v) for v in props]
        tt_o, cl, lg_o = op.verify(rows, sm)
        tt_g, a_g = eng.dfl_verify_block(rows, temperature=temperature, seed=seed)
        lg_g = eng.dfl_read_logits(0, B)
        r, m = check_logits(lg_g, lg_o, f"verify logits at n={n}")
        res.max_rel_l1, res.max_abs = max(res.max_rel_l1, r), max(res.max_abs, m)
        for i in range(B):
            if tt_g[i] != tt_o[i]:
                lim_i = lim
                if temperature is not None:
                    # a logit error of at most d moves every p_j by a factor within exp(+-d/T), so each
                    # cumulative edge, relative to the total, by at most expm1(2 d / T)
                    d = float(np.abs(np.asarray(lg_g[i], np.float64) - np.asarray(lg_o[i], np.float64)).max())
                    lim_i = max(lim, math.expm1(2.0 * d / temperature))
                assert cl[i] < lim_i, f"target token row {i} at n={n}: {tt_g[i]} vs {tt_o[i]} (closeness {cl[i]})"
                res.near_ties += 1
        a_o = oracle.accept_length(rows[1:], list(tt_g[:-1]))
        assert a_g == a_o, f"accepted {a_g} vs {a_o} at n={n}"
        kept = eng.dfl_commit_accepted(n_gen - len(tokens))
        emit = [int(v) for v in tt_g[:kept]]
        assert kept == min(a_g + 1, n_gen - len(tokens))
        op.target.commit(kept)
        res.passes += 1
        res.accepted.append(a_g)
        tokens += emit
    res.tokens = tokens
    assert eng.dfl_positions_held() == op.target.n
    return res, plain
