"""Oracle for the DFlash speculative-decode step: the target's batched verify, the draft's block
forward, acceptance, commit and snapshot. TEST INFRASTRUCTURE ONLY: imported by tests/, by the
smoke check and by the benchmark's CPU-baseline leg; never by the library.

Plain and slow on purpose. Every product runs in dfl_oracle.c (double, ascending k); everything else
here is double-precision numpy on one row at a time. Activations, keys, values and taps are the pages'
"floats" (KV planes of "2 x 256 floats per position"; taps of "(P+tokens)*T*H floats"): every value is
rounded to float32 where the model stores it. Weights are Q4_1 or bf16 as stored.

Sources (pages, by title and section):
  * 1bit engine PR "npu forward: Gemma4 verifies a draft in one batched pass; KV row width per layer",
    "What changes": the batched body builds every row's per-layer inputs, runs the PLE gate and
    projection as M-row GEMMs then the layer scalar; a KV-shared layer reads its owner's plane and
    appends nothing; shared layers use the double-wide MLP; KV width per layer (sliding layers hold
    2 x 256 floats per position, full layers 2 x 512); a shared layer holds no plane of its own and the
    positions-held count ignores it. "Proof": k rows of a batched pass equal k sequential steps;
    commit_verify_rows(2) after 3 held leaves 5; the next step equals a forward that saw only the
    accepted rows. Reviewer excerpt of kv_widths() and of the sandwich-norm flag.
  * Model card "Nemotron-3.5-Bolt-E4B-DFlash-NPU2": spec table (draft shape, taps = zero-based layer
    outputs fused by fc, fc and norms in BF16) and "How it is used" (propose up to 7 tokens; keep the
    longest agreeing prefix plus one target token; with a sampler every position is sampled and
    compared with the draft).
  * 1bit engine PR "a Gemma4 pack stops re-reading its weights every token; tools/dflash_acceptance",
    item 2 and the tool's header: the draft's block is the target's embeddings of [token s, mask,
    mask, ...] times the draft's embedding scale, its context the tapped rows of positions 0..s-1;
    block rows after the first go through the target's head; argmax takes the first maximum; after a
    pass that accepted a, the next pass starts a + 1 later.
"""
from __future__ import annotations

import copy
from dataclasses import dataclass
from typing import Dict, List, Optional

import numpy as np

from . import _native as nat

F32, F64 = np.float32, np.float64


# ---- elementwise definitions (double precision, stored as float32) -----------------------------
def rmsnorm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm of each row of x: x * (mean(x^2) + eps)^(-1/2) * w."""
    xd = np.asarray(x, F64)
    ms = np.mean(xd * xd, axis=-1, keepdims=True)
    return (xd / np.sqrt(ms + eps) * np.asarray(w, F64)).astype(F32)


def rope(v: np.ndarray, pos: int, base: float) -> np.ndarray:
    """Rotate pairs (i, i + d/2) of a head vector by pos * base^(-2i/d) (half-split rotary embedding)."""
    d = v.shape[-1]
    h = d // 2
    theta = np.power(F64(base), -2.0 * np.arange(h, dtype=F64) / d)
    ang = F64(pos) * theta
    c, s = np.cos(ang), np.sin(ang)
    a, b = np.asarray(v[..., :h], F64), np.asarray(v[..., h:], F64)
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1).astype(F32)


def silu(g: np.ndarray) -> np.ndarray:
    """SiLU (the "swish" gate of SwiGLU): g * sigmoid(g) = g / (1 + exp(-g))."""
    gd = np.asarray(g, F64)
    return gd / (1.0 + np.exp(-gd))


def swiglu(gu: np.ndarray, F: int) -> np.ndarray:
    """SwiGLU of a fused gate|up product: silu(gate) * up, the gate being the first F columns and up the
    next F (the fused matrix is named "gate|up", gate first)."""
    return (silu(gu[..., :F]) * np.asarray(gu[..., F:2 * F], F64)).astype(F32)


def ple_tail(x: np.ndarray, p_l: np.ndarray, Wg: np.ndarray, Wp: np.ndarray, w_norm: np.ndarray, lam: float,
             eps: float) -> np.ndarray:
    """Per-layer-embedding tail of one target layer (1bit engine PR "npu forward: Gemma4 verifies a draft
    in one batched pass", "What changes": the PLE gate and projection as M-row GEMMs, then the layer
    scalar). The gate reads the residual stream x itself; z = silu(x . Wg) * p_l (the token's row of the
    per-layer table); y = z . Wp is normed and added to x, and the sum is multiplied by lambda."""
    t = nat.linear_q41(x, Wg)
    z = (silu(t) * np.asarray(p_l, F64)).astype(F32)
    y = nat.linear_q41(z, Wp)
    xs = add(x, rmsnorm(y, w_norm, eps))
    return (np.asarray(xs, F64) * F64(np.float32(lam))).astype(F32)


def attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """softmax(K q * scale) V for one query over the given keys (rows of K, V)."""
    s = (np.asarray(K, F64) * np.asarray(q, F64)).sum(axis=1) * scale
    p = np.exp(s - s.max())
    return ((p[:, None] * np.asarray(V, F64)).sum(axis=0) / p.sum()).astype(F32)


def add(x, y):
    return (np.asarray(x, F64) + np.asarray(y, F64)).astype(F32)


def argmax_first(logits: np.ndarray) -> int:
    """Index of the first maximum (ties go to the smallest index)."""
    return int(np.argmax(logits))


def top2_gap(logits: np.ndarray) -> float:
    s = np.partition(np.asarray(logits, F64), -2)
    return float(s[-1] - s[-2])


# ---- KV planes ------------------------------------------------------------------------------------
def kv_widths(cfg) -> List[int]:
    """Floats per position of each layer's own plane: 2 * kv_heads * head_dim for a layer that holds
    one, 0 for a KV-shared layer (its rows live in its owner's plane)."""
    return [cfg.kv_width(l) for l in range(cfg.n_layers)]


def keep_positions(planes: Dict[int, np.ndarray], widths: List[int], n: int) -> None:
    """Cut every plane to its first n positions, each at its own layer's width."""
    for l, p in planes.items():
        planes[l] = p[: n * widths[l]].copy()


def positions_held(planes: Dict[int, np.ndarray], widths: List[int]) -> int:
    """Positions held, counted over the planes that exist (shared layers have none)."""
    counts = {len(p) // widths[l] for l, p in planes.items()}
    if len(counts) != 1:
        raise RuntimeError(f"planes disagree on positions held: {sorted(counts)}")
    return counts.pop()


# ---- target -----------------------------------------------------------------------------------------
class Target:
    """The target model with one KV plane per layer that holds its own (linear storage: position j is row
    j). Options that model other storage, for the tests that show which ones the pins reject:
      ring_capacity: sliding layers also keep their rows in a ring of that many slots (slot = position mod
        capacity), as a fixed-size device arena would, and attention reads them from the ring. A ring of
        W + R_max - 1 slots holds every key any row of a pass of up to R_max rows still needs; a ring of W
        slots does not (a pass overwrites keys its own first rows, or the rows kept after a rollback, need).
      width_mutant: count every layer that holds a plane at this one width (the pages' single-width defect).
      shared_appends: a KV-shared layer also appends its owner's new rows to a plane of its own (a
        defect: such a layer must hold nothing)."""

    def __init__(self, cfg, W: dict, tap_layers=(), width_mutant: Optional[int] = None,
                 ring_capacity: Optional[int] = None, shared_appends: bool = False):
        self.cfg = cfg
        self.W = W
        self.tap_layers = tuple(tap_layers)
        self.norm = {k: nat.bf16_decode(v) for k, v in W.items() if k.endswith("norm")}
        self.lam = [float(nat.bf16_decode(W[f"t{l}.lambda"])[0]) if cfg.ple_dim else 1.0
                    for l in range(cfg.n_layers)]
        w = kv_widths(cfg)
        # a mutant that counts every layer at one width, to show the tests catch it
        self.widths = [width_mutant if (width_mutant and w[l]) else w[l] for l in range(cfg.n_layers)]
        self.planes: Dict[int, np.ndarray] = {l: np.zeros(0, F32) for l in range(cfg.n_layers) if cfg.is_owner(l)}
        self.shared_appends = shared_appends
        if shared_appends:
            for l in range(cfg.n_layers):
                if not cfg.is_owner(l):
                    self.planes[l] = np.zeros(0, F32)
                    self.widths[l] = w[cfg.kv_owner[l]]
        self.ring_capacity = ring_capacity
        self.rings: Dict[int, np.ndarray] = {}
        if ring_capacity:
            for l in range(cfg.n_layers):
                if cfg.is_owner(l) and cfg.layer_type[l] == 0:
                    self.rings[l] = np.zeros((ring_capacity, w[l]), F32)
        self.record = None               # optional dict: per-layer intermediates of the last forward
        self.n = 0                       # committed positions
        self.pending = 0                 # rows of the last forward not yet committed
        self.taps = np.zeros((0, len(self.tap_layers) * cfg.hidden), F32)

    # state
    def positions_held(self) -> int:
        return positions_held(self.planes, self.widths)

    def plane(self, l: int) -> Optional[np.ndarray]:
        """Layer l's own plane (None for a KV-shared layer, which holds none)."""
        return self.planes.get(l)

    def commit(self, keep: int) -> None:
        """commit_verify_rows(keep): positions held become n + keep; the later pending rows go."""
        if not (0 <= keep <= self.pending):
            raise ValueError("keep out of range")
        self.n += keep
        keep_positions(self.planes, self.widths, self.n)
        self.taps = self.taps[: self.n].copy()
        self.pending = 0

    def snapshot(self):
        if self.pending:
            raise RuntimeError("snapshot needs a committed state")
        return copy.deepcopy((self.n, self.planes, self.taps, self.rings))

    def restore(self, snap) -> None:
        n, planes, taps, rings = copy.deepcopy(snap)
        self.n, self.planes, self.taps, self.rings, self.pending = n, planes, taps, rings, 0

    # one batched pass
    def forward(self, tokens, head_rows: Optional[int] = None) -> np.ndarray:
        """Run rows `tokens` at positions n, n+1, ... through every layer (layer by layer, each row on
        its own); append their keys and values; return fp32 logits [k][vocab] (or of the last head_rows
        rows only). The rows stay pending until commit()."""
        if self.pending:
            raise RuntimeError("a verify is pending")
        c, W = self.cfg, self.W
        tokens = np.asarray(tokens, np.int64)
        k = len(tokens)
        H, hd, nq = c.hidden, c.head_dim, c.n_heads
        pos = self.n + np.arange(k)
        x = (np.asarray(nat.bf16_decode(W["emb"][tokens]), F64) * F64(np.float32(c.emb_scale))).astype(F32)
        ple = nat.bf16_decode(W["ple_table"][tokens]) if c.ple_dim else None
        taps = np.zeros((k, len(self.tap_layers) * H), F32)
        for l in range(c.n_layers):
            p = f"t{l}."
            own, nkv = c.kv_owner[l], c.kv_heads[l]
            base = c.rope_base_full if c.layer_type[l] else c.rope_base_sliding
            h = rmsnorm(x, self.norm[p + "attn_norm"], c.eps)
            y = nat.linear_q41(h, W[p + "wqkv"] if own == l else W[p + "wq"])
            q = y[:, : nq * hd].reshape(k, nq, hd)
            q = np.stack([rope(rmsnorm(q[i], self.norm[p + "q_norm"], c.eps), pos[i], base) for i in range(k)])
            if own == l:
                kk = y[:, nq * hd:(nq + nkv) * hd].reshape(k, nkv, hd)
                vv = y[:, (nq + nkv) * hd:(nq + 2 * nkv) * hd]
                kk = np.stack([rope(rmsnorm(kk[i], self.norm[p + "k_norm"], c.eps), pos[i], base) for i in range(k)])
                rows = np.concatenate([kk.reshape(k, -1), vv], axis=1).astype(F32)
                self.planes[l] = np.concatenate([self.planes[l], rows.reshape(-1)])
                if l in self.rings:
                    for i in range(k):
                        self.rings[l][pos[i] % self.ring_capacity] = rows[i]
            elif self.shared_appends:
                # the defect: the owner's new rows appended again to a plane of this layer's own
                w_own = 2 * nkv * hd
                self.planes[l] = np.concatenate([self.planes[l], self.planes[own][-k * w_own:]])
            width = self.widths[own]
            plane = self.planes[own].reshape(-1, width) if width == 2 * nkv * hd else None
            if plane is None:   # only the width mutant gets here: read the plane at its true row length
                plane = self.planes[own][: len(self.planes[own]) // (2 * nkv * hd) * (2 * nkv * hd)]
                plane = plane.reshape(-1, 2 * nkv * hd)
            o = np.zeros((k, nq, hd), F32)
            grp = nq // nkv
            for i in range(k):
                hi = pos[i] + 1
                lo = max(0, hi - c.window) if c.layer_type[l] == 0 else 0
                if own in self.rings:   # keys and values as the ring holds them now
                    rows_i = self.rings[own][np.arange(lo, hi) % self.ring_capacity]
                else:
                    rows_i = plane[lo:hi]
                for hq in range(nq):
                    g = hq // grp
                    Kj = rows_i[:, g * hd:(g + 1) * hd]
                    Vj = rows_i[:, (nkv + g) * hd:(nkv + g + 1) * hd]
                    o[i, hq] = attend(q[i, hq], Kj, Vj, 1.0 / np.sqrt(hd))
            if self.record is not None:
                self.record[l] = {"h": h.copy(), "qkv": y.copy(), "q": q.reshape(k, -1).copy(),
                                  "o": o.reshape(k, nq * hd).copy()}
            y = nat.linear_q41(o.reshape(k, nq * hd), W[p + "wo"])
            x = add(x, rmsnorm(y, self.norm[p + "post_attn_norm"], c.eps))
            b = rmsnorm(x, self.norm[p + "pre_ffn_norm"], c.eps)
            a = swiglu(nat.linear_q41(b, W[p + "wgu"]), c.ffn[l])
            y = nat.linear_q41(a, W[p + "wd"])
            x = add(x, rmsnorm(y, self.norm[p + "post_ffn_norm"], c.eps))
            if c.ple_dim:
                P = c.ple_dim
                x = ple_tail(x, ple[:, l * P:(l + 1) * P], W[p + "wple_g"], W[p + "wple_p"],
                             self.norm[p + "ple_norm"], self.lam[l], c.eps)
            if l in self.tap_layers:
                ti = self.tap_layers.index(l)
                taps[:, ti * H:(ti + 1) * H] = x
            if self.record is not None:
                self.record[l]["x"] = x.copy()
        self.last_hidden = x
        self.pending = k
        self.taps = np.concatenate([self.taps, taps])
        return self.head(x if head_rows is None else x[k - head_rows:])

    def head(self, x: np.ndarray) -> np.ndarray:
        return nat.linear_bf16(rmsnorm(x, self.norm["final_norm"], self.cfg.eps), self.W["head"])


# ---- draft -------------------------------------------------------------------------------------------
class Draft:
    """The DFlash draft: context = fc-fused taps of committed positions; a block of [token, mask, ...]
    attends to its context (window) and bidirectionally to itself."""

    def __init__(self, dcfg, W: dict, target_cfg):
        self.cfg = dcfg
        self.tcfg = target_cfg
        self.W = W
        self.norm = {k: nat.bf16_decode(v) for k, v in W.items() if k.endswith("norm")}
        d = dcfg
        self.kv = d.n_kv_heads * d.head_dim
        self.ctx_k = [np.zeros((0, self.kv), F32) for _ in range(d.n_layers)]
        self.ctx_v = [np.zeros((0, self.kv), F32) for _ in range(d.n_layers)]

    @property
    def n_ctx(self) -> int:
        return self.ctx_k[0].shape[0]

    def snapshot(self):
        return copy.deepcopy((self.ctx_k, self.ctx_v))

    def restore(self, snap) -> None:
        self.ctx_k, self.ctx_v = copy.deepcopy(snap)

    def truncate(self, n: int) -> None:
        self.ctx_k = [a[:n].copy() for a in self.ctx_k]
        self.ctx_v = [a[:n].copy() for a in self.ctx_v]

    def context_rows(self, taps: np.ndarray) -> np.ndarray:
        """c_j = RMSNorm_hidden(concat taps_j . fc) for each row of taps."""
        d = self.cfg
        return rmsnorm(nat.linear_bf16(taps, self.W["d.fc"]), self.norm["d.hidden_norm"], d.eps)

    def append_ctx(self, taps: np.ndarray) -> None:
        """Make the rows `taps` (positions n_ctx, n_ctx+1, ...) context: each layer's key and value of
        c_j, with the key normed and rotated at position j."""
        d = self.cfg
        r = taps.shape[0]
        if r == 0:
            return
        pos = self.n_ctx + np.arange(r)
        cb = self.context_rows(taps)
        nq, hd = d.n_heads, d.head_dim
        for l in range(d.n_layers):
            p = f"d{l}."
            Wkv = self.W[p + "wqkv"][nq * hd:]
            y = nat.linear_q41(cb, Wkv)
            kk = y[:, : self.kv].reshape(r, d.n_kv_heads, hd)
            kk = np.stack([rope(rmsnorm(kk[i], self.norm[p + "k_norm"], d.eps), pos[i], d.rope_base) for i in range(r)])
            self.ctx_k[l] = np.concatenate([self.ctx_k[l], kk.reshape(r, -1)])
            self.ctx_v[l] = np.concatenate([self.ctx_v[l], y[:, self.kv:]])

    def block(self, token: int, emb: np.ndarray, head: np.ndarray):
        """Draft block at positions n..n+B-1 (n = context rows held) for rows [token, mask, ...].
        Returns (proposals for positions n+1..n+B-1, their fp32 logits)."""
        d, W = self.cfg, self.W
        B, n = d.block, self.n_ctx
        H, nq, nkv, hd = d.hidden, d.n_heads, d.n_kv_heads, d.head_dim
        toks = np.array([token] + [d.mask_token] * (B - 1), np.int64)
        pos = n + np.arange(B)
        x = (np.asarray(nat.bf16_decode(emb[toks]), F64) * F64(np.float32(d.emb_scale))).astype(F32)
        lo = max(0, n - d.window) if d.window else 0
        grp = nq // nkv
        for l in range(d.n_layers):
            p = f"d{l}."
            h = rmsnorm(x, self.norm[p + "attn_norm"], d.eps)
            y = nat.linear_q41(h, W[p + "wqkv"])
            q = y[:, : nq * hd].reshape(B, nq, hd)
            q = np.stack([rope(rmsnorm(q[i], self.norm[p + "q_norm"], d.eps), pos[i], d.rope_base) for i in range(B)])
            kk = y[:, nq * hd:(nq + nkv) * hd].reshape(B, nkv, hd)
            kk = np.stack([rope(rmsnorm(kk[i], self.norm[p + "k_norm"], d.eps), pos[i], d.rope_base) for i in range(B)])
            Kb = kk.reshape(B, -1)
            Vb = y[:, (nq + nkv) * hd:]
            Kall = np.concatenate([self.ctx_k[l][lo:n], Kb])
            Vall = np.concatenate([self.ctx_v[l][lo:n], Vb])
            o = np.zeros((B, nq, hd), F32)
            for i in range(B):
                for hq in range(nq):
                    g = hq // grp
                    o[i, hq] = attend(q[i, hq], Kall[:, g * hd:(g + 1) * hd], Vall[:, g * hd:(g + 1) * hd],
                                      1.0 / np.sqrt(hd))
            x = add(x, nat.linear_q41(o.reshape(B, -1), W[p + "wo"]))
            b = rmsnorm(x, self.norm[p + "ffn_norm"], d.eps)
            a = swiglu(nat.linear_q41(b, W[p + "wgu"]), d.ffn)
            x = add(x, nat.linear_q41(a, W[p + "wd"]))
        self.last_hidden = x
        logits = nat.linear_bf16(rmsnorm(x[1:], self.norm["d.final_norm"], d.eps), head)
        return np.array([argmax_first(r) for r in logits], np.int32), logits
