"""Seeded synthetic models and token streams for the DFlash speculative-decode step.

This module only draws random numbers and stores them in the formats the step reads:
Q4_1 blocks (fp16 scale d, fp16 minimum m, 32 four-bit codes) for the layer matrices, and
bf16 bit patterns for embeddings, norms, the draft's fc and the per-layer-embedding table.
It holds none of the step's arithmetic (no dequantisation, no linear algebra, no sampling),
so the CUDA path and the oracle can both read what it writes without sharing any code.

Shapes follow the pages' E4B pair: the model card "Nemotron-3.5-Bolt-E4B-DFlash-NPU2" (spec
table: draft of 5 Qwen3-style layers, hidden 2560, FFN 5120, 32 query / 8 key-value heads of 128,
attention window 1024, block 8, taps at target layers 5, 11, 17, 23, 35; "Q4_1 (5 bits per
weight with scales and minimums)") and the 1bit engine PR "Gemma4 verifies a draft in one
batched pass" ("What changes": sliding vs full KV widths, KV-shared layers, per-layer
embeddings, double-wide MLP on shared layers).
"""
from __future__ import annotations

import json
import zlib
from dataclasses import asdict, dataclass, field, replace
from typing import Dict, Iterator, Optional, Tuple

import numpy as np

SLIDING, FULL = 0, 1
QBLOCK = 32            # Q4_1 block length along the reduction dimension
QBLOCK_BYTES = 20      # fp16 d, fp16 m, 16 bytes of codes

SEED_WEIGHTS, SEED_PROMPT, SEED_CORRUPT, SEED_SAMPLE = 0, 1, 2, 3


# ----------------------------------------------------------------------------------------------
# configurations
# ----------------------------------------------------------------------------------------------
@dataclass(frozen=True)
class TargetConfig:
    name: str
    n_layers: int
    hidden: int
    vocab: int
    n_heads: int                 # query heads (every layer)
    head_dim: int
    layer_type: Tuple[int, ...]  # SLIDING / FULL per layer
    kv_heads: Tuple[int, ...]    # key-value heads per layer
    kv_owner: Tuple[int, ...]    # layer whose plane a layer reads; == l for a layer with its own plane
    ffn: Tuple[int, ...]         # FFN width per layer
    window: int                  # sliding window (keys visible, including the query's own position)
    rope_base_sliding: float = 10000.0
    rope_base_full: float = 1000000.0
    ple_dim: int = 0             # per-layer-embedding width (0: none, and no layer scalar)
    eps: float = 1e-6
    emb_scale: float = 1.0
    norm_init: str = "ones"      # "ones" or "random" (U[0.75, 1.25])

    def is_owner(self, l: int) -> bool:
        return self.kv_owner[l] == l

    def kv_width(self, l: int) -> int:
        """Floats per position in layer l's own plane (0 for a KV-shared layer, which holds none)."""
        return 2 * self.kv_heads[l] * self.head_dim if self.is_owner(l) else 0


@dataclass(frozen=True)
class DraftConfig:
    n_layers: int
    hidden: int
    ffn: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    window: int                  # context keys visible to a block (0: unlimited)
    block: int
    taps: Tuple[int, ...]        # target layers whose outputs feed fc, ascending
    mask_token: int
    rope_base: float = 1000000.0
    eps: float = 1e-6
    emb_scale: float = 1.0
    norm_init: str = "ones"


@dataclass(frozen=True)
class PairConfig:
    target: TargetConfig
    draft: DraftConfig
    max_ctx: int = 4096          # positions the KV arena holds
    r_max: int = 16              # rows one verify or prefill chunk may carry
    sigma: float = 0.02          # std of the Q4_1 layer matrices before packing
    fc_sigma: float = 0.02


def _layer_types_e4b(n: int) -> Tuple[int, ...]:
    # five sliding layers, then one full layer
    return tuple(FULL if l % 6 == 5 else SLIDING for l in range(n))


def _owners(types, first_shared: int) -> Tuple[int, ...]:
    """A KV-shared layer reads the plane of the last non-shared layer of the same attention type."""
    owners = []
    for l, t in enumerate(types):
        if l < first_shared:
            owners.append(l)
        else:
            cand = [j for j in range(first_shared) if types[j] == t]
            if not cand:
                raise ValueError(f"layer {l}: no non-shared layer of type {t}")
            owners.append(cand[-1])
    return tuple(owners)


def tiny_pair() -> PairConfig:
    """4 target layers (0-2 sliding, window 64; 3 full), hidden 256, 4 query heads of 64, vocab 2048;
    a 1-layer draft fusing taps of target layers 1 and 3."""
    types = (SLIDING, SLIDING, SLIDING, FULL)
    t = TargetConfig(
        name="tiny", n_layers=4, hidden=256, vocab=2048, n_heads=4, head_dim=64,
        layer_type=types, kv_heads=tuple(1 if x == SLIDING else 2 for x in types),
        kv_owner=(0, 1, 2, 3), ffn=(512,) * 4, window=64)
    d = DraftConfig(n_layers=1, hidden=256, ffn=512, n_heads=4, n_kv_heads=1, head_dim=64,
                    window=0, block=8, taps=(1, 3), mask_token=2047)
    return PairConfig(t, d, max_ctx=256, r_max=16)


def tiny_shared_pair() -> PairConfig:
    """6 layers: 0, 1, 3 sliding, 2 full; layer 4 (sliding) reads layer 3's plane, layer 5 (full) reads
    layer 2's; PLE width 32; double-wide MLP on 4-5; random norms and non-unit embedding scales."""
    types = (SLIDING, SLIDING, FULL, SLIDING, SLIDING, FULL)
    t = TargetConfig(
        name="tiny-shared", n_layers=6, hidden=256, vocab=2048, n_heads=4, head_dim=64,
        layer_type=types, kv_heads=tuple(1 if x == SLIDING else 2 for x in types),
        kv_owner=_owners(types, 4), ffn=(512, 512, 512, 512, 1024, 1024), window=16,
        ple_dim=32, emb_scale=0.75, norm_init="random")
    d = DraftConfig(n_layers=2, hidden=256, ffn=512, n_heads=4, n_kv_heads=2, head_dim=64,
                    window=24, block=8, taps=(1, 3, 5), mask_token=2047, emb_scale=1.25,
                    norm_init="random")
    return PairConfig(t, d, max_ctx=256, r_max=16)


def e4b_target(n_layers: int = 42, first_shared: int = 24, vocab: int = 262144) -> TargetConfig:
    types = _layer_types_e4b(n_layers)
    owners = _owners(types, first_shared)
    return TargetConfig(
        name="e4b", n_layers=n_layers, hidden=2560, vocab=vocab, n_heads=12, head_dim=256,
        layer_type=types, kv_heads=tuple(1 if x == SLIDING else 2 for x in types),
        kv_owner=owners,
        ffn=tuple(10240 if owners[l] == l else 20480 for l in range(n_layers)),
        window=512, ple_dim=256)


def e4b_draft(vocab: int = 262144) -> DraftConfig:
    return DraftConfig(n_layers=5, hidden=2560, ffn=5120, n_heads=32, n_kv_heads=8, head_dim=128,
                       window=1024, block=8, taps=(5, 11, 17, 23, 35), mask_token=vocab - 1)


def e4b_pair(max_ctx: int = 2048) -> PairConfig:
    """The E4B-shaped pair: 42 target layers (5 sliding : 1 full, layers 24-41 KV-shared with a
    double-wide MLP, PLE 256 per layer, vocab 262144) and the 5-layer draft."""
    return PairConfig(e4b_target(), e4b_draft(), max_ctx=max_ctx, r_max=16)


def b27_target(n_layers: int = 62, vocab: int = 262144) -> TargetConfig:
    """A 27B-class dense target: hidden 5376, 32 query heads of 128 over 16 key-value heads in every
    layer, FFN 21504, five sliding layers (window 1024) to one full layer, no KV sharing and no PLE
    (about 25.6e9 layer weights, 16 GB as Q4_1)."""
    types = _layer_types_e4b(n_layers)
    return TargetConfig(
        name="27b", n_layers=n_layers, hidden=5376, vocab=vocab, n_heads=32, head_dim=128,
        layer_type=types, kv_heads=(16,) * n_layers, kv_owner=tuple(range(n_layers)),
        ffn=(21504,) * n_layers, window=1024)


def b27_draft(vocab: int = 262144, taps: Tuple[int, ...] = (1, 16, 31, 46, 61)) -> DraftConfig:
    """The draft for the 27B-class target: five layers at the target's width (32/8 heads of 128, FFN
    twice the width), fusing five taps spread evenly over the target's depth."""
    return DraftConfig(n_layers=5, hidden=5376, ffn=10752, n_heads=32, n_kv_heads=8, head_dim=128,
                       window=1024, block=8, taps=taps, mask_token=vocab - 1)


def b27_pair(max_ctx: int = 2048) -> PairConfig:
    """The 27B-class pair: 62 dense target layers and the 5-layer draft, vocab 262144."""
    return PairConfig(b27_target(), b27_draft(), max_ctx=max_ctx, r_max=16)


def b27_cut(max_ctx: int = 256, n_layers: int = 6, vocab: int = 32768) -> PairConfig:
    """Six layers of the 27B-class target (five sliding, one full) at full per-layer shapes with vocab
    32768, and the full draft tapping layers 1..5: every product shape of the 27B pair at a size the
    oracle runs in seconds."""
    t = b27_target(n_layers=n_layers, vocab=vocab)
    d = b27_draft(vocab=vocab, taps=tuple(range(1, n_layers)))
    return PairConfig(t, d, max_ctx=max_ctx, r_max=16)


PAIRS = {"tiny": tiny_pair, "tiny-shared": tiny_shared_pair, "e4b": e4b_pair, "27b": b27_pair}

_TYPE_NAMES = {SLIDING: "sliding", FULL: "full"}


def pair_to_json(pc: PairConfig) -> str:
    """The pair's configuration as one JSON document (layer types by name), the file form of a model
    that config_from_pair mirrors into the library's dfl_config; pair_from_json reads it back."""
    d = asdict(pc)
    d["target"]["layer_type"] = [_TYPE_NAMES[t] for t in pc.target.layer_type]
    return json.dumps(d, indent=1)


def pair_from_json(text: str) -> PairConfig:
    """A PairConfig from pair_to_json's document. Unknown or missing fields and unknown layer types are
    refused (TypeError, ValueError) rather than defaulted."""
    d = json.loads(text)
    names = {v: k for k, v in _TYPE_NAMES.items()}
    t = dict(d.pop("target"))
    bad = [v for v in t.get("layer_type", []) if v not in names]
    if bad:
        raise ValueError(f"unknown layer types {bad}")
    t["layer_type"] = tuple(names[v] for v in t["layer_type"])
    for k in ("kv_heads", "kv_owner", "ffn"):
        t[k] = tuple(int(v) for v in t[k])
    dr = dict(d.pop("draft"))
    dr["taps"] = tuple(int(v) for v in dr["taps"])
    return PairConfig(TargetConfig(**t), DraftConfig(**dr), **d)


# ----------------------------------------------------------------------------------------------
# storage formats
# ----------------------------------------------------------------------------------------------
def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (the storage format of bf16 tensors)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)


def pack_q41(w: np.ndarray) -> np.ndarray:
    """Pack a float32 matrix [N out][K in] as Q4_1 blocks of 32 along K: uint8 [N][K/32][20].

    Block layout (little-endian): bytes 0-1 fp16 scale d, bytes 2-3 fp16 minimum m, bytes 4-19 the
    32 codes, element i in byte 4 + i//2, low nibble for even i, high nibble for odd i.
    Codes: d = (max - min) / 15 and m = min, both rounded to fp16; q = clamp(rint((x - m) / d), 0, 15)
    computed with the rounded d and m (q = 0 when d = 0)."""
    N, K = w.shape
    if K % QBLOCK:
        raise ValueError("K must be a multiple of 32")
    b = np.ascontiguousarray(w, dtype=np.float32).reshape(N, K // QBLOCK, QBLOCK)
    mn = b.min(axis=2)
    mx = b.max(axis=2)
    d16 = ((mx - mn) / np.float32(15.0)).astype(np.float16)
    m16 = mn.astype(np.float16)
    d = d16.astype(np.float32)
    m = m16.astype(np.float32)
    inv = np.where(d > 0, np.float32(1.0) / np.where(d > 0, d, np.float32(1.0)), np.float32(0.0))
    q = np.rint((b - m[..., None]) * inv[..., None])
    q = np.clip(q, 0, 15).astype(np.uint8)
    out = np.empty((N, K // QBLOCK, QBLOCK_BYTES), np.uint8)
    out[..., 0:2] = d16.view(np.uint8).reshape(N, K // QBLOCK, 2)
    out[..., 2:4] = m16.view(np.uint8).reshape(N, K // QBLOCK, 2)
    out[..., 4:] = q[..., 0::2] | (q[..., 1::2] << np.uint8(4))
    return out


# ----------------------------------------------------------------------------------------------
# tensors
# ----------------------------------------------------------------------------------------------
@dataclass(frozen=True)
class TensorSpec:
    name: str
    kind: str                 # "q41" (shape = (N, K)), "bf16", "norm", "scalar"
    shape: Tuple[int, ...]
    sigma: float = 1.0


def target_specs(t: TargetConfig, sigma: float) -> list:
    H, hd, nq = t.hidden, t.head_dim, t.n_heads
    # the embedding table and the output head are two tensors (the draft shares both); the head's
    # scale gives logits of standard deviation about 2 for a unit-RMS final hidden state
    specs = [TensorSpec("emb", "bf16", (t.vocab, H), 1.0), TensorSpec("head", "bf16", (t.vocab, H), 2.0 / H ** 0.5),
             TensorSpec("final_norm", "norm", (H,))]
    if t.ple_dim:
        specs.append(TensorSpec("ple_table", "bf16", (t.vocab, t.n_layers * t.ple_dim), 1.0))
    for l in range(t.n_layers):
        p = f"t{l}."
        nkv = t.kv_heads[l]
        specs += [TensorSpec(p + "attn_norm", "norm", (H,)), TensorSpec(p + "q_norm", "norm", (hd,)),
                  TensorSpec(p + "post_attn_norm", "norm", (H,)),
                  TensorSpec(p + "pre_ffn_norm", "norm", (H,)), TensorSpec(p + "post_ffn_norm", "norm", (H,))]
        if t.is_owner(l):
            specs += [TensorSpec(p + "k_norm", "norm", (hd,)),
                      TensorSpec(p + "wqkv", "q41", ((nq + 2 * nkv) * hd, H), sigma)]
        else:
            specs.append(TensorSpec(p + "wq", "q41", (nq * hd, H), sigma))
        specs += [TensorSpec(p + "wo", "q41", (H, nq * hd), sigma),
                  TensorSpec(p + "wgu", "q41", (2 * t.ffn[l], H), sigma),
                  TensorSpec(p + "wd", "q41", (H, t.ffn[l]), sigma)]
        if t.ple_dim:
            specs += [TensorSpec(p + "wple_g", "q41", (t.ple_dim, H), sigma),
                      TensorSpec(p + "wple_p", "q41", (H, t.ple_dim), sigma),
                      TensorSpec(p + "ple_norm", "norm", (H,)),
                      TensorSpec(p + "lambda", "scalar", (1,))]
    return specs


def draft_specs(d: DraftConfig, sigma: float, fc_sigma: float) -> list:
    H, hd = d.hidden, d.head_dim
    T = len(d.taps)
    specs = [TensorSpec("d.fc", "bf16", (H, T * H), fc_sigma), TensorSpec("d.hidden_norm", "norm", (H,)),
             TensorSpec("d.final_norm", "norm", (H,))]
    for l in range(d.n_layers):
        p = f"d{l}."
        specs += [TensorSpec(p + "attn_norm", "norm", (H,)), TensorSpec(p + "q_norm", "norm", (hd,)),
                  TensorSpec(p + "k_norm", "norm", (hd,)), TensorSpec(p + "ffn_norm", "norm", (H,)),
                  TensorSpec(p + "wqkv", "q41", ((d.n_heads + 2 * d.n_kv_heads) * hd, H), sigma),
                  TensorSpec(p + "wo", "q41", (H, d.n_heads * hd), sigma),
                  TensorSpec(p + "wgu", "q41", (2 * d.ffn, H), sigma),
                  TensorSpec(p + "wd", "q41", (H, d.ffn), sigma)]
    return specs


def pair_specs(pc: PairConfig) -> list:
    return target_specs(pc.target, pc.sigma) + draft_specs(pc.draft, pc.sigma, pc.fc_sigma)


_ROW_CHUNK = 1 << 13   # rows per independently seeded chunk of a large bf16 table / Q4_1 matrix


def _rng(seed: int, name: str, chunk: int = 0) -> np.random.Generator:
    return np.random.default_rng([seed, zlib.crc32(name.encode()), chunk])


def make_rows(spec: TensorSpec, seed: int, r0: int, r1: int, norm_init: str = "ones") -> np.ndarray:
    """Rows [r0, r1) of a tensor (rows = first dimension); r0 must be a multiple of the chunk size."""
    if spec.kind in ("norm", "scalar"):
        rng = _rng(seed, spec.name)
        n = spec.shape[0]
        if spec.kind == "scalar":
            v = rng.uniform(0.5, 1.0, size=n).astype(np.float32)       # layer scalar in [0.5, 1)
        elif norm_init == "random":
            v = rng.uniform(0.75, 1.25, size=n).astype(np.float32)
        else:
            v = np.ones(n, np.float32)
        return bf16_bits(v)[r0:r1]
    if r0 % _ROW_CHUNK:
        raise ValueError("row ranges must start on a chunk boundary")
    cols = int(np.prod(spec.shape[1:]))
    parts = []
    for c0 in range(r0, r1, _ROW_CHUNK):
        c1 = min(c0 + _ROW_CHUNK, r1, spec.shape[0])
        rng = _rng(seed, spec.name, c0 // _ROW_CHUNK)
        full = min(c0 + _ROW_CHUNK, spec.shape[0]) - c0
        x = rng.standard_normal((full, cols), dtype=np.float32)[: c1 - c0]
        x *= np.float32(spec.sigma)
        parts.append(pack_q41(x) if spec.kind == "q41" else bf16_bits(x))
    return np.concatenate(parts) if len(parts) > 1 else parts[0]


def make_tensor(spec: TensorSpec, seed: int = SEED_WEIGHTS, norm_init: str = "ones") -> np.ndarray:
    return make_rows(spec, seed, 0, spec.shape[0], norm_init)


def _norm_kind(pc: PairConfig, name: str) -> str:
    return pc.draft.norm_init if name.startswith("d") else pc.target.norm_init


def _job(args):
    spec, seed, r0, r1, ni = args
    return spec.name, r0, make_rows(spec, seed, r0, r1, ni)


def generate(pc: PairConfig, seed: int = SEED_WEIGHTS, workers: int = 1,
             only: Optional[set] = None) -> Dict[str, np.ndarray]:
    """All tensors of a pair, by name. Deterministic for any worker count."""
    out: Dict[str, np.ndarray] = {}
    for name, arr in iter_tensors(pc, seed, workers, only):
        out[name] = arr
    return out


def iter_tensors(pc: PairConfig, seed: int = SEED_WEIGHTS, workers: int = 1,
                 only: Optional[set] = None) -> Iterator[Tuple[str, np.ndarray]]:
    """Yield (name, array) for every tensor; large tensors are built in row chunks, in parallel when
    workers > 1 (a spawn pool, safe to start before or after CUDA is initialised)."""
    specs = [s for s in pair_specs(pc) if only is None or s.name in only]
    jobs, sizes = [], {}
    for s in specs:
        ni = _norm_kind(pc, s.name)
        rows = s.shape[0]
        if s.kind in ("norm", "scalar") or rows <= _ROW_CHUNK:
            jobs.append((s, seed, 0, rows, ni))
            sizes[s.name] = 1
        else:
            n = 0
            for r0 in range(0, rows, _ROW_CHUNK):
                jobs.append((s, seed, r0, min(r0 + _ROW_CHUNK, rows), ni))
                n += 1
            sizes[s.name] = n
    if workers <= 1:
        pending: Dict[str, list] = {}
        for j in jobs:
            name, r0, arr = _job(j)
            pending.setdefault(name, []).append((r0, arr))
            if len(pending[name]) == sizes[name]:
                yield name, _join(pending.pop(name))
        return
    import multiprocessing as mp
    from concurrent.futures import ProcessPoolExecutor
    with ProcessPoolExecutor(max_workers=workers, mp_context=mp.get_context("spawn")) as ex:
        pending = {}
        for name, r0, arr in ex.map(_job, jobs, chunksize=1):
            pending.setdefault(name, []).append((r0, arr))
            if len(pending[name]) == sizes[name]:
                yield name, _join(pending.pop(name))


def _join(parts):
    parts.sort(key=lambda p: p[0])
    return parts[0][1] if len(parts) == 1 else np.concatenate([p[1] for p in parts])


# ----------------------------------------------------------------------------------------------
# token streams
# ----------------------------------------------------------------------------------------------
def prompt(vocab: int, length: int, seed: int = SEED_PROMPT, request: int = 0) -> np.ndarray:
    """A prompt of token ids uniform over the vocabulary."""
    rng = np.random.default_rng([seed, 1 + request])
    return rng.integers(0, vocab, size=length, dtype=np.int64).astype(np.int32)


@dataclass
class Corruption:
    """Per-position corruption of a planted draft: position q is replaced when hit[q], by repl[q]."""
    hit: np.ndarray
    repl: np.ndarray

    def propose(self, greedy: np.ndarray, positions: np.ndarray) -> np.ndarray:
        """The planted proposal for each absolute position: the target's own token unless corrupted."""
        g = greedy[positions]
        return np.where(self.hit[positions], self.repl[positions], g).astype(np.int32)


def corruption(p: float, vocab: int, length: int, seed: int = SEED_CORRUPT, request: int = 0) -> Corruption:
    rng = np.random.default_rng([seed, 1 + request])
    u = rng.random(length)
    repl = rng.integers(0, vocab, size=length, dtype=np.int64).astype(np.int32)
    return Corruption(hit=u < p, repl=repl)


def fc_taps(n_rows: int, width: int, seed: int = SEED_PROMPT) -> np.ndarray:
    """Tapped target features N(0, 1) as float32 [n_rows][width] (the draft-alone workload)."""
    rng = np.random.default_rng([seed, 77])
    return rng.standard_normal((n_rows, width), dtype=np.float32)


def activations(m: int, k: int, seed: int) -> np.ndarray:
    """GEMM activations N(0, 1) as bf16 bits [m][k] (the isolated GEMM sweep)."""
    rng = np.random.default_rng([seed, 99])
    return bf16_bits(rng.standard_normal((m, k), dtype=np.float32))
