"""Pins of the oracle to facts fixed outside it: exact rational arithmetic, closed forms, a second
independent implementation of a format, published generator outputs and the pages' own numbers.
CPU only."""
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

import gen
import oracle
from oracle import model as om

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append(line.split())
    return rows


def _half_exact(bits: int) -> Fraction:
    """Exact value of an fp16 bit pattern via the struct module's binary16 codec."""
    return Fraction(struct.unpack("<e", struct.pack("<H", bits))[0])


def _block(d_bits, m_bits, codes):
    b = bytearray(struct.pack("<HH", d_bits, m_bits))
    for i in range(16):
        b.append((codes[2 * i] & 15) | ((codes[2 * i + 1] & 15) << 4))
    return np.frombuffer(bytes(b), np.uint8)


# ---- P1: Q4_1 dequantisation ---------------------------------------------------------------------
HALF_GRID = [0x0000, 0x8000, 0x0001, 0x03FF, 0x0400, 0x3C00, 0xBC00, 0x2E66, 0xB4CD, 0x7BFF, 0xFBFF, 0x1234, 0x5140]


def test_q41_dequant_brute_force_exact():
    """Every code 0..15 against a grid of fp16 scales and minimums (zeros, subnormals, negatives,
    the largest finite): w = d*q + m, exact."""
    for d_bits in HALF_GRID:
        for m_bits in HALF_GRID:
            codes = [i % 16 for i in range(32)]
            w = oracle.q41_dequant(_block(d_bits, m_bits, codes))
            d, m = _half_exact(d_bits), _half_exact(m_bits)
            for i in range(32):
                assert Fraction(w[i]) == d * (i % 16) + m, (hex(d_bits), hex(m_bits), i)


def test_q41_nibble_order():
    """Element i sits in byte 4 + i//2, low nibble for even i (a block with q_i = 15 - i%16 and d = 1)."""
    codes = [15 - (i % 16) for i in range(32)]
    w = oracle.q41_dequant(_block(0x3C00, 0x0000, codes))
    assert list(w.astype(int)) == codes
    raw = bytes(_block(0x3C00, 0, codes))
    assert raw[4] == (15 | (14 << 4)) and raw[5] == (13 | (12 << 4))


def test_half_decode_matches_struct():
    bits = np.arange(0, 65536, dtype=np.uint16)
    bits = bits[((bits >> 10) & 31) != 31]           # finite only
    got = oracle.half_decode(bits)
    want = np.array([struct.unpack("<e", struct.pack("<H", int(b)))[0] for b in bits[::97]])
    np.testing.assert_array_equal(got[::97], want)


def test_generator_quantiser_error_bound():
    """Generator packing: every weight is within d/2 of its code's value plus the fp16 rounding of the
    minimum (closed-form bound of the round-to-nearest quantiser)."""
    rng = np.random.default_rng(5)
    w = (rng.standard_normal((64, 256)) * 0.02).astype(np.float32)
    blocks = gen.pack_q41(w)
    deq = oracle.q41_dequant(blocks).reshape(64, 256)
    d = oracle.half_decode(blocks[..., 0:2].copy().view(np.uint16)[..., 0])
    m = oracle.half_decode(blocks[..., 2:4].copy().view(np.uint16)[..., 0])
    mn = w.reshape(64, 8, 32).min(axis=2)
    bound = d / 2 + np.abs(m - mn) + 16 * np.abs(d - (w.reshape(64, 8, 32).max(2) - mn) / 15) + 1e-12
    err = np.abs(deq.reshape(64, 8, 32) - w.reshape(64, 8, 32)).max(axis=2)
    assert (err <= bound).all()


# ---- bf16 rounding: two independent implementations of round-to-nearest-even ---------------------
def test_bf16_round_ties_to_even():
    x = np.array([1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 2 ** -130 * 1.5, 3.0e38], np.float32)
    want = np.array([1.0, 1.0, 1 + 2 ** -6, -1.0, 2 ** -130 * 1.5, 3.0e38], np.float64)
    got = oracle.bf16r(x).astype(np.float64)
    assert got[0] == want[0] and got[1] == want[1] and got[2] == want[2] and got[3] == want[3]
    assert got[4] == np.float32(2 ** -130 * 1.5)          # 1.5 * 2^-130 is a bf16 subnormal
    assert abs(got[5] - want[5]) / want[5] < 2 ** -8


def test_bf16_round_agrees_with_bit_trick():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(200000).astype(np.float32) * 10.0 ** rng.integers(-40, 38, 200000),
                        rng.standard_normal(1000).astype(np.float32) * np.float32(1e-39)]).astype(np.float32)
    a = oracle.bf16r(x)
    b = (gen.bf16_bits(x).astype(np.uint32) << 16).view(np.float32)
    np.testing.assert_array_equal(a, b)


# ---- P2: products ---------------------------------------------------------------------------------
def _deq_numpy(W):
    """Independent dequantisation with numpy's fp16 codec (w = d*q + m in float64)."""
    d = W[..., 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    m = W[..., 2:4].copy().view(np.float16)[..., 0].astype(np.float64)
    lo, hi = W[..., 4:] & 15, W[..., 4:] >> 4
    q = np.empty(W.shape[:-1] + (32,), np.float64)
    q[..., 0::2], q[..., 1::2] = lo, hi
    return (d[..., None] * q + m[..., None]).reshape(W.shape[0], -1)       # [N][K]


def test_linear_one_hot_returns_weight_row_exactly():
    rng = np.random.default_rng(2)
    W = gen.pack_q41((rng.standard_normal((48, 96)) * 0.02).astype(np.float32))
    ref = _deq_numpy(W)
    for k in (0, 1, 31, 32, 95):
        x = np.zeros((1, 96), np.float32)
        x[0, k] = 1.0
        y = oracle.linear_q41(x, W)
        np.testing.assert_array_equal(y[0].astype(np.float64), ref[:, k].astype(np.float32).astype(np.float64))


def test_linear_off_diagonal_catches_transpose():
    """One nonzero weight at (output 3, input 40) of a 64-in x 8-out matrix."""
    w = np.zeros((8, 64), np.float32)
    w[3, 40] = 0.5
    W = gen.pack_q41(w)
    x = np.zeros((2, 64), np.float32)
    x[0, 40] = 2.0
    x[1, 3] = 2.0
    y = oracle.linear_q41(x, W)
    assert y[0, 3] == pytest.approx(1.0, abs=1e-3) and np.count_nonzero(np.abs(y[0]) > 1e-3) == 1
    assert np.all(np.abs(y[1]) < 1e-3)


def test_linear_random_within_fp32_bound():
    rng = np.random.default_rng(3)
    K, N, R = 512, 40, 3
    W = gen.pack_q41((rng.standard_normal((N, K)) * 0.02).astype(np.float32))
    x = oracle.bf16r(rng.standard_normal((R, K)).astype(np.float32))
    ref = x.astype(np.float64) @ _deq_numpy(W).T
    y = oracle.linear_q41(x, W).astype(np.float64)
    bound = 2.0 ** -24 * (np.abs(x.astype(np.float64)) @ np.abs(_deq_numpy(W)).T) + 1e-30
    assert np.all(np.abs(y - ref) <= bound)
    # rows do not depend on the batch
    y1 = oracle.linear_q41(x[1:2], W)
    np.testing.assert_array_equal(y1[0], y[1].astype(np.float32))


def test_linear_bf16_matches_exact():
    rng = np.random.default_rng(4)
    Wb = gen.bf16_bits(rng.standard_normal((30, 70)).astype(np.float32))
    x = oracle.bf16r(rng.standard_normal((2, 70)).astype(np.float32))
    Wf = (Wb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ref = x.astype(np.float64) @ Wf.T
    y = oracle.linear_bf16(x, Wb).astype(np.float64)
    assert np.all(np.abs(y - ref) <= 2.0 ** -24 * np.abs(x.astype(np.float64)) @ np.abs(Wf).T + 1e-30)


# ---- closed forms: norm, rotation, attention ----------------------------------------------------
def test_rmsnorm_constant_vector():
    c, n, eps = 3.0, 64, 1e-6
    w = np.linspace(0.5, 1.5, n).astype(np.float32)
    y = oracle.rmsnorm(np.full(n, c, np.float32), w, eps)
    np.testing.assert_allclose(y, (c / np.sqrt(c * c + eps) * w.astype(np.float64)).astype(np.float32), rtol=0, atol=0)


def test_rope_identity_norm_and_relative_position():
    rng = np.random.default_rng(6)
    v = rng.standard_normal(64).astype(np.float32)
    np.testing.assert_array_equal(oracle.rope(v, 0, 10000.0), v)
    r = oracle.rope(v, 777, 10000.0)
    assert np.linalg.norm(r.astype(np.float64)) == pytest.approx(np.linalg.norm(v.astype(np.float64)), rel=1e-6)
    e0 = np.zeros(64, np.float32)
    e0[0] = 1.0
    r0 = oracle.rope(e0, 5, 10000.0)           # pair (0, 32), angle 5 * base^0 = 5 rad
    assert r0[0] == pytest.approx(np.cos(5.0), abs=1e-7) and r0[32] == pytest.approx(np.sin(5.0), abs=1e-7)
    q, k = rng.standard_normal(64).astype(np.float32), rng.standard_normal(64).astype(np.float32)
    a = np.dot(oracle.rope(q, 100, 1e4).astype(np.float64), oracle.rope(k, 90, 1e4).astype(np.float64))
    b = np.dot(oracle.rope(q, 20, 1e4).astype(np.float64), oracle.rope(k, 10, 1e4).astype(np.float64))
    assert a == pytest.approx(b, rel=1e-5)


def test_attention_closed_forms():
    rng = np.random.default_rng(7)
    q = rng.standard_normal(16).astype(np.float32)
    K1, V1 = rng.standard_normal((1, 16)).astype(np.float32), rng.standard_normal((1, 16)).astype(np.float32)
    np.testing.assert_array_equal(oracle.attend(q, K1, V1, 0.25), V1[0])
    K = np.repeat(K1, 5, axis=0)
    V = rng.standard_normal((5, 16)).astype(np.float32)
    np.testing.assert_allclose(oracle.attend(q, K, V, 0.25), V.astype(np.float64).mean(0), rtol=1e-6, atol=1e-7)


def test_sliding_window_excludes_key_at_p_minus_w():
    """A one-layer all-sliding target: row p's logits ignore the token at p - W and see p - W + 1."""
    base = gen.tiny_pair()
    t = base.target
    t1 = gen.TargetConfig(name="w", n_layers=1, hidden=t.hidden, vocab=t.vocab, n_heads=t.n_heads,
                          head_dim=t.head_dim, layer_type=(0,), kv_heads=(1,), kv_owner=(0,), ffn=(512,), window=8)
    pc = gen.PairConfig(t1, base.draft)
    W = gen.generate(pc, only={s.name for s in gen.target_specs(t1, pc.sigma)})
    toks = list(gen.prompt(t1.vocab, 20))
    p, Wn = 19, 8

    def last_logits(seq):
        tg = om.Target(t1, W)
        return tg.forward(seq)[-1]

    ref = last_logits(toks)
    a = list(toks)
    a[p - Wn] = (a[p - Wn] + 1) % t1.vocab
    np.testing.assert_array_equal(last_logits(a), ref)
    b = list(toks)
    b[p - Wn + 1] = (b[p - Wn + 1] + 1) % t1.vocab
    assert not np.array_equal(last_logits(b), ref)


# ---- sampling -------------------------------------------------------------------------------------
def test_uniform_published_splitmix64_outputs():
    rows = {int(r[0]): int(r[1], 16) for r in _golden("splitmix64_seed0.txt")[1:]}
    for pos in (0, 1, 2):
        assert oracle.uniform(0, pos) == (rows[pos + 1] >> 11) * 2.0 ** -53


def test_sampling_reduces_to_argmax():
    rng = np.random.default_rng(8)
    l = rng.standard_normal(1000).astype(np.float32)
    for u in (0.0, 0.3, 0.999999):
        assert oracle.sample(l, 1e-4, u)[0] == int(np.argmax(l))
    oh = np.full(50, -1e4, np.float32)
    oh[17] = 0.0
    assert oracle.sample(oh, 0.8, 0.5)[0] == 17


def test_sampling_distribution_chi_square():
    """V = 8 toy: 100000 draws with independent uniforms follow softmax(l / T)."""
    from scipy import stats
    l = np.array([0.3, -1.0, 2.0, 0.0, 1.1, -0.4, 0.9, 1.7], np.float32)
    T = 0.8
    p = np.exp((l.astype(np.float64) - l.max()) / T)
    p /= p.sum()
    counts = np.zeros(8)
    for i in range(100000):
        counts[oracle.sample(l, T, oracle.uniform(11, i))[0]] += 1
    chi = stats.chisquare(counts, p * 100000)
    assert chi.pvalue > 1e-3


# ---- P4, P11: width arithmetic and positions held (the pages' numbers) ------------------------------
def test_kv_widths_e4b_match_pages():
    g = {r[0]: int(r[1]) for r in _golden("kv_width_pins.txt")}
    cfg = gen.e4b_target()
    w = oracle.kv_widths(cfg)
    for l in range(cfg.n_layers):
        if not cfg.is_owner(l):
            assert w[l] == g["shared_width"]
        elif cfg.layer_type[l] == gen.FULL:
            assert w[l] == g["full_width"]
        else:
            assert w[l] == g["sliding_width"]
    assert g["prompt_positions"] * g["full_width"] == g["prompt_floats_full_plane"]
    assert [l for l in range(42) if w[l] == 0] == list(range(24, 42))
    assert cfg.kv_owner[24] == 22 and cfg.kv_owner[29] == 23       # last non-shared of the same type


def test_commit_positions_held_pages_example():
    g = {r[0]: int(r[1]) for r in _golden("kv_width_pins.txt")}
    pc = gen.tiny_shared_pair()
    W = gen.generate(pc)
    tg = om.Target(pc.target, W)
    tg.forward(gen.prompt(pc.target.vocab, g["held_before"]))
    tg.commit(g["held_before"])
    tg.forward([1, 2, 3, 4][: g["verify_rows"]])
    tg.commit(g["keep"])
    assert tg.positions_held() == g["held_after"] == tg.n


# ---- P9: acceptance accounting ----------------------------------------------------------------------
def test_acceptance_tool_accounting():
    rows = _golden("acceptance_tool_walk.txt")
    tot = [r for r in rows if r[0] == "total"][0]
    for r in rows:
        if r[0] in ("total", "tokens_per_pass_total"):
            continue
        assert f"{int(r[2]) / int(r[1]):.2f}" == r[3]
    passes, acc = int(tot[1]), int(tot[2])
    assert f"{acc / passes:.2f}" == tot[3]
    tpp = [r for r in rows if r[0] == "tokens_per_pass_total"][0][1]
    assert f"{(acc + passes) / passes:.2f}" == tpp          # each pass also emits the target's token


def test_accept_length_definition():
    assert oracle.accept_length([5, 6, 7], [5, 6, 7]) == 3
    assert oracle.accept_length([5, 6, 7], [5, 9, 7]) == 1
    assert oracle.accept_length([5, 6, 7], [4, 6, 7]) == 0


@pytest.mark.parametrize("p,expect", [(0.1, 5.695), (0.3, 3.141), (0.6, 1.666)])
def test_planted_walk_expected_tokens_per_step(p, expect):
    """A walk over a planted stream (no model): mean tokens per pass = 1 + sum_i (1-p)^i, i = 1..7."""
    L = 200000
    G = np.random.default_rng(9).integers(0, 1 << 30, L + 16)
    cor = gen.corruption(p, 1 << 30, L + 16, seed=21)
    n, passes, toks = 0, 0, 0
    while n < L:
        props = cor.propose(G, np.arange(n + 1, n + 8))
        a = oracle.accept_length(list(props), list(G[n + 1:n + 8]))
        n += a + 1
        passes += 1
        toks += a + 1
    assert toks / passes == pytest.approx(expect, rel=0.02)


# ---- SwiGLU gate and the per-layer-embedding tail --------------------------------------------------
def test_silu_closed_forms():
    """silu(x) = x * sigmoid(x): silu(0) = 0, silu(1) = e / (1 + e), silu(x) - x -> 0 as x -> +inf,
    silu(x) -> 0 as x -> -inf, silu(-x) = silu(x) - x, slope 1/2 at 0. A plain sigmoid, a tanh gate or
    a sign slip fails one of them."""
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    assert oracle.silu(np.array([1.0]))[0] == pytest.approx(np.e / (1.0 + np.e), rel=1e-15)
    big = oracle.silu(np.array([40.0, -40.0]))
    assert abs(big[0] - 40.0) < 1e-12 and abs(big[1]) < 1e-12
    x = np.random.default_rng(12).standard_normal(1000) * 5.0
    np.testing.assert_allclose(oracle.silu(-x), oracle.silu(x) - x, rtol=0, atol=1e-13)
    h = 1e-6
    assert (oracle.silu(np.array([h]))[0] - oracle.silu(np.array([-h]))[0]) / (2 * h) == pytest.approx(0.5, abs=1e-9)


def test_swiglu_gate_is_the_first_half():
    """gate|up: the gate is the first F columns. With gate -20 and up 3 the unit is shut (about -1e-7);
    the halves swapped would give silu(3) * -20 = -57.1. With gate 30 and up 2 it passes 2 * 30."""
    gu = np.array([[-20.0, 3.0], [30.0, 2.0]], np.float32)
    a = oracle.swiglu(gu, 1)
    assert abs(a[0, 0]) < 1e-6
    assert a[1, 0] == pytest.approx(60.0, rel=1e-6)
    assert abs(oracle.swiglu(gu[:, ::-1].copy(), 1)[0, 0] + 57.1) < 0.1   # the swap is visible


def _ple_fixture(seed=13, H=64, P=32):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((3, H)) * 2.0).astype(np.float32)
    p_l = rng.standard_normal((3, P)).astype(np.float32)
    Wg = gen.pack_q41((rng.standard_normal((P, H)) * 0.3).astype(np.float32))
    Wp = gen.pack_q41((rng.standard_normal((H, P)) * 0.3).astype(np.float32))
    w = oracle.bf16_decode(gen.bf16_bits(rng.uniform(0.75, 1.25, H).astype(np.float32)))
    return x, p_l, Wg, Wp, w


def test_ple_tail_order():
    """The PLE tail: gate on the residual stream itself, projection normed BEFORE the add, layer scalar
    AFTER it (1bit engine PR "npu forward: Gemma4 verifies a draft in one batched pass", "What changes":
    PLE gate and projection, then the layer scalar)."""
    x, p_l, Wg, Wp, w = _ple_fixture()
    lam, eps = 0.625, 1e-6
    lam_x = (x.astype(np.float64) * np.float64(np.float32(lam))).astype(np.float32)
    # a zero projection contributes exactly nothing: x * lambda
    Wp0 = gen.pack_q41(np.zeros((x.shape[1], p_l.shape[1]), np.float32))
    np.testing.assert_array_equal(oracle.ple_tail(x, p_l, Wg, Wp0, w, lam, eps), lam_x)
    # a zero norm weight also gives x * lambda: the norm applies to the projection before the add
    # (a norm after the add would give zero)
    np.testing.assert_array_equal(oracle.ple_tail(x, p_l, Wg, Wp, np.zeros_like(w), lam, eps), lam_x)
    # lambda after the add: halving lambda halves the result exactly
    full = oracle.ple_tail(x, p_l, Wg, Wp, w, 1.0, eps)
    np.testing.assert_array_equal(oracle.ple_tail(x, p_l, Wg, Wp, w, 0.5, eps), (full * np.float32(0.5)))
    # the gate reads x itself, not a normed copy: the added term changes when x is scaled
    d1 = full.astype(np.float64) - x
    d2 = oracle.ple_tail(2 * x, p_l, Wg, Wp, w, 1.0, eps).astype(np.float64) - 2 * x.astype(np.float64)
    assert np.abs(d1 - d2).max() > 1e-2
    # the token's per-layer row multiplies the gate: a zero row adds nothing
    np.testing.assert_array_equal(oracle.ple_tail(x, np.zeros_like(p_l), Wg, Wp, w, 1.0, eps), x)


def test_products_do_not_depend_on_thread_count():
    """The oracle's products split only independent output columns over threads: one thread and all
    threads give the same bits (so the CPU baseline may use any count)."""
    rng = np.random.default_rng(17)
    W = gen.pack_q41((rng.standard_normal((96, 256)) * 0.02).astype(np.float32))
    x = rng.standard_normal((3, 256)).astype(np.float32)
    n = oracle.threads()
    try:
        oracle.set_threads(1)
        a = oracle.linear_q41(x, W)
    finally:
        oracle.set_threads(n)
    np.testing.assert_array_equal(a, oracle.linear_q41(x, W))
