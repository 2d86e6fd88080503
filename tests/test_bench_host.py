"""The benchmark's host arithmetic on the CPU: the roofline figures it derives from the in-pass stamps,
the draft block's algorithmic bytes against the closed form of the draft's shapes, and the step loop's
token and acceptance bookkeeping over a stand-in engine."""
import hashlib
import os

import numpy as np
import pytest

import gen

bench = pytest.importorskip("bench")


def _prof(q=(230, 1.86, 3.72e9), f=(1, 0.0143, 1.3e8), h=(2, 0.506, 2.684e9), rest=((47, 0.53, 0), (52, 0.196, 0),
                                                                                      (140, 0.528, 0))):
    return [q, f, h] + list(rest)


def test_roofline_figures():
    """achieved = bytes / summed in-pass time; frac against the given peak; per-launch averages; class
    shares of the step; the rest of the step is what no stamped class covers."""
    steps, ms_step = 1, 3.97
    pk = {"hbm_gbs": 6774.6, "src": "measured"}
    r = bench.roofline(_prof(), steps, ms_step, pk)
    assert r["achieved"] == pytest.approx(3.72e9 / 1.86e-3 / 1e9, rel=1e-3)
    assert r["frac"] == pytest.approx(r["achieved"] / 6774.6, rel=1e-3)
    assert r["frac_vs_8TBs"] == pytest.approx(r["achieved"] / 8000.0, rel=1e-3)
    assert r["launches"] == 230 and r["avg_launch_us"] == pytest.approx(1.86e3 / 230, abs=0.01)
    assert r["bytes_per_launch"] == round(3.72e9 / 230)
    assert r["head"]["achieved"] == pytest.approx(2.684e9 / 0.506e-3 / 1e9, rel=1e-3)
    b = r["breakdown"]
    assert b["q41_products"]["share_of_step"] == pytest.approx(1.86 / 3.97, abs=1e-3)
    total = 1.86 + 0.0143 + 0.506 + 0.53 + 0.196 + 0.528
    assert b["untimed_rest_ms_per_step"] == pytest.approx(3.97 - total, abs=1e-3)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 6774.6


def test_roofline_traffic_only_for_the_captured_source():
    """traffic scales the captured kernel's DRAM / algorithmic ratio to the step's average launch, and is
    null once the product kernel's source no longer hashes to the captured one."""
    pk = {"hbm_gbs": 6774.6, "src": "measured"}
    src = os.path.join(bench.ROOT, "dflash_speculative_decode_gb300", "csrc", "gemm.cu")
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    cap = bench.TRAFFIC_CAPTURE
    r = bench.roofline(_prof(), 1, 3.97, pk)
    if cap["gemm_cu_sha16"] == sha:
        assert r["traffic"] == round(3.72e9 / 230 * cap["dram_bytes"] / cap["algorithmic_bytes"])
    else:
        assert r["traffic"] is None
    saved = dict(cap)
    try:
        cap["gemm_cu_sha16"] = "0" * 16
        assert bench.roofline(_prof(), 1, 3.97, pk)["traffic"] is None
    finally:
        cap.clear()
        cap.update(saved)


def test_draft_block_bytes_closed_form():
    """E4B draft: 5 layers of q|k|v 2560 x (32 + 2 * 8) * 128, o 4096 x 2560, gate|up 2560 x 10240,
    down 5120 x 2560 at 0.625 bytes per weight (204.8 MB), the 2560 x 262144 bf16 head once, and the
    fp32 context planes of at most 1024 rows (5 layers x 2 x 8 heads x 128)."""
    pc = gen.e4b_pair(max_ctx=4160)
    weights = 5 * (2560 * 48 * 128 + 4096 * 2560 + 2560 * 10240 + 5120 * 2560)
    assert weights * 0.625 == pytest.approx(204.8e6, rel=1e-3)
    head = 262144 * 2560 * 2
    for ctx in (30, 1024, 4096):
        kv = 5 * min(ctx, 1024) * 2 * 8 * 128 * 4
        assert bench.draft_block_bytes(pc, ctx) == pytest.approx(weights * 0.625 + head + kv, rel=1e-12)
    assert bench.draft_block_bytes(pc, 4096) == bench.draft_block_bytes(pc, 1024)


class _TruthEngine:
    """Bookkeeping stand-in for run_steps: the target's token for position q is truth[q] whatever the
    rows, proposals come from the planted table, and the calls keep positions held as the ABI does."""

    def __init__(self, truth, block, n0):
        from dflash_speculative_decode_gb300 import DFL_KEEP_ACCEPTED
        self.truth, self.n, self.keep_code = truth, n0, DFL_KEEP_ACCEPTED
        self.cfg = type("cfg", (), {"block": block})()
        self.table = None
        self.pending = None
        self.restores = 0

    def dfl_restore(self, snap):
        self.n = snap
        self.restores += 1

    def dfl_positions_held(self):
        return self.n

    def dfl_draft_block(self, last, want=True):
        return np.zeros(self.cfg.block - 1, np.int32) if want else None

    def dfl_plant_proposals(self, table):
        self.table = table

    def dfl_verify_block(self, rows, k=None):
        n, B = self.n, self.cfg.block
        if rows is None:
            rows = [0] + [int(v) for v in self.table[n + 1:n + B]]
        tt = [int(self.truth[n + i + 1]) for i in range(len(rows))]
        a = 0
        while a < len(rows) - 1 and rows[1 + a] == tt[a]:
            a += 1
        self.pending = a
        return np.asarray(tt, np.int32), a

    def dfl_commit_verify_rows(self, keep):
        assert keep == self.keep_code
        self.n += self.pending + 1
        self.pending = None


@pytest.mark.parametrize("host", [False, True])
def test_run_steps_counts_and_acceptance(host):
    """run_steps counts a + 1 tokens per pass, restarts from the snapshot once a decode has produced
    n_gen tokens, and reports every pass's accepted length; the first proposal's hit rate and the tokens
    per pass match the planted corruption's expectations (1 - p, and 1 + sum_i (1 - p)^i)."""
    B, p, n0, n_gen, steps = 8, 0.3, 40, 512, 3000
    L = n0 + n_gen + 64
    truth = np.random.default_rng(5).integers(0, 1000, size=L + 32).astype(np.int32)
    table = gen.corruption(p, 1000, L + 32).propose(truth, np.arange(L + 32))
    eng = _TruthEngine(truth, B, n0)
    acc = []
    toks = bench.run_steps(eng, None, table, int(truth[n0]), n0, n0, steps, n_gen,
                           host_rows=table if host else None, accepted=acc)
    assert len(acc) == steps and toks == sum(a + 1 for a in acc)
    assert eng.restores >= toks // (n_gen + B) - 1
    st = bench.acceptance(acc, B)
    assert sum(st["histogram"]) == steps == st["passes"]
    assert st["tokens_per_pass"] == pytest.approx(toks / steps, abs=1e-4)
    # the corruption is keyed by position and every decode restarts from the same prefix, so the passes
    # revisit one sample of about 170 pass positions: statistical tolerances of a few standard errors
    assert st["first_proposal_hit_rate"] == pytest.approx(1 - p, abs=0.06)
    assert st["tokens_per_pass"] == pytest.approx(1 + sum((1 - p) ** i for i in range(1, B)), rel=0.08)
