"""ctypes binding of include/dfl.h: the same names, argument marshalling only.

Every step of the decode runs in libdfl.so's CUDA kernels. PyTorch is used here only to allocate the
caller-owned device buffers and to hand over the current CUDA stream. Loading fails loudly when the
library has not been built: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdfl.so")

MAX_LAYERS, MAX_TAPS, MAX_ROWS = 64, 8, 16
DFL_OK, DFL_E_INVALID_ARG, DFL_E_STATE, DFL_E_CAPACITY, DFL_E_UNSUPPORTED, DFL_E_CUDA, DFL_E_TIMEOUT = 0, -1, -2, -3, -4, -5, -6
DFL_KEEP_ACCEPTED = -1
DFL_OPT_KEEP_LOGITS, DFL_OPT_GRAPHS, DFL_OPT_STOP_LAYER, DFL_OPT_PROFILE, DFL_OPT_ATTN_CLUSTER = 1, 2, 3, 4, 5
DFL_OPT_TEST_STALL, DFL_OPT_FUSE_STEPS, DFL_OPT_PLE_SPLIT = 6, 7, 8
ERRORS = {DFL_E_INVALID_ARG: "DFL_E_INVALID_ARG", DFL_E_STATE: "DFL_E_STATE", DFL_E_CAPACITY: "DFL_E_CAPACITY",
          DFL_E_UNSUPPORTED: "DFL_E_UNSUPPORTED", DFL_E_CUDA: "DFL_E_CUDA", DFL_E_TIMEOUT: "DFL_E_TIMEOUT"}


class dfl_config(ctypes.Structure):
    _fields_ = [
        ("n_layers", ctypes.c_int32), ("hidden", ctypes.c_int32), ("vocab", ctypes.c_int32),
        ("n_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("window", ctypes.c_int32),
        ("ple_dim", ctypes.c_int32),
        ("layer_type", ctypes.c_int32 * MAX_LAYERS), ("kv_heads", ctypes.c_int32 * MAX_LAYERS),
        ("kv_owner", ctypes.c_int32 * MAX_LAYERS), ("ffn", ctypes.c_int32 * MAX_LAYERS),
        ("rope_base_sliding", ctypes.c_float), ("rope_base_full", ctypes.c_float), ("eps", ctypes.c_float),
        ("emb_scale", ctypes.c_float),
        ("d_layers", ctypes.c_int32), ("d_ffn", ctypes.c_int32), ("d_heads", ctypes.c_int32),
        ("d_kv_heads", ctypes.c_int32), ("d_head_dim", ctypes.c_int32), ("d_window", ctypes.c_int32),
        ("block", ctypes.c_int32), ("n_taps", ctypes.c_int32), ("mask_token", ctypes.c_int32),
        ("taps", ctypes.c_int32 * MAX_TAPS),
        ("d_rope_base", ctypes.c_float), ("d_eps", ctypes.c_float), ("d_emb_scale", ctypes.c_float),
        ("max_ctx", ctypes.c_int32), ("prefill_rows", ctypes.c_int32),
    ]


class dfl_sizes(ctypes.Structure):
    _fields_ = [("weights_bytes", ctypes.c_uint64), ("state_bytes", ctypes.c_uint64),
                ("workspace_bytes", ctypes.c_uint64)]


class dfl_buffers(ctypes.Structure):
    _fields_ = [("weights", ctypes.c_void_p), ("state", ctypes.c_void_p), ("workspace", ctypes.c_void_p)]


class dfl_sampling(ctypes.Structure):
    _fields_ = [("temperature", ctypes.c_float), ("seed", ctypes.c_uint64)]


P = ctypes.POINTER
i32p = P(ctypes.c_int32)
vp = ctypes.c_void_p

# name -> (restype, argtypes); every entry point declared in include/dfl.h
SIGNATURES = {
    "dfl_required_bytes": (ctypes.c_int, [P(dfl_config), P(dfl_sizes)]),
    "dfl_init": (ctypes.c_int, [P(dfl_config), P(dfl_buffers), vp, P(vp)]),
    "dfl_load_tensor": (ctypes.c_int, [vp, ctypes.c_char_p, vp, ctypes.c_size_t]),
    "dfl_prefill": (ctypes.c_int, [vp, i32p, ctypes.c_int, P(dfl_sampling), i32p]),
    "dfl_draft_block": (ctypes.c_int, [vp, ctypes.c_int32, i32p]),
    "dfl_verify_block": (ctypes.c_int, [vp, i32p, ctypes.c_int, P(dfl_sampling), i32p, i32p]),
    "dfl_commit_verify_rows": (ctypes.c_int, [vp, ctypes.c_int]),
    "dfl_commit_accepted": (ctypes.c_int, [vp, ctypes.c_int, ctypes.c_int32, i32p, i32p]),
    "dfl_snapshot_bytes": (ctypes.c_int64, [vp]),
    "dfl_snapshot": (ctypes.c_int, [vp, vp, ctypes.c_size_t]),
    "dfl_restore": (ctypes.c_int, [vp, vp, ctypes.c_size_t]),
    "dfl_kv_widths": (ctypes.c_int, [vp, i32p]),
    "dfl_positions_held": (ctypes.c_int64, [vp]),
    "dfl_set_option": (ctypes.c_int, [vp, ctypes.c_int, ctypes.c_int]),
    "dfl_read_logits": (ctypes.c_int, [vp, ctypes.c_int, P(ctypes.c_float), ctypes.c_int]),
    "dfl_read_taps": (ctypes.c_int, [vp, ctypes.c_int, ctypes.c_int, P(ctypes.c_float)]),
    "dfl_draft_append_taps": (ctypes.c_int, [vp, vp, ctypes.c_int]),
    "dfl_debug_read": (ctypes.c_int, [vp, ctypes.c_char_p, vp, ctypes.c_size_t]),
    "dfl_plant_proposals": (ctypes.c_int, [vp, vp, ctypes.c_int]),
    "dfl_launch_count": (ctypes.c_int64, [vp]),
    "dfl_profile_read": (ctypes.c_int, [vp, ctypes.c_int, P(ctypes.c_int64), P(ctypes.c_double), P(ctypes.c_double)]),
    "dfl_last_error": (ctypes.c_char_p, [vp]),
    "dfl_destroy": (None, [vp]),
    "dfl_q41_image_bytes": (ctypes.c_int64, [ctypes.c_int, ctypes.c_int]),
    "dfl_q41_pack": (ctypes.c_int, [vp, ctypes.c_int, ctypes.c_int, vp, vp]),
    "dfl_act_bytes": (ctypes.c_int64, [ctypes.c_int, ctypes.c_int]),
    "dfl_act_pack": (ctypes.c_int, [vp, ctypes.c_int, ctypes.c_int, vp, vp]),
    "dfl_q41_gemm_scratch_bytes": (ctypes.c_int64, [ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "dfl_q41_gemm": (ctypes.c_int, [vp, ctypes.c_int, ctypes.c_int, vp, ctypes.c_int, vp, vp, ctypes.c_size_t, vp]),
    "dfl_q41_gemm_status": (ctypes.c_int, [vp, vp]),
    "dfl_q41_gemm_tc_scratch_bytes": (ctypes.c_int64, [ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "dfl_q41_gemm_tc": (ctypes.c_int, [vp, ctypes.c_int, ctypes.c_int, vp, ctypes.c_int, vp, vp, ctypes.c_size_t, vp]),
    "dfl_bf16_image_bytes": (ctypes.c_int64, [ctypes.c_int, ctypes.c_int]),
    "dfl_bf16_pack": (ctypes.c_int, [vp, ctypes.c_int, ctypes.c_int, vp, vp]),
    "dfl_bf16_head_scratch_bytes": (ctypes.c_int64, [ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "dfl_bf16_head_argmax": (ctypes.c_int, [vp, ctypes.c_int, ctypes.c_int, vp, ctypes.c_int, vp, vp, vp,
                                            ctypes.c_size_t, vp]),
    "dfl_q41_gemm_noalloc": (ctypes.c_int, [vp, ctypes.c_int, ctypes.c_int, vp, ctypes.c_int, vp, vp]),
    "dfl_q41_gemm_noalloc_max_scratch": (ctypes.c_int64, []),
    "dfl_q41_gemm_noalloc_status": (ctypes.c_int, [vp]),
    "dfl_q41_gemm_noalloc_reset": (ctypes.c_int, [vp]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library. Raises when libdfl.so is missing (build it with build.py / build())."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libdfl.so is not built ({LIB_PATH}); run dflash_speculative_decode_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


class DflError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code


def config_from_pair(pc, prefill_rows: int = 0) -> dfl_config:
    """dfl_config from a pair description (attributes as in the seeded generator's PairConfig);
    prefill_rows > 0 lets dfl_prefill take that many prompt rows per pass on the tcgen05 products."""
    t, d = pc.target, pc.draft
    c = dfl_config()
    c.n_layers, c.hidden, c.vocab = t.n_layers, t.hidden, t.vocab
    c.n_heads, c.head_dim, c.window, c.ple_dim = t.n_heads, t.head_dim, t.window, t.ple_dim
    for l in range(t.n_layers):
        c.layer_type[l], c.kv_heads[l], c.kv_owner[l], c.ffn[l] = t.layer_type[l], t.kv_heads[l], t.kv_owner[l], t.ffn[l]
    c.rope_base_sliding, c.rope_base_full, c.eps, c.emb_scale = t.rope_base_sliding, t.rope_base_full, t.eps, t.emb_scale
    c.d_layers, c.d_ffn, c.d_heads, c.d_kv_heads, c.d_head_dim = d.n_layers, d.ffn, d.n_heads, d.n_kv_heads, d.head_dim
    c.d_window, c.block, c.n_taps, c.mask_token = d.window, d.block, len(d.taps), d.mask_token
    for i, l in enumerate(d.taps):
        c.taps[i] = l
    c.d_rope_base, c.d_eps, c.d_emb_scale = d.rope_base, d.eps, d.emb_scale
    c.max_ctx = pc.max_ctx
    c.prefill_rows = prefill_rows
    return c


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(i32p)


def _sampling(temperature, seed):
    if temperature is None or temperature <= 0:
        return None
    s = dfl_sampling()
    s.temperature, s.seed = float(temperature), int(seed) & 0xFFFFFFFFFFFFFFFF
    return ctypes.byref(s)


class Engine:
    """One dfl context over torch-allocated device buffers on the current CUDA stream."""

    def __init__(self, cfg: dfl_config, device="cuda:0"):
        import torch
        self.torch = torch
        self.L = lib()
        self.cfg = cfg
        sz = dfl_sizes()
        self._check(self.L.dfl_required_bytes(ctypes.byref(cfg), ctypes.byref(sz)), "dfl_required_bytes")
        self.sizes = sz
        self.device = torch.device(device)
        mk = lambda n: torch.empty(max(int(n), 256), dtype=torch.uint8, device=self.device)
        self.bw, self.bs, self.bx = mk(sz.weights_bytes), mk(sz.state_bytes), mk(sz.workspace_bytes)
        bufs = dfl_buffers(self.bw.data_ptr(), self.bs.data_ptr(), self.bx.data_ptr())
        self.stream = torch.cuda.current_stream(self.device)
        ctx = ctypes.c_void_p()
        self._check(self.L.dfl_init(ctypes.byref(cfg), ctypes.byref(bufs), ctypes.c_void_p(self.stream.cuda_stream),
                                    ctypes.byref(ctx)), "dfl_init")
        self.ctx = ctx

    def _check(self, rc, what):
        if rc != DFL_OK:
            msg = self.L.dfl_last_error(self.ctx).decode() if getattr(self, "ctx", None) else what
            raise DflError(rc, f"{what}: {msg}")

    def close(self):
        if getattr(self, "ctx", None):
            self.L.dfl_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---- tensors ----
    def load_tensor(self, name: str, arr: np.ndarray):
        t = self.torch.from_numpy(np.ascontiguousarray(arr).view(np.uint8).reshape(-1)).to(self.device, non_blocking=False)
        self._check(self.L.dfl_load_tensor(self.ctx, name.encode(), ctypes.c_void_p(t.data_ptr()), t.numel()),
                    f"dfl_load_tensor({name})")
        self.stream.synchronize()

    def load(self, tensors):
        for name, arr in (tensors.items() if hasattr(tensors, "items") else tensors):
            self.load_tensor(name, arr)

    # ---- the step ----
    def dfl_prefill(self, tokens, temperature=None, seed=0) -> int:
        t = _i32(tokens)
        out = np.zeros(1, np.int32)
        self._check(self.L.dfl_prefill(self.ctx, _ptr(t), len(t), _sampling(temperature, seed), _ptr(out)), "dfl_prefill")
        return int(out[0])

    def dfl_draft_block(self, last_tok: int, want=True):
        out = np.zeros(max(self.cfg.block - 1, 1), np.int32)
        self._check(self.L.dfl_draft_block(self.ctx, int(last_tok), _ptr(out) if want else None), "dfl_draft_block")
        return out[: self.cfg.block - 1] if want else None

    def dfl_verify_block(self, rows, k=None, temperature=None, seed=0):
        if rows is None:
            r, kk = None, int(k)
        else:
            r = _i32(rows)
            kk = len(r)
        tt = np.zeros(kk, np.int32)
        acc = np.zeros(1, np.int32)
        self._check(self.L.dfl_verify_block(self.ctx, _ptr(r) if r is not None else None, kk,
                                            _sampling(temperature, seed), _ptr(tt), _ptr(acc)), "dfl_verify_block")
        return tt, int(acc[0])

    def dfl_commit_verify_rows(self, keep: int):
        self._check(self.L.dfl_commit_verify_rows(self.ctx, int(keep)), "dfl_commit_verify_rows")

    def dfl_commit_accepted(self, max_keep: int, stop_token: int = -1):
        """Returns the rows kept; with a stop token, (kept, stopped)."""
        kept = np.zeros(1, np.int32)
        stopped = np.zeros(1, np.int32)
        self._check(self.L.dfl_commit_accepted(self.ctx, int(max_keep), int(stop_token), _ptr(kept), _ptr(stopped)),
                    "dfl_commit_accepted")
        return int(kept[0]) if stop_token < 0 else (int(kept[0]), bool(stopped[0]))

    def dfl_snapshot_bytes(self) -> int:
        return int(self.L.dfl_snapshot_bytes(self.ctx))

    def dfl_snapshot(self):
        n = self.dfl_snapshot_bytes()
        buf = self.torch.empty(n, dtype=self.torch.uint8, device=self.device)
        self._check(self.L.dfl_snapshot(self.ctx, ctypes.c_void_p(buf.data_ptr()), n), "dfl_snapshot")
        return buf

    def dfl_restore(self, buf):
        self._check(self.L.dfl_restore(self.ctx, ctypes.c_void_p(buf.data_ptr()), buf.numel()), "dfl_restore")

    def dfl_kv_widths(self) -> np.ndarray:
        out = np.zeros(self.cfg.n_layers, np.int32)
        self._check(self.L.dfl_kv_widths(self.ctx, _ptr(out)), "dfl_kv_widths")
        return out

    def dfl_positions_held(self) -> int:
        return int(self.L.dfl_positions_held(self.ctx))

    def dfl_set_option(self, option: int, value: int):
        self._check(self.L.dfl_set_option(self.ctx, option, value), "dfl_set_option")

    def dfl_read_logits(self, which: int, rows: int) -> np.ndarray:
        out = np.zeros((rows, self.cfg.vocab), np.float32)
        self._check(self.L.dfl_read_logits(self.ctx, which, out.ctypes.data_as(P(ctypes.c_float)), rows), "dfl_read_logits")
        return out

    def dfl_read_taps(self, pos0: int, rows: int) -> np.ndarray:
        out = np.zeros((rows, self.cfg.n_taps * self.cfg.hidden), np.float32)
        self._check(self.L.dfl_read_taps(self.ctx, pos0, rows, out.ctypes.data_as(P(ctypes.c_float))), "dfl_read_taps")
        return out

    def dfl_debug_read(self, name: str, shape, dtype) -> np.ndarray:
        out = np.zeros(shape, dtype)
        self._check(self.L.dfl_debug_read(self.ctx, name.encode(), out.ctypes.data_as(vp), out.nbytes), "dfl_debug_read")
        return out

    def dfl_plant_proposals(self, table_dev):
        self._check(self.L.dfl_plant_proposals(self.ctx, ctypes.c_void_p(table_dev.data_ptr()), table_dev.numel()),
                    "dfl_plant_proposals")

    def dfl_launch_count(self) -> int:
        return int(self.L.dfl_launch_count(self.ctx))

    def dfl_profile_read(self, cls: int):
        n, ms, by = ctypes.c_int64(), ctypes.c_double(), ctypes.c_double()
        self._check(self.L.dfl_profile_read(self.ctx, cls, ctypes.byref(n), ctypes.byref(ms), ctypes.byref(by)),
                    "dfl_profile_read")
        return n.value, ms.value, by.value

    def dfl_draft_append_taps(self, taps_dev):
        rows = taps_dev.shape[0]
        self._check(self.L.dfl_draft_append_taps(self.ctx, ctypes.c_void_p(taps_dev.data_ptr()), rows),
                    "dfl_draft_append_taps")
