"""CPU: the C-ABI library builds, loads without a GPU, and exports every entry point include/dfl.h
declares; the Python binding names the same set."""
import ctypes
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "dfl.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dfl_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    from dflash_speculative_decode_gb300 import build
    path = build.build()
    L = ctypes.CDLL(path)
    names = _declared()
    assert len(names) >= 20
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing


def test_binding_covers_header():
    from dflash_speculative_decode_gb300 import _abi
    assert sorted(_abi.SIGNATURES) == _declared()


def test_required_bytes_without_gpu():
    """Size planning is host arithmetic: it runs without a device."""
    import gen
    from dflash_speculative_decode_gb300 import _abi
    L = _abi.lib()
    for pc in (gen.tiny_pair(), gen.tiny_shared_pair(), gen.e4b_pair()):
        cfg = _abi.config_from_pair(pc)
        sz = _abi.dfl_sizes()
        assert L.dfl_required_bytes(ctypes.byref(cfg), ctypes.byref(sz)) == 0
        assert sz.weights_bytes > 0 and sz.state_bytes > 0 and sz.workspace_bytes > 0
    e4b = _abi.config_from_pair(gen.e4b_pair())
    sz = _abi.dfl_sizes()
    L.dfl_required_bytes(ctypes.byref(e4b), ctypes.byref(sz))
    # Q4_1 layer weights (0.625 B/weight) + bf16 embedding, head, PLE table and fc
    assert 11.5e9 < sz.weights_bytes < 13.5e9


def test_required_bytes_27b_and_long_prefill():
    """The 27B-class pair fits the part (16 GB of Q4_1 layers + bf16 tables); long prefill passes add
    their row buffers, product scratch and longer sliding rings, and bad prefill_rows are refused."""
    import gen
    from dflash_speculative_decode_gb300 import _abi
    L = _abi.lib()
    sz = _abi.dfl_sizes()
    cfg = _abi.config_from_pair(gen.b27_pair())
    assert L.dfl_required_bytes(ctypes.byref(cfg), ctypes.byref(sz)) == 0
    assert 21e9 < sz.weights_bytes < 24e9
    base = (sz.state_bytes, sz.workspace_bytes)
    cfg = _abi.config_from_pair(gen.b27_pair(), prefill_rows=1024)
    assert L.dfl_required_bytes(ctypes.byref(cfg), ctypes.byref(sz)) == 0
    assert sz.state_bytes > base[0] and sz.workspace_bytes > base[1]
    assert sz.weights_bytes + sz.state_bytes + sz.workspace_bytes < 60e9
    for bad in (100, 130, 8208, -16):
        cfg = _abi.config_from_pair(gen.tiny_pair(), prefill_rows=bad)
        assert L.dfl_required_bytes(ctypes.byref(cfg), ctypes.byref(sz)) == _abi.DFL_E_INVALID_ARG, bad
    cfg = _abi.config_from_pair(gen.tiny_pair())
    cfg.hidden = 8320                          # past the widest row step
    assert L.dfl_required_bytes(ctypes.byref(cfg), ctypes.byref(sz)) == _abi.DFL_E_INVALID_ARG


def test_tc_scratch_sizes():
    from dflash_speculative_decode_gb300 import _abi
    L = _abi.lib()
    Kp = 2560
    assert L.dfl_q41_gemm_tc_scratch_bytes(2560, 10240, 2048) == 1024 + 2 * 10240 * Kp * 2 + 2 * 2048 * Kp * 2
    assert L.dfl_q41_gemm_tc_scratch_bytes(96, 64, 1) == 1024 + 2 * 64 * 128 * 2 + 2 * 1024   # K padded to 128
    assert L.dfl_q41_gemm_tc_scratch_bytes(2560, 48, 128) == -1    # N not a multiple of 32
    assert L.dfl_q41_gemm_tc_scratch_bytes(2560, 64, 0) == -1


def test_bad_configuration_is_refused():
    import gen
    from dflash_speculative_decode_gb300 import _abi
    L = _abi.lib()
    sz = _abi.dfl_sizes()
    cfg = _abi.config_from_pair(gen.tiny_pair())
    cfg.kv_owner[2] = 3                       # a later layer cannot own an earlier layer's plane
    assert L.dfl_required_bytes(ctypes.byref(cfg), ctypes.byref(sz)) == _abi.DFL_E_INVALID_ARG
    cfg = _abi.config_from_pair(gen.tiny_pair())
    cfg.block = 17
    assert L.dfl_required_bytes(ctypes.byref(cfg), ctypes.byref(sz)) == _abi.DFL_E_INVALID_ARG
    cfg = _abi.config_from_pair(gen.tiny_shared_pair())
    cfg.kv_owner[5] = 3                       # owner of another attention type
    assert L.dfl_required_bytes(ctypes.byref(cfg), ctypes.byref(sz)) == _abi.DFL_E_INVALID_ARG


def test_q41_sizes():
    from dflash_speculative_decode_gb300 import _abi
    L = _abi.lib()
    assert L.dfl_q41_image_bytes(2560, 4096) == 2560 * 4096 * 5 // 8
    assert L.dfl_q41_image_bytes(32, 64) == 64 * 64 * 5 // 8      # K padded to 64
    assert L.dfl_q41_image_bytes(30, 64) == -1
    assert L.dfl_q41_gemm_scratch_bytes(2560, 4096, 17) == -1


def test_binding_constants_match_header():
    """Every enum constant of include/dfl.h that the binding names has the header's value."""
    from dflash_speculative_decode_gb300 import _abi
    src = open(os.path.join(ROOT, "include", "dfl.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    header = {}
    for body in re.findall(r"enum\s*\{(.*?)\}", src, flags=re.S):
        for name, val in re.findall(r"\b(DFL_[A-Z0-9_]+)\s*=\s*(-?\d+)", body):
            header[name] = int(val)
    assert {"DFL_OPT_KEEP_LOGITS", "DFL_OPT_PROFILE", "DFL_OPT_ATTN_CLUSTER", "DFL_E_INVALID_ARG"} <= set(header)
    named = {n: getattr(_abi, n) for n in header if hasattr(_abi, n)}
    assert len(named) >= 8
    assert all(named[n] == header[n] for n in named), {n: (named[n], header[n]) for n in named if named[n] != header[n]}
