"""The model configuration's file form: every pair survives pair_to_json / pair_from_json unchanged, the
library sees the same dfl_config and sizes from the document as from the pair, and malformed documents
are refused."""
import ctypes
import json

import pytest

import gen
from dflash_speculative_decode_gb300._abi import config_from_pair, dfl_sizes, lib


@pytest.mark.parametrize("name", sorted(gen.PAIRS) + ["27b-cut"])
def test_round_trip_and_library_view(name):
    pc = gen.b27_cut() if name == "27b-cut" else gen.PAIRS[name]()
    back = gen.pair_from_json(gen.pair_to_json(pc))
    assert back == pc
    a, b = config_from_pair(pc, prefill_rows=128), config_from_pair(back, prefill_rows=128)
    assert bytes(a) == bytes(b)
    L = lib()
    sa, sb = dfl_sizes(), dfl_sizes()
    assert L.dfl_required_bytes(ctypes.byref(a), ctypes.byref(sa)) == 0
    assert L.dfl_required_bytes(ctypes.byref(b), ctypes.byref(sb)) == 0
    assert bytes(sa) == bytes(sb)


def test_layer_types_are_named():
    d = json.loads(gen.pair_to_json(gen.e4b_pair()))
    assert d["target"]["layer_type"][:6] == ["sliding"] * 5 + ["full"]
    assert d["draft"]["taps"] == [5, 11, 17, 23, 35]


def test_malformed_documents_are_refused():
    d = json.loads(gen.pair_to_json(gen.tiny_pair()))
    bad_type = json.loads(json.dumps(d))
    bad_type["target"]["layer_type"][0] = "local"
    with pytest.raises(ValueError):
        gen.pair_from_json(json.dumps(bad_type))
    extra = json.loads(json.dumps(d))
    extra["draft"]["heads"] = 4
    with pytest.raises(TypeError):
        gen.pair_from_json(json.dumps(extra))
    missing = json.loads(json.dumps(d))
    del missing["target"]["window"]
    with pytest.raises(TypeError):
        gen.pair_from_json(json.dumps(missing))
