"""The error path of a prefill: a prefill over held positions whose bounded waits give up (the test
option DFL_OPT_TEST_STALL, no fault) leaves the context refusing work until a snapshot is restored.
Collected after the parity files (file name)."""
import numpy as np
import pytest

import gen

pytestmark = pytest.mark.gpu


def test_failed_prefill_refuses_until_restore():
    """A prefill over held positions whose passes give up (DFL_OPT_TEST_STALL) returns DFL_E_TIMEOUT with
    positions held unchanged. Its 40 rows are more than the sliding rings' slack (window + 15 slots), so
    the passes that ran overwrote ring slots of the held window: the context then refuses passes and
    snapshots (DFL_E_STATE) until a restore, after which it matches a context that never failed. A failed
    prefill into an empty context needs no restore."""
    from dflash_speculative_decode_gb300 import DFL_OPT_KEEP_LOGITS, DflError
    from dflash_speculative_decode_gb300._abi import DFL_E_STATE, DFL_E_TIMEOUT, DFL_OPT_TEST_STALL
    from gpu_harness import engine
    pc = gen.tiny_pair()
    W = gen.generate(pc)
    V = pc.target.vocab
    prompt = gen.prompt(V, 90, request=31)
    more = gen.prompt(V, 40, request=32)
    rows = [int(t) for t in gen.prompt(V, 8, request=33)]
    a = engine(pc, W)
    a.dfl_set_option(DFL_OPT_KEEP_LOGITS, 1)
    a.dfl_prefill(prompt)
    snap = a.dfl_snapshot()
    a.dfl_set_option(DFL_OPT_TEST_STALL, 1)
    with pytest.raises(DflError) as ei:
        a.dfl_prefill(more)
    assert ei.value.code == DFL_E_TIMEOUT
    assert a.dfl_positions_held() == 90
    a.dfl_set_option(DFL_OPT_TEST_STALL, 0)
    for call in (lambda: a.dfl_verify_block(rows), lambda: a.dfl_prefill(more), lambda: a.dfl_draft_block(rows[0]),
                 lambda: a.dfl_snapshot()):
        with pytest.raises(DflError) as ei:
            call()
        assert ei.value.code == DFL_E_STATE
    a.dfl_restore(snap)
    tt_a, acc_a = a.dfl_verify_block(rows)
    b = engine(pc, W)
    b.dfl_set_option(DFL_OPT_KEEP_LOGITS, 1)
    b.dfl_prefill(prompt)
    tt_b, acc_b = b.dfl_verify_block(rows)
    np.testing.assert_array_equal(a.dfl_read_logits(0, 8), b.dfl_read_logits(0, 8))
    assert list(tt_a) == list(tt_b) and acc_a == acc_b
    # an empty context: the failed prefill leaves nothing to protect, the next prefill runs
    e = engine(pc, W)
    e.dfl_set_option(DFL_OPT_TEST_STALL, 1)
    with pytest.raises(DflError) as ei:
        e.dfl_prefill(more)
    assert ei.value.code == DFL_E_TIMEOUT and e.dfl_positions_held() == 0
    e.dfl_set_option(DFL_OPT_TEST_STALL, 0)
    e.dfl_set_option(DFL_OPT_KEEP_LOGITS, 1)
    e.dfl_prefill(prompt)
    tt_e, _ = e.dfl_verify_block(rows)
    np.testing.assert_array_equal(e.dfl_read_logits(0, 8), b.dfl_read_logits(0, 8))
