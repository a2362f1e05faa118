"""GPU: failures come back as status codes and leave the context usable.

No test here faults or hangs the GPU: a block-table entry outside the pool
is caught by the widening kernel's range check before any access, and the
timeout case uses the test hook that points the kernel's first wait at a
barrier nothing arrives at, so the bounded wait runs out and every thread
exits through the normal teardown."""
import numpy as np
import pytest

from pa_testutil import run_gpu, to_device
from synth.workloads import Workload

pytestmark = pytest.mark.gpu

WL = Workload("err", 16, 2, ((0, 640),), 1, 8, seed=61)


def test_bad_block_table_entry_reports_bad_page_then_recovers():
    from synth import make_inputs
    inp = make_inputs(WL)
    good, rc = run_gpu(inp)
    assert rc == 0
    inp.block_table = inp.block_table.copy()
    inp.block_table[0, 3] = inp.k_pool.shape[0] + 5
    _, rc = run_gpu(inp)
    import windowed_prefill_attention_gb300 as pa
    assert rc == pa.PA_EBADPAGE
    inp.block_table[0, 3] = -7
    _, rc = run_gpu(inp)
    assert rc == pa.PA_EBADPAGE


def test_timeout_is_reported_and_context_stays_usable():
    import torch

    import windowed_prefill_attention_gb300 as pa
    from synth import make_inputs
    inp = make_inputs(WL)
    d = to_device(inp)
    out = torch.zeros_like(d["q"])
    h = pa.pa_create(16, 2, inp.k_pool.shape[0], inp.block_table.shape[1], wait_timeout_ms=20, debug_stall=True)
    try:
        pa.pa_prefill_batch(h, inp.seq_desc, d["q"], d["k_pool"], d["v_pool"], d["k_scale"], d["v_scale"],
                            d["block_table"], 1, 8, WL.sm_scale, out)
        assert pa.pa_last_error(h) == pa.PA_ETIMEOUT
        assert pa.pa_last_error(h) == pa.PA_OK  # cleared
    finally:
        pa.pa_destroy(h)
    good, rc = run_gpu(inp)
    assert rc == 0 and np.isfinite(good).all()


def test_invalid_calls_are_rejected_before_launch():
    import torch

    import windowed_prefill_attention_gb300 as pa
    from synth import make_inputs
    inp = make_inputs(WL)
    d = to_device(inp)
    out = torch.zeros_like(d["q"])
    h = pa.pa_create(16, 2, inp.k_pool.shape[0], inp.block_table.shape[1])
    args = (d["q"], d["k_pool"], d["v_pool"], d["k_scale"], d["v_scale"], d["block_table"])
    try:
        with pytest.raises(pa.PAError):           # empty query range
            pa.pa_prefill(h, *args, 0, 0, 640, 1, 8, 0.0625, out)
        with pytest.raises(pa.PAError):           # queries past the context
            pa.pa_prefill(h, *args, 600, 100, 640, 1, 8, 0.0625, out)
        with pytest.raises(pa.PAError):           # context longer than the block table row
            pa.pa_prefill(h, *args, 0, 640, 640 + 16 * 200, 1, 8, 0.0625, out)
        with pytest.raises(pa.PAError):           # misaligned output
            pa.pa_prefill(h, *args, 0, 640, 640, 1, 8, 0.0625, out.view(-1)[1:1 + out.numel() - 8])
        with pytest.raises(pa.PAError):           # NaN softmax scale
            pa.pa_prefill(h, *args, 0, 640, 640, 1, 8, float("nan"), out)
        assert pa.pa_last_error(h) == pa.PA_OK
    finally:
        pa.pa_destroy(h)
