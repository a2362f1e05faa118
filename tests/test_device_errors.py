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


def test_host_path_drains_its_copies_before_returning_an_error():
    """pa_prefill_host on the 32k workload (about 300 MB of pinned input, a
    millisecond or more of copies) with the test hook that fails the call
    while it is still enqueuing, after the pool's and the first chunks'
    copies were issued: the call returns PA_ECUDA only once both copy streams
    are idle, so none of them still reads the caller's buffers.  The handle
    then serves a normal call with the same result as the device entry point."""
    import torch

    import windowed_prefill_attention_gb300 as pa
    from synth import CONFIGS, make_inputs
    inp = make_inputs(CONFIGS["32k"])
    wl = inp.wl
    pin = lambda a: torch.from_numpy(a).pin_memory()  # noqa: E731
    hq = torch.from_numpy(inp.q.view(np.int16)).pin_memory()
    hk, hv, hks, hvs, hbt = (pin(inp.k_pool), pin(inp.v_pool), pin(inp.k_scale), pin(inp.v_scale),
                             pin(inp.block_table))
    hout = torch.empty_like(hq).pin_memory()
    args = (inp.seq_desc, hq, hk, hv, hks, hvs, hbt, wl.n_sink_blk, wl.n_win_blk, wl.sm_scale, hout)
    h = pa.pa_create(wl.n_q_heads, wl.n_kv_heads, inp.k_pool.shape[0], inp.block_table.shape[1],
                     debug_fail_host=True)
    try:
        for _ in range(2):
            with pytest.raises(pa.PAError) as ei:
                pa.pa_prefill_host(h, *args)
            assert ei.value.code == pa.PA_ECUDA
            assert pa.pa_debug_copy_streams_idle(h)
    finally:
        pa.pa_destroy(h)
    h = pa.pa_create(wl.n_q_heads, wl.n_kv_heads, inp.k_pool.shape[0], inp.block_table.shape[1])
    try:
        pa.pa_prefill_host(h, *args)
        assert pa.pa_debug_copy_streams_idle(h)
    finally:
        pa.pa_destroy(h)
    b = hout.view(torch.bfloat16).float().numpy()
    a, rc = run_gpu(inp)
    assert rc == 0 and np.array_equal(a, b)
