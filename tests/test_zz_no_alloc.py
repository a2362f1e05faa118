"""GPU: the allocation-free entry point.

pa_prefill_noalloc serves callers that may not call cudaMalloc (an engine
that has reserved nearly all device memory for its own KV-cache pool, or a
latency-critical path where an allocation is not allowed).  Its scratch is a
static device array shared by every call, so these tests call it several
times in a row, on different shapes, and check each output against the
handle-based entry point.  Both run the same widening and attention kernels
on the same work units (each unit's output depends on that unit alone), so
the outputs are equal bit for bit; a wrong stride in how the static array is
carved up would show as a difference.  The file is named so that pytest
collects it last.
"""
import ctypes as C

import numpy as np
import pytest

from pa_testutil import TOL_MAX, TOL_MEAN, norm_errors, run_gpu, to_device
from synth import CONFIGS, make_inputs
from synth.workloads import Workload

pytestmark = pytest.mark.gpu


def call_noalloc(inp, S, W):
    """One pa_prefill_noalloc call through the C ABI; returns (out, status)."""
    import torch

    import windowed_prefill_attention_gb300 as pa
    wl = inp.wl
    q_off, q_start, n_q, n_ctx = inp.seq_desc[0].tolist()
    d = to_device(inp)
    out = torch.full_like(d["q"], float("nan"))
    ptr = lambda t: C.c_void_p(t.data_ptr())  # noqa: E731
    rc = pa._lib.pa_prefill_noalloc(wl.n_q_heads, wl.n_kv_heads, inp.k_pool.shape[0], inp.block_table.shape[1],
                                    ptr(d["q"]), ptr(d["k_pool"]), ptr(d["v_pool"]), ptr(d["k_scale"]),
                                    ptr(d["v_scale"]), ptr(d["block_table"]), q_start, n_q, n_ctx, S, W,
                                    C.c_float(wl.sm_scale), ptr(out),
                                    C.c_void_p(torch.cuda.current_stream().cuda_stream))
    return out.float().cpu().numpy(), rc


CASES = [
    (CONFIGS["4k"], 1, 256),
    (Workload("na_win", 16, 2, ((1003, 1517),), 1, 8, seed=71, outlier_frac=0.02), 1, 8),
    (CONFIGS["tiny"], 0, 16),
]


def test_noalloc_matches_handle_entry_point_on_consecutive_calls():
    for wl, S, W in CASES + CASES[:1]:
        inp = make_inputs(wl)
        ref, rc_ref = run_gpu(inp, S=S, W=W)
        assert rc_ref == 0
        for _ in range(2):
            got, rc = call_noalloc(inp, S, W)
            assert rc == 0
            assert np.isfinite(got).all()
            mx, mean = norm_errors(got.astype(np.float64), ref.astype(np.float64))
            assert mx <= TOL_MAX and mean <= TOL_MEAN, (wl.name, mx, mean)
            assert np.array_equal(got, ref), wl.name


def test_noalloc_work_list_has_the_planner_order():
    """The work list the ordering kernel builds on the device is pa_plan's, unit
    for unit (longest first, ties by first token then kv head)."""
    import windowed_prefill_attention_gb300 as pa
    for wl, S, W in CASES:
        inp = make_inputs(wl)
        _, rc = call_noalloc(inp, S, W)
        assert rc == 0
        want, _, _ = pa.pa_plan(wl.n_q_heads, wl.n_kv_heads, inp.seq_desc, S, W)
        got = pa.pa_debug_noalloc_units(len(want))
        assert np.array_equal(got, want), wl.name
        assert np.all(np.diff(got[:, 3]) <= 0)  # decreasing key tiles


def test_noalloc_rejects_contexts_beyond_its_scratch():
    import windowed_prefill_attention_gb300 as pa
    inp = make_inputs(CONFIGS["tiny"])
    wl = inp.wl
    d = to_device(inp)
    ptr = lambda t: C.c_void_p(t.data_ptr())  # noqa: E731
    # a 64k-token context needs ~130 MB of widened rows, far beyond the array
    big = 65536
    rc = pa._lib.pa_prefill_noalloc(wl.n_q_heads, wl.n_kv_heads, inp.k_pool.shape[0], big // 16, ptr(d["q"]),
                                    ptr(d["k_pool"]), ptr(d["v_pool"]), ptr(d["k_scale"]), ptr(d["v_scale"]),
                                    ptr(d["block_table"]), 0, big, big, 0, 0, C.c_float(0.0625), ptr(d["q"]), None)
    assert rc == pa.PA_ENOSCRATCH
    assert "scratch" in pa.pa_strerror(rc)
    # positions past 2^30 are rejected before any arithmetic on them
    for q_start, n_q, n_ctx in ((2 ** 30 - 5, 10, 2 ** 30 + 5), (2 ** 31 - 8, 4, 2 ** 31 - 1)):
        rc = pa._lib.pa_prefill_noalloc(wl.n_q_heads, wl.n_kv_heads, inp.k_pool.shape[0], 2 ** 27,
                                        ptr(d["q"]), ptr(d["k_pool"]), ptr(d["v_pool"]), ptr(d["k_scale"]),
                                        ptr(d["v_scale"]), ptr(d["block_table"]), q_start, n_q, n_ctx, 0, 0,
                                        C.c_float(0.0625), ptr(d["q"]), None)
        assert rc == pa.PA_EINVAL, (q_start, rc)
