"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Every workload of the benchmark at full size (sampled rows for the long
ones), in the launch configuration bench.py times (pa_prefill_batch), plus
edge cases of the mask and the shapes.  The bar is the stated tolerance:
max |err| <= 3e-2 * max(1, |ref|) and mean |err| / max(1, |ref|) <= 1e-2.

A tighter check compares against the oracle's walk through the method's
own quantisation steps, so a kernel bug hidden inside the quantisation
budget still shows.  Its bound comes from the arithmetic: the output is
rounded to bf16, whose 8-bit significand has unit roundoff 2^-8 ~ 3.9e-3
(relative, so at most 3.9e-3 after normalising by max(1, |ref|)); P' is
rounded to fp16 on both sides, where the two roundings differ (the GPU's
running max lags by up to 2^8 and its V-scale normaliser shifts P'), each
adding <= 2^-11 * sum_j p_j |V_j| / l, about 2^-11 on data without outliers;
the fp32 accumulation adds ~1e-6.  So 5e-3 on the max and 5e-4 on the mean,
on workloads without outliers.  With outlier tokens (K and V x8) the sum of
|p_j V_j| reaches ~8x the output scale and cancels, so the fp16 rounding
noise of the two sides alone reaches ~1e-2 and this comparison resolves no
more than the one against the definition; it is not run there.
On the u8 grid a code may flip by one where the GPU's fp32 exp and the
oracle's fp64 exp straddle a rounding boundary (1/255 of the tile's largest
P' times one value), hence 1.5e-2 / 1e-3 there.
"""
import dataclasses

import numpy as np
import pytest

import oracle
from pa_testutil import TOL_MAX, TOL_MEAN, compare, norm_errors, run_gpu, sample_rows
from synth import CONFIGS, make_inputs
from synth.workloads import Workload

pytestmark = pytest.mark.gpu

# keys per tile of the kernel: the u8 grid of P' is per row and per tile
KEY_TILE = 128

FULL = {
    "tiny": None,       # all rows
    "4k": 600,          # random tokens (x all heads) plus edges
    "32k": 256,
    "64k": 192,
    "chunked": 256,
    "chunked_ragged": 256,
}


@pytest.fixture(scope="module")
def inputs():
    cache = {}

    def get(name):
        if name not in cache:
            cache[name] = make_inputs(CONFIGS[name])
        return cache[name]
    return get


# Errors measured on GB300 with the default containers (max / mean normalised
# error on each workload's sampled rows).  Besides the pages' bound, each
# workload must stay within 2.5x of its own record, so that an accuracy
# regression far inside that bound still shows.
RECORDED = {
    "tiny": (4.0e-3, 2.0e-4),
    "4k": (4.1e-3, 7.6e-5),
    "32k": (7.2e-3, 1.3e-3),
    "64k": (7.8e-3, 1.3e-3),
    "chunked": (7.7e-3, 1.3e-3),
    "chunked_ragged": (7.7e-3, 1.3e-3),
}
REGRESSION_FACTOR = 2.5


@pytest.mark.parametrize("name", list(FULL))
def test_default_mode_matches_oracle(name, inputs):
    inp = inputs(name)
    out, rc = run_gpu(inp)
    assert rc == 0
    rows = oracle.all_rows(inp) if FULL[name] is None else sample_rows(inp, FULL[name])
    mx, mean = compare(out, inp, rows)
    print("%s: max %.3g mean %.3g over %d rows" % (name, mx, mean, len(rows)))
    assert mx <= TOL_MAX and mean <= TOL_MEAN
    rec_max, rec_mean = RECORDED[name]
    assert mx <= REGRESSION_FACTOR * rec_max and mean <= REGRESSION_FACTOR * rec_mean, (name, mx, mean)
    # rows outside every query range are never written: every output row is finite
    assert np.isfinite(out).all()


CLEAN_CHUNKED = dataclasses.replace(CONFIGS["chunked_ragged"], name="chunked_clean", outlier_frac=0.0)


@pytest.mark.parametrize("name", ["tiny", "4k", "chunked_clean"])
def test_default_mode_matches_method_steps(name, inputs):
    inp = inputs(name) if name != "chunked_clean" else make_inputs(CLEAN_CHUNKED)
    out, rc = run_gpu(inp)
    assert rc == 0
    rows = oracle.all_rows(inp) if name == "tiny" else sample_rows(inp, 200)
    ref = oracle.method(oracle.Problem.from_inputs(inp), rows, oracle.Q_LOSSLESS, oracle.P_F16, tile=KEY_TILE)
    mx, mean = norm_errors(out[rows[:, 0], rows[:, 1]].astype(np.float64), ref)
    print("%s vs method: max %.3g mean %.3g" % (name, mx, mean))
    assert mx <= 5e-3 and mean <= 5e-4


@pytest.mark.parametrize("name", ["tiny", "4k"])
def test_int8_grids_match_oracle_on_clean_data(name, inputs):
    """The pages' literal int8 Q / u8 P grids, on the workloads without outliers."""
    inp = inputs(name)
    out, rc = run_gpu(inp, q_mode=1, p_mode=1)
    assert rc == 0
    rows = oracle.all_rows(inp) if name == "tiny" else sample_rows(inp, 300)
    mx, mean = compare(out, inp, rows)
    assert mx <= TOL_MAX and mean <= TOL_MEAN
    ref = oracle.method(oracle.Problem.from_inputs(inp), rows, oracle.Q_INT8, oracle.P_U8, tile=KEY_TILE)
    mx2, mean2 = norm_errors(out[rows[:, 0], rows[:, 1]].astype(np.float64), ref)
    print("%s int8 grids: vs exact %.3g/%.3g, vs method %.3g/%.3g" % (name, mx, mean, mx2, mean2))
    assert mx2 <= 1.5e-2 and mean2 <= 1e-3


def test_int8_q_grid_alone_follows_method():
    inp = make_inputs(CLEAN_CHUNKED)
    out, rc = run_gpu(inp, q_mode=1, p_mode=0)
    assert rc == 0
    rows = sample_rows(inp, 100)
    ref = oracle.method(oracle.Problem.from_inputs(inp), rows, oracle.Q_INT8, oracle.P_F16, tile=KEY_TILE)
    mx, mean = norm_errors(out[rows[:, 0], rows[:, 1]].astype(np.float64), ref)
    assert mx <= 5e-3 and mean <= 5e-4


EDGE = {
    # name: (workload, S, W)
    "window_off": (Workload("e_off", 16, 2, ((0, 2048),), 1, 256, seed=31), 1, 0),
    "window_negative": (Workload("e_neg", 16, 2, ((0, 1500),), 2, 256, seed=32), 2, -1),
    "window_one_block": (Workload("e_w1", 16, 2, ((0, 1200),), 0, 1, seed=33, outlier_frac=0.02), 0, 1),
    "sink_covers_window_start": (Workload("e_sink", 16, 2, ((0, 1600),), 1, 4, seed=34), 90, 4),
    "no_sink": (Workload("e_nosink", 16, 2, ((0, 1600),), 0, 8, seed=35), 0, 8),
    "single_query_long_context": (Workload("e_one", 16, 2, ((5000, 1),), 1, 256, seed=36), 1, 256),
    "ragged_rows": (Workload("e_rag", 16, 2, ((0, 1001),), 1, 16, seed=37), 1, 16),
    "unaligned_start": (Workload("e_una", 16, 2, ((1003, 517),), 1, 8, seed=38), 1, 8),
    "gqa_4_window": (Workload("e_g4", 8, 2, ((37, 700),), 2, 3, seed=39), 2, 3),
    "gqa_2": (Workload("e_g2", 8, 4, ((0, 600),), 1, 5, seed=40), 1, 5),
    "gqa_1": (Workload("e_g1", 4, 4, ((11, 333),), 1, 2, seed=41), 1, 2),
    "gqa_16": (Workload("e_g16", 32, 2, ((0, 500),), 1, 4, seed=42), 1, 4),
    "many_sequences": (Workload("e_many", 16, 2, ((0, 16), (100, 1), (7, 300), (2000, 64), (33, 33)), 1, 4,
                                seed=43, outlier_frac=0.05), 1, 4),
    # the widest groups pa_create accepts: 4, 2 and 1 tokens per CTA (Q boxes {64, G, 128 / G})
    "gqa_32": (Workload("e_g32", 64, 2, ((0, 300),), 1, 4, seed=46, outlier_frac=0.02), 1, 4),
    "gqa_64": (Workload("e_g64", 64, 1, ((5, 203),), 1, 3, seed=47), 1, 3),
    "gqa_128": (Workload("e_g128", 128, 1, ((0, 150),), 1, 2, seed=48), 1, 2),
    # the most kv heads pa_create accepts
    "kv_heads_8": (Workload("e_h8", 64, 8, ((0, 400),), 1, 4, seed=49, outlier_frac=0.02), 1, 4),
    "kv_heads_8_gqa_16": (Workload("e_h8g16", 128, 8, ((3, 120), (40, 77)), 2, 3, seed=50), 2, 3),
}


@pytest.mark.parametrize("case", list(EDGE))
def test_edge_cases_match_oracle(case):
    wl, S, W = EDGE[case]
    inp = make_inputs(wl)
    out, rc = run_gpu(inp, S=S, W=W)
    assert rc == 0
    rows = oracle.all_rows(inp) if inp.q.shape[0] * inp.q.shape[1] <= 20000 else sample_rows(inp, 400)
    mx, mean = compare(out, inp, rows, n_sink_blk=S, n_win_blk=W)
    print("%s: max %.3g mean %.3g" % (case, mx, mean))
    assert mx <= TOL_MAX and mean <= TOL_MEAN


def test_window_covering_context_equals_window_off_bitwise():
    inp = make_inputs(Workload("e_cov", 16, 2, ((0, 1024),), 1, 64, seed=44))
    a, rc1 = run_gpu(inp, S=1, W=64)
    b, rc2 = run_gpu(inp, S=1, W=0)
    assert rc1 == 0 and rc2 == 0
    assert np.array_equal(a, b)


def test_page_permutation_is_bitwise_invariant():
    wl = Workload("e_perm", 16, 2, ((0, 900),), 1, 8, seed=45, outlier_frac=0.02)
    inp = make_inputs(wl)
    a, _ = run_gpu(inp)
    perm = np.random.default_rng(7).permutation(inp.k_pool.shape[0])
    for arr in ("k_pool", "v_pool", "k_scale", "v_scale"):
        x = getattr(inp, arr)
        y = np.empty_like(x)
        y[perm] = x
        setattr(inp, arr, y)
    bt = inp.block_table.copy()
    bt[bt >= 0] = perm[bt[bt >= 0]]
    inp.block_table = bt
    b, rc = run_gpu(inp)
    assert rc == 0 and np.array_equal(a, b)


# the host-buffer path splits the query rows into chunks that overlap the
# copies with the computation: one or several sequences, whole and cut
HOST_CASES = {
    "4k": None,
    "chunked_ragged": None,
    "32k": None,
    "cuts_unaligned": Workload("hcut", 16, 2, ((12005, 9000), (300, 700)), 1, 256, seed=71, outlier_frac=0.01),
}


@pytest.mark.parametrize("name", list(HOST_CASES))
def test_host_buffer_entry_point_matches_device_entry_point(name, inputs):
    import torch

    import windowed_prefill_attention_gb300 as pa
    inp = inputs(name) if HOST_CASES[name] is None else make_inputs(HOST_CASES[name])
    a, rc = run_gpu(inp)
    assert rc == 0
    wl = inp.wl
    h = pa.pa_create(wl.n_q_heads, wl.n_kv_heads, inp.k_pool.shape[0], inp.block_table.shape[1])
    try:
        out = torch.empty(inp.q.shape, dtype=torch.int16).pin_memory()
        pa.pa_prefill_host(h, inp.seq_desc, torch.from_numpy(inp.q.view(np.int16)), inp.k_pool, inp.v_pool,
                           inp.k_scale, inp.v_scale, inp.block_table, wl.n_sink_blk, wl.n_win_blk, wl.sm_scale, out)
    finally:
        pa.pa_destroy(h)
    b = out.view(torch.bfloat16).float().numpy()
    # one plan and one widening pass for the whole call: each chunk's units are
    # computed exactly as in the one-launch device path
    assert np.array_equal(a, b)


@pytest.mark.parametrize("name", ["tiny", "4k", "32k"])
def test_output_gate_matches_oracle(name):
    """pa_prefill_batch_gated against the fp64 definition of the gated output."""
    from synth import make_gate
    from synth.workloads import bf16_bits_to_f32
    inp = make_inputs(CONFIGS[name])
    g_bits = make_gate(inp)
    out, rc = run_gpu(inp, gate_bits=g_bits)
    assert rc == 0
    n = FULL.get(name)
    rows = oracle.all_rows(inp) if n is None else sample_rows(inp, n, seed=11)
    ref = oracle.gate(oracle.exact(oracle.Problem.from_inputs(inp), rows),
                      bf16_bits_to_f32(g_bits)[rows[:, 0], rows[:, 1]])
    got = out[rows[:, 0], rows[:, 1]].astype(np.float64)
    assert np.isfinite(got).all()
    mx, mean = norm_errors(got, ref)
    assert mx <= TOL_MAX and mean <= TOL_MEAN, (name, mx, mean)


def test_output_gate_special_values_bitwise():
    """Gate 0 halves the ungated bf16 output exactly; gate +40 (sigmoid = 1 in
    fp32) returns it unchanged."""
    inp = make_inputs(CONFIGS["4k"])
    plain, rc0 = run_gpu(inp)
    half, rc1 = run_gpu(inp, gate_bits=np.zeros_like(inp.q))
    one, rc2 = run_gpu(inp, gate_bits=np.full_like(inp.q, 0x4220))  # bf16 40.0
    assert rc0 == rc1 == rc2 == 0
    assert np.array_equal(half, plain * 0.5)
    assert np.array_equal(one, plain)


@pytest.mark.parametrize("n_win_blk", [256, 0], ids=["window", "window_off"])
def test_contexts_beyond_64k_match_oracle(inputs, n_win_blk):
    """131072-token context (beyond the pages' fallback point), sampled rows:
    with the 256-block window, and with the window off (full causal, every
    row up to 131072 keys; fewer sampled tokens, the oracle walks them all)."""
    inp = inputs("128k")
    out, rc = run_gpu(inp, W=n_win_blk)
    assert rc == 0
    rows = sample_rows(inp, 160 if n_win_blk else 24, seed=13, edge=4)
    mx, mean = compare(out, inp, rows, n_win_blk=n_win_blk)
    assert mx <= TOL_MAX and mean <= TOL_MEAN, (n_win_blk, mx, mean)
