"""GPU: split-KV decode (one new token per sequence) through the C ABI,
against the fp64 definition.

A decode call is an attention call whose every sequence has one query row,
the context's last token, so the workloads and the oracle are the prefill's:
sequences (q_start, n_q) = (n_ctx - 1, 1).
"""
import numpy as np
import pytest

import oracle
from pa_testutil import TOL_MAX, TOL_MEAN, norm_errors, to_device
from synth import make_inputs
from synth.workloads import Workload

pytestmark = pytest.mark.gpu


def _decode_wl(name, hq, hkv, ctxs, S, W, seed, outliers=0.01):
    return Workload(name, hq, hkv, tuple((c - 1, 1) for c in ctxs), S, W, seed=seed, outlier_frac=outliers)


def run_decode(inp, S=None, W=None, bt=None):
    import torch

    import windowed_prefill_attention_gb300 as pa
    wl = inp.wl
    d = to_device(inp)
    if bt is not None:
        d["block_table"] = torch.from_numpy(bt).cuda()
    out = torch.full_like(d["q"], float("nan"))
    h = pa.pa_create(wl.n_q_heads, wl.n_kv_heads, inp.k_pool.shape[0], inp.block_table.shape[1])
    try:
        pa.pa_decode(h, inp.seq_desc, d["q"], d["k_pool"], d["v_pool"], d["k_scale"], d["v_scale"], d["block_table"],
                     wl.n_sink_blk if S is None else S, wl.n_win_blk if W is None else W, wl.sm_scale, out)
        rc = pa.pa_last_error(h)
    finally:
        pa.pa_destroy(h)
    return out.float().cpu().numpy(), rc


CASES = {
    # contexts around split (256 keys) and window (4096 keys) edges, one-block and one-token contexts
    "mixed": _decode_wl("dec_mixed", 16, 2, (4096, 32000, 17, 1, 12005, 256, 257, 4112, 65536), 1, 256, 41),
    "window_off": _decode_wl("dec_nowin", 16, 2, (300, 5000, 16, 4097), 1, 0, 42),
    "no_sink": _decode_wl("dec_nosink", 16, 2, (9000, 4096, 100), 0, 64, 43),
    "sink_in_window": _decode_wl("dec_sinkwin", 16, 2, (200, 1000), 4, 10, 44),
    "gqa1": _decode_wl("dec_g1", 4, 4, (3000, 700), 1, 128, 45),
    "gqa2": _decode_wl("dec_g2", 8, 4, (2049, 33), 2, 32, 46),
    "gqa4": _decode_wl("dec_g4", 8, 2, (6000,), 1, 256, 47),
    "many": _decode_wl("dec_many", 16, 2, tuple(int(x) for x in np.random.default_rng(48).integers(1, 20000, 40)),
                       1, 256, 48),
    # window off on long contexts: each (sequence, kv head) pair spans dozens of CTAs and partials
    "long_pairs": _decode_wl("dec_long", 8, 2, (40000, 36001, 1), 1, 0, 50),
    # more than one launch's table (512 sequences): short contexts, many pairs per CTA
    "over_512": _decode_wl("dec_600", 4, 2, tuple(int(x) for x in np.random.default_rng(51).integers(1, 300, 600)),
                           1, 8, 51, outliers=0.0),
    "kv_heads_8": _decode_wl("dec_h8", 8, 8, (5000, 129, 70000), 1, 256, 52),
    # ~43.8k visible blocks: more than one wave of 128-block runs holds, so equal runs over several waves
    "multi_wave": _decode_wl("dec_waves", 8, 1, (70000,) * 9 + (69999,), 1, 0, 53, outliers=0.0),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_decode_matches_oracle(case):
    inp = make_inputs(CASES[case])
    out, rc = run_decode(inp)
    assert rc == 0
    rows = oracle.all_rows(inp)
    ref = oracle.exact(oracle.Problem.from_inputs(inp), rows)
    got = out[rows[:, 0], rows[:, 1]].astype(np.float64)
    assert np.isfinite(got).all()
    mx, mean = norm_errors(got, ref)
    assert mx <= TOL_MAX and mean <= TOL_MEAN, (case, mx, mean)


def test_decode_rejects_prefill_shaped_sequences_and_wide_groups():
    import windowed_prefill_attention_gb300 as pa
    inp = make_inputs(CASES["window_off"])
    bad = inp.seq_desc.copy()
    bad[0, 1] -= 1  # not the context's last token
    with pytest.raises(pa.PAError):
        run_decode(type(inp)(inp.wl, inp.q, inp.k_pool, inp.v_pool, inp.k_scale, inp.v_scale, inp.block_table, bad))
    wide = make_inputs(_decode_wl("dec_g16", 32, 2, (100,), 1, 8, 49))
    with pytest.raises(pa.PAError):
        run_decode(wide)


def test_decode_bad_page_is_reported():
    import windowed_prefill_attention_gb300 as pa
    inp = make_inputs(CASES["no_sink"])
    bt = inp.block_table.copy()
    bt[0, (inp.seq_desc[0, 3] - 1) // 16] = inp.k_pool.shape[0] + 9  # the query's own block: always visible
    _, rc = run_decode(inp, bt=bt)
    assert rc == pa.PA_EBADPAGE


def test_decode_repeated_calls_on_one_handle_are_identical():
    """Calls on one handle, with batches of other sizes and split counts in
    between (its partials buffer grows and is reused), give the bits of a call
    on a fresh handle."""
    import torch

    import windowed_prefill_attention_gb300 as pa
    big, small = make_inputs(CASES["many"]), make_inputs(CASES["mixed"])
    ref_big, rc0 = run_decode(big)
    ref_small, rc1 = run_decode(small)
    assert rc0 == 0 and rc1 == 0
    wl = big.wl
    pool = max(big.k_pool.shape[0], small.k_pool.shape[0])
    width = max(big.block_table.shape[1], small.block_table.shape[1])
    h = pa.pa_create(wl.n_q_heads, wl.n_kv_heads, pool, width)
    try:
        for inp, ref in ((big, ref_big), (small, ref_small), (big, ref_big), (small, ref_small), (small, ref_small)):
            d = to_device(inp)
            bt = np.zeros((inp.block_table.shape[0], width), np.int32)  # the handle's row stride
            bt[:, :inp.block_table.shape[1]] = inp.block_table
            d["block_table"] = torch.from_numpy(bt).cuda()
            out = torch.full_like(d["q"], float("nan"))
            pa.pa_decode(h, inp.seq_desc, d["q"], d["k_pool"], d["v_pool"], d["k_scale"], d["v_scale"],
                         d["block_table"], inp.wl.n_sink_blk, inp.wl.n_win_blk, inp.wl.sm_scale, out)
            assert pa.pa_last_error(h) == 0
            assert np.array_equal(out.float().cpu().numpy(), ref, equal_nan=True)
    finally:
        pa.pa_destroy(h)


def test_decode_full_size_bench_configuration():
    """The bench's decode step at full size, in its launch configuration: 64
    sequences at a 32768-token context, 16 q / 2 kv heads, 1 sink block + a
    256-block window (one wave of cost-balanced runs), every output row against
    the fp64 definition.  Only the 257 visible pages of a sequence hold data
    (random codes, scales in [1e-3, 2e-2]); its other block-table entries
    point at a valid page that the mask never visits."""
    from synth.workloads import Inputs
    rng = np.random.default_rng(123)
    n_seq, ctx, hq, hkv, S, W = 64, 32768, 16, 2, 1, 256
    pages = ctx // 16
    vis_blocks = [0] + list(range(pages - W, pages))
    n_pool = n_seq * len(vis_blocks)
    perm = rng.permutation(n_pool).astype(np.int32)
    bt = np.zeros((n_seq, pages), dtype=np.int32)
    bt[:, vis_blocks] = perm.reshape(n_seq, len(vis_blocks))
    def codes():  # int8 codes in [-127, 127]: random 64-bit words as bytes, -128 raised to -127
        n = n_pool * 16 * hkv * 256
        c = rng.integers(0, 2**63, size=n // 8, dtype=np.uint64).view(np.int8).reshape(n_pool, 16, hkv, 256)
        return np.maximum(c, np.int8(-127))
    k_pool, v_pool = codes(), codes()
    k_scale = (rng.random((n_pool, 16, hkv), dtype=np.float32) * 0.019 + 0.001).astype(np.float32)
    v_scale = (rng.random((n_pool, 16, hkv), dtype=np.float32) * 0.019 + 0.001).astype(np.float32)
    q32 = rng.standard_normal((n_seq, hq, 256), dtype=np.float32)
    u = q32.view(np.uint32)
    q = ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)
    desc = np.array([(s, ctx - 1, 1, ctx) for s in range(n_seq)], dtype=np.int32)
    wl = Workload("dec_bench", hq, hkv, tuple((ctx - 1, 1) for _ in range(n_seq)), S, W, seed=0)
    inp = Inputs(wl, q, k_pool, v_pool, k_scale, v_scale, bt, desc)
    out, rc = run_decode(inp)
    assert rc == 0
    rows = oracle.all_rows(inp)
    ref = oracle.exact(oracle.Problem.from_inputs(inp), rows)
    got = out[rows[:, 0], rows[:, 1]].astype(np.float64)
    assert np.isfinite(got).all()
    mx, mean = norm_errors(got, ref)
    assert mx <= TOL_MAX and mean <= TOL_MEAN, (mx, mean)

