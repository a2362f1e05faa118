"""GPU: KV append (the step before the path) through the C ABI.

The new tokens' K/V rows are quantised per (token, kv head) and written into
the paged pool through the block table.  Codes and scales are integer / fp32
decisions taken in the same precision on both sides, so the pool the kernel
writes must equal the oracle's bit for bit, every other slot unchanged.
"""
import dataclasses

import numpy as np
import pytest

import oracle
from pa_testutil import TOL_MAX, TOL_MEAN, norm_errors, run_gpu, sample_rows
from synth import CONFIGS, make_inputs
from synth.workloads import Inputs

pytestmark = pytest.mark.gpu


def _bf16_bits(x):
    b = np.asarray(x, dtype=np.float32).view(np.uint32)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def _new_rows(n_new, hkv, seed, outliers=True):
    rng = np.random.default_rng(seed)
    x = rng.normal(size=(n_new, hkv, 256)).astype(np.float32)
    if outliers:  # a few x8 tokens and an all-zero row
        x[rng.choice(n_new, size=max(1, n_new // 100), replace=False)] *= 8
        x[n_new // 2, 0] = 0.0
    return _bf16_bits(x)


def _append_gpu(inp, seq, tok_start, kn_bits, vn_bits, bt_row=None):
    import torch

    import windowed_prefill_attention_gb300 as pa
    wl = inp.wl
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    kp, vp, ks, vs = dev(inp.k_pool), dev(inp.v_pool), dev(inp.k_scale), dev(inp.v_scale)
    bt = dev(inp.block_table[seq] if bt_row is None else bt_row)
    kn = dev(kn_bits.view(np.int16)).view(torch.bfloat16)
    vn = dev(vn_bits.view(np.int16)).view(torch.bfloat16)
    h = pa.pa_create(wl.n_q_heads, wl.n_kv_heads, inp.k_pool.shape[0], inp.block_table.shape[1])
    try:
        pa.pa_kv_append(h, kn, vn, tok_start, bt, kp, vp, ks, vs)
        rc = pa.pa_last_error(h)
    finally:
        pa.pa_destroy(h)
    return [t.cpu().numpy() for t in (kp, vp, ks, vs)], rc


@pytest.mark.parametrize("seq,tok_start,n_new", [(3, 12005, 2048), (0, 1024, 2048), (1, 6144, 1), (2, 30720, 17)],
                         ids=["ragged_start", "aligned", "one_token", "short"])
def test_kv_append_is_bit_exact(seq, tok_start, n_new):
    inp = make_inputs(CONFIGS["chunked_ragged"])
    hkv = inp.wl.n_kv_heads
    kn, vn = _new_rows(n_new, hkv, 100 + seq), _new_rows(n_new, hkv, 200 + seq)
    (kp, vp, ks, vs), rc = _append_gpu(inp, seq, tok_start, kn, vn)
    assert rc == 0
    want = oracle.kv_append(inp.k_pool, inp.v_pool, inp.k_scale, inp.v_scale, inp.block_table[seq], tok_start, kn, vn)
    for got, ref in zip((kp, vp, ks, vs), want):
        assert np.array_equal(got.view(np.uint8) if got.dtype == np.int8 else got.view(np.uint32),
                              ref.view(np.uint8) if ref.dtype == np.int8 else ref.view(np.uint32))


def _tie_rows(n_new, hkv, seed):
    """Rows whose quotients x / scale sit on or next to half-integers, where
    the kernel's reciprocal shortcut hands over to the division: the golden
    row (scale 2, odd integers: exact ties), exact ties at the power-of-two
    scales 1/2 and 4, and bf16 rows at non-power-of-two scales whose
    quotients crowd around k + 0.5."""
    import json
    import os
    gold = json.load(open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "kv_codes.json")))
    rng = np.random.default_rng(seed)
    rows = np.zeros((n_new, hkv, 256), dtype=np.float32)
    for i in range(n_new):
        for g in range(hkv):
            kind = (i * hkv + g) % 4
            if kind == 0:
                r = np.asarray(gold["values"], dtype=np.float32)
            elif kind in (1, 2):
                sc = 0.5 if kind == 1 else 4.0
                k = rng.integers(-126, 126, size=256)
                r = ((k + 0.5) * sc).astype(np.float32)  # exact ties
                r[0] = 127.0 * sc                           # the row's absmax: scale = sc exactly
            else:
                am = np.float32(rng.uniform(1.0, 100.0))
                sc = np.float32(am / np.float32(127.0))
                k = rng.integers(-126, 126, size=256)
                r = ((k + 0.5 + rng.uniform(-3e-4, 3e-4, size=256)) * sc).astype(np.float32)
                r[0] = am
            rows[i, g] = r
    return _bf16_bits(rows)


def test_kv_append_half_way_codes_are_bit_exact():
    inp = make_inputs(CONFIGS["chunked_ragged"])
    hkv = inp.wl.n_kv_heads
    kn, vn = _tie_rows(64, hkv, 7), _tie_rows(64, hkv, 8)
    (kp, vp, ks, vs), rc = _append_gpu(inp, 0, 1024, kn, vn)
    assert rc == 0
    want = oracle.kv_append(inp.k_pool, inp.v_pool, inp.k_scale, inp.v_scale, inp.block_table[0], 1024, kn, vn)
    for got, ref in zip((kp, vp, ks, vs), want):
        assert np.array_equal(got.view(np.uint8) if got.dtype == np.int8 else got.view(np.uint32),
                              ref.view(np.uint8) if ref.dtype == np.int8 else ref.view(np.uint32))


def test_append_then_prefill_matches_oracle():
    """A fresh chunk appended on the GPU, then prefilled over the pool it wrote:
    against the fp64 definition on the oracle's own appended pool."""
    inp = make_inputs(CONFIGS["chunked_ragged"])
    seq, (q_off, q_start, n_q, n_ctx) = 3, inp.seq_desc[3].tolist()
    hkv = inp.wl.n_kv_heads
    kn, vn = _new_rows(n_q, hkv, 300), _new_rows(n_q, hkv, 301)
    (kp, vp, ks, vs), rc = _append_gpu(inp, seq, q_start, kn, vn)
    assert rc == 0
    new = dataclasses.replace(inp, k_pool=kp, v_pool=vp, k_scale=ks, v_scale=vs)
    out, rc = run_gpu(new)
    assert rc == 0
    kp2, vp2, ks2, vs2 = oracle.kv_append(inp.k_pool, inp.v_pool, inp.k_scale, inp.v_scale, inp.block_table[seq],
                                          q_start, kn, vn)
    ref_inp = Inputs(inp.wl, inp.q, kp2, vp2, ks2, vs2, inp.block_table, inp.seq_desc)
    rows = sample_rows(ref_inp, 128, seed=17)
    rows = rows[(rows[:, 0] >= q_off) & (rows[:, 0] < q_off + n_q)]
    ref = oracle.exact(oracle.Problem.from_inputs(ref_inp), rows)
    mx, mean = norm_errors(out[rows[:, 0], rows[:, 1]].astype(np.float64), ref)
    assert mx <= TOL_MAX and mean <= TOL_MEAN, (mx, mean)


def test_kv_append_bad_page_is_reported_and_skipped():
    import windowed_prefill_attention_gb300 as pa
    inp = make_inputs(CONFIGS["chunked_ragged"])
    hkv = inp.wl.n_kv_heads
    bt = inp.block_table[0].copy()
    bt[(1024 + 20) // 16] = inp.k_pool.shape[0] + 5  # the page of tokens 1040..1055: outside the pool
    kn, vn = _new_rows(64, hkv, 400), _new_rows(64, hkv, 401)
    (kp, vp, ks, vs), rc = _append_gpu(inp, 0, 1024, kn, vn, bt_row=bt)
    assert rc == pa.PA_EBADPAGE
    want = oracle.kv_append(inp.k_pool, inp.v_pool, inp.k_scale, inp.v_scale, inp.block_table[0], 1024, kn, vn)
    bits = lambda a: a.view(np.uint8) if a.dtype == np.int8 else a.view(np.uint32)  # noqa: E731 (NaN-safe)
    for got, ref, orig in zip((kp, vp, ks, vs), want, (inp.k_pool, inp.v_pool, inp.k_scale, inp.v_scale)):
        good = np.ones(got.shape[:2], dtype=bool)
        good[inp.block_table[0][(1024 + 20) // 16]] = False  # the slots the bad entry stood for keep old values
        assert np.array_equal(bits(got)[good], bits(ref)[good])
        assert np.array_equal(bits(got)[~good], bits(orig)[~good])


def test_kv_append_scale_is_the_rounded_quotient_for_every_bf16_magnitude():
    """The kernel's scale absmax / 127 (a reciprocal product and one FMA
    correction, no division) against the IEEE quotient, for every positive
    finite bf16 absmax: one row per value, K and V, every kv head."""
    import dataclasses as dc
    inp = make_inputs(CONFIGS["chunked_ragged"])
    hkv = inp.wl.n_kv_heads
    mags = np.arange(0x0001, 0x7F80, dtype=np.uint32)  # bf16 bit patterns of the positive finite values
    n_new = len(mags)
    pages = (n_new + 15) // 16
    a = (mags << 16).view(np.float32)
    rows = np.zeros((n_new, hkv, 256), dtype=np.float32)
    rows[:, :, 0] = a[:, None]                      # the row's absmax
    rows[:, :, 1] = -a[:, None] * np.float32(0.37)  # and a code that is not +-127
    bits = _bf16_bits(rows)
    pool = dc.replace(inp, k_pool=np.zeros((pages, 16, hkv, 256), np.int8),
                      v_pool=np.zeros((pages, 16, hkv, 256), np.int8),
                      k_scale=np.zeros((pages, 16, hkv), np.float32), v_scale=np.zeros((pages, 16, hkv), np.float32),
                      block_table=np.arange(pages, dtype=np.int32)[None, :])
    (kp, vp, ks, vs), rc = _append_gpu(pool, 0, 0, bits, bits, bt_row=np.arange(pages, dtype=np.int32))
    assert rc == 0
    want_scale = (a / np.float32(127.0)).astype(np.float32)
    for sc in (ks, vs):
        got = sc.reshape(-1, hkv)[:n_new]
        assert np.array_equal(got.view(np.uint32), np.repeat(want_scale[:, None], hkv, 1).view(np.uint32))
    want = oracle.kv_append(pool.k_pool, pool.v_pool, pool.k_scale, pool.v_scale, np.arange(pages, dtype=np.int32),
                            0, bits, bits)
    for got, ref in zip((kp, vp), want[:2]):
        assert np.array_equal(got.view(np.uint8), ref.view(np.uint8))


def test_kv_append_full_size_bench_configuration():
    """The bench's append at full size: every one of the 32k workload's 32768
    tokens, 2 kv heads, quantised into its pool through its block table
    (N(0,1) rows with 1 % of tokens x8, one all-zero row); every code and
    scale of the pool equals the oracle's, every other slot unchanged."""
    inp = make_inputs(CONFIGS["32k"])
    hkv = inp.wl.n_kv_heads
    q_off, q_start, n_q, n_ctx = inp.seq_desc[0].tolist()
    kn, vn = _new_rows(n_q, hkv, 300), _new_rows(n_q, hkv, 301)
    (kp, vp, ks, vs), rc = _append_gpu(inp, 0, q_start, kn, vn)
    assert rc == 0
    want = oracle.kv_append(inp.k_pool, inp.v_pool, inp.k_scale, inp.v_scale, inp.block_table[0], q_start, kn, vn)
    for got, ref in zip((kp, vp, ks, vs), want):
        bits = (lambda a: a.view(np.uint8)) if got.dtype == np.int8 else (lambda a: a.view(np.uint32))
        assert np.array_equal(bits(got), bits(ref))

