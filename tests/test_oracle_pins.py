"""Pins for the oracle, against things other than the oracle itself.

Each test checks the fp64 oracle (oracle/pa_oracle.c) against an independent
route: a dense numpy/scipy brute force with the mask written as explicit
block sets, closed forms (first token, zero softmax scale, identical keys),
invariances (page permutation, window covering the context == window off),
values printed on the pages (the ~2.08 TFLOP figure at 32k), and hand-derived
quantisation codes.  CPU only.
"""
import json
import os

import numpy as np
import pytest
import scipy.special

import oracle
from synth import CONFIGS, make_inputs
from synth.workloads import Workload, bf16_bits_to_f32

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

SMALL = {
    "tiny": CONFIGS["tiny"],
    # window of 3 blocks + 1 sink block over 200 tokens (partial last page)
    "small_win": Workload("small_win", 4, 2, ((0, 200),), n_sink_blk=1, n_win_blk=3, seed=11),
    # two sequences, q_start off the 16-grid, 2 sink blocks, outliers
    "small_chunk": Workload("small_chunk", 4, 2, ((37, 50), (100, 61)), n_sink_blk=2, n_win_blk=2, seed=12,
                            outlier_frac=0.05),
    # GQA 8:1 like the large configs, window off
    "small_causal": Workload("small_causal", 8, 1, ((5, 91),), n_sink_blk=1, n_win_blk=0, seed=13),
}


def brute_force(inp, n_sink_blk, n_win_blk, sm_scale):
    """Dense attention per row; the visible set is built as a set of 16-token
    blocks: the sink blocks plus the last W blocks ending at n_blk_q = (t+16)/16."""
    HQ, HKV = inp.q.shape[1], inp.k_pool.shape[2]
    G = HQ // HKV
    out = np.zeros(inp.q.shape, dtype=np.float64)
    for s, (q_off, q_start, n_q, n_ctx) in enumerate(inp.seq_desc):
        tok = np.arange(n_ctx)
        phys, slot = inp.block_table[s, tok // 16], tok % 16
        K = inp.k_pool[phys, slot].astype(np.float64) * inp.k_scale[phys, slot][..., None].astype(np.float64)
        V = inp.v_pool[phys, slot].astype(np.float64) * inp.v_scale[phys, slot][..., None].astype(np.float64)
        Q = bf16_bits_to_f32(inp.q[q_off:q_off + n_q]).astype(np.float64)
        for i in range(n_q):
            t = q_start + i
            n_blk_q = (t + 16) // 16
            if n_win_blk > 0:
                blocks = set(range(n_sink_blk)) | set(range(max(0, n_blk_q - n_win_blk), n_blk_q))
            else:
                blocks = set(range(n_blk_q))
            keys = np.array([j for j in range(t + 1) if j // 16 in blocks])
            for h in range(HQ):
                g = h // G
                w = scipy.special.softmax(sm_scale * (K[keys, g] @ Q[i, h]))
                out[q_off + i, h] = w @ V[keys, g]
    return out


def run_exact(inp, **kw):
    prob = oracle.Problem.from_inputs(inp, **kw)
    rows = oracle.all_rows(inp)
    return oracle.exact(prob, rows).reshape(inp.q.shape)


def norm_err(a, ref):
    return np.abs(a - ref) / np.maximum(1.0, np.abs(ref))


@pytest.mark.parametrize("name", list(SMALL))
def test_exact_matches_dense_bruteforce(name):
    wl = SMALL[name]
    inp = make_inputs(wl)
    got = run_exact(inp)
    ref = brute_force(inp, wl.n_sink_blk, wl.n_win_blk, wl.sm_scale)
    assert norm_err(got, ref).max() < 1e-12


def test_window_covering_context_equals_window_off():
    wl = SMALL["small_chunk"]
    inp = make_inputs(wl)
    n_blocks = max(wl.n_ctx) // 16 + 1
    a = run_exact(inp, n_win_blk=n_blocks)
    b = run_exact(inp, n_win_blk=0)
    c = run_exact(inp, n_win_blk=-3, n_sink_blk=5)
    assert np.array_equal(a, b) and np.array_equal(b, c)
    ref = brute_force(inp, 0, 0, wl.sm_scale)
    assert norm_err(a, ref).max() < 1e-12


def test_first_token_returns_its_value():
    inp = make_inputs(SMALL["small_win"])
    got = run_exact(inp)
    p = inp.block_table[0, 0]
    for h in range(inp.q.shape[1]):
        g = h // (inp.q.shape[1] // inp.k_pool.shape[2])
        v0 = inp.v_pool[p, 0, g].astype(np.float64) * np.float64(inp.v_scale[p, 0, g])
        assert np.array_equal(got[0, h], v0)


@pytest.mark.parametrize("name", ["small_win", "small_chunk"])
def test_zero_softmax_scale_gives_mean_of_visible_values(name):
    wl = SMALL[name]
    inp = make_inputs(wl)
    got = run_exact(inp, sm_scale=0.0)
    HQ, HKV = inp.q.shape[1], inp.k_pool.shape[2]
    for s, (q_off, q_start, n_q, n_ctx) in enumerate(inp.seq_desc):
        tok = np.arange(n_ctx)
        phys, slot = inp.block_table[s, tok // 16], tok % 16
        V = inp.v_pool[phys, slot].astype(np.float64) * inp.v_scale[phys, slot][..., None].astype(np.float64)
        for i in range(n_q):
            t = q_start + i
            lo = max(0, t // 16 + 1 - wl.n_win_blk)
            keep = [j for j in range(t + 1) if j // 16 < wl.n_sink_blk or j // 16 >= lo]
            for h in range(HQ):
                ref = V[keep, h // (HQ // HKV)].mean(axis=0)
                assert norm_err(got[q_off + i, h], ref).max() < 1e-13


def test_identical_keys_give_mean_of_values():
    wl = SMALL["small_win"]
    inp = make_inputs(wl)
    inp.k_pool[:] = inp.k_pool[inp.block_table[0, 0], 0, 0][None, None, None, :]
    inp.k_scale[:] = np.float32(0.03)
    got = run_exact(inp)
    ref = run_exact(inp, sm_scale=0.0)
    assert norm_err(got, ref).max() < 1e-13


def test_page_permutation_is_bit_identical():
    wl = SMALL["small_chunk"]
    inp = make_inputs(wl)
    base = run_exact(inp)
    rng = np.random.default_rng(99)
    perm = rng.permutation(inp.k_pool.shape[0])       # new slot of old page p is perm[p]
    for arr in ("k_pool", "v_pool", "k_scale", "v_scale"):
        a = getattr(inp, arr)
        b = np.empty_like(a)
        b[perm] = a
        setattr(inp, arr, b)
    bt = inp.block_table.copy()
    bt[bt >= 0] = perm[bt[bt >= 0]]
    inp.block_table = bt
    assert np.array_equal(run_exact(inp), base)


def closed_form_count(t, S, W):
    if W <= 0:
        return t + 1
    lo = max(0, t // 16 + 1 - W)
    if lo <= S:
        return t + 1
    return 16 * S + (t - 16 * lo + 1)


def test_visible_count_closed_form():
    for S in (0, 1, 3):
        for W in (-1, 0, 1, 2, 5, 256):
            for t in list(range(0, 300)) + [4095, 4096, 32767]:
                assert oracle.visible_count(t, S, W) == closed_form_count(t, S, W), (t, S, W)


def test_flop_count_matches_pages():
    g = json.load(open(os.path.join(GOLDEN, "flops_32k.json")))
    pairs = oracle.visible_pairs(0, g["n_ctx"], g["n_sink_blk"], g["n_win_blk"])
    tflop = pairs * g["n_q_heads"] * 4 * g["head_dim"] / 1e12
    assert abs(tflop - g["tflop_per_layer"]) / g["tflop_per_layer"] < g["printed_precision_rel"]


def test_block_lists_closed_form():
    cases = [(0, 256, 0, 16), (0, 4096, 1, 256), (37, 50, 2, 2), (1000, 700, 1, 8), (12005, 300, 1, 4),
             (64, 64, 0, 0), (3, 29, 3, 1)]
    for q_start, n_q, S, W in cases:
        got = oracle.block_lists(q_start, n_q, S, W, cap=600)
        for r, qb in enumerate(range(q_start // 16, (q_start + n_q - 1) // 16 + 1)):
            if W > 0:
                want = sorted(set(range(min(S, qb + 1))) | set(range(max(0, qb + 1 - W), qb + 1)))
            else:
                want = list(range(qb + 1))
            row = got[r][got[r] >= 0].tolist()
            assert row == want, (q_start, n_q, S, W, qb)


def test_gather_matches_fancy_indexing():
    wl = SMALL["small_chunk"]
    inp = make_inputs(wl)
    prob = oracle.Problem.from_inputs(inp)
    for s in range(inp.n_seq):
        n_ctx = int(inp.seq_desc[s, 3])
        tok = np.arange(n_ctx)
        phys, slot = inp.block_table[s, tok // 16], tok % 16
        for g in range(inp.k_pool.shape[2]):
            k, v, ks, vs = oracle.gather(prob, s, g, n_ctx)
            assert np.array_equal(k, inp.k_pool[phys, slot, g])
            assert np.array_equal(v, inp.v_pool[phys, slot, g])
            assert np.array_equal(ks, inp.k_scale[phys, slot, g])
            assert np.array_equal(vs, inp.v_scale[phys, slot, g])


@pytest.mark.parametrize("name", ["tiny", "small_win", "small_chunk", "small_causal"])
@pytest.mark.parametrize("tile", [16, 48, 64])
def test_online_softmax_equals_two_pass(name, tile):
    inp = make_inputs(SMALL[name])
    prob = oracle.Problem.from_inputs(inp)
    rows = oracle.all_rows(inp)
    a = oracle.exact(prob, rows)
    b = oracle.method(prob, rows, oracle.Q_LOSSLESS, oracle.P_EXACT, tile=tile)
    assert norm_err(b, a).max() < 1e-12


def test_q_int8_codes_golden():
    g = json.load(open(os.path.join(GOLDEN, "q_int8_codes.json")))
    for case in g["cases"]:
        bits = (np.asarray(case["row"], np.float32).view(np.uint32) >> 16).astype(np.uint16)
        codes, scale = oracle.quantize_q_row(bits)
        assert codes.tolist() == case["codes"]
        assert abs(float(scale) - case["scale"]) <= 1e-8


def test_p_u8_codes_golden():
    g = json.load(open(os.path.join(GOLDEN, "p_u8_codes.json")))
    for case in g["cases"]:
        codes, sp = oracle.quantize_p_u8(np.asarray(case["p"]), case.get("prev_scale", 1.0))
        assert codes.tolist() == case["codes"]
        assert abs(sp - case["scale"]) <= 1e-15


def test_int8_q_is_lossless_on_the_int8_grid():
    """Queries whose entries are integers times 2^-5 with absmax 127*2^-5 are
    quantised without loss, so the method equals the definition."""
    wl = SMALL["small_chunk"]
    inp = make_inputs(wl)
    rng = np.random.default_rng(5)
    codes = rng.integers(-127, 128, size=inp.q.shape).astype(np.float32)
    codes[..., 0] = 127.0
    inp.q = (np.ascontiguousarray(codes * np.float32(2.0 ** -5)).view(np.uint32) >> 16).astype(np.uint16)
    prob = oracle.Problem.from_inputs(inp, sm_scale=1.0 / 256)
    rows = oracle.all_rows(inp)
    a = oracle.exact(prob, rows)
    b = oracle.method(prob, rows, oracle.Q_INT8, oracle.P_EXACT)
    assert norm_err(b, a).max() < 1e-12


def _constant_p_case(vscale_of_tile):
    """Causal workload, sm_scale 0 (all p = 1), V scale constant over each
    64-key tile, so every tile's P' is one value: its quantisation is exact."""
    wl = Workload("cp", 4, 1, ((0, 300),), n_sink_blk=0, n_win_blk=0, seed=21)
    inp = make_inputs(wl)
    tok = np.arange(300)
    phys, slot = inp.block_table[0, tok // 16], tok % 16
    inp.v_scale[phys, slot, 0] = vscale_of_tile(tok // 64).astype(np.float32)
    prob = oracle.Problem.from_inputs(inp, sm_scale=0.0)
    return prob, oracle.all_rows(inp)


def test_u8_p_rescale_chain_is_exact_when_lossless():
    prob, rows = _constant_p_case(lambda tile: 0.01 * (1.0 + 0.7 * (tile % 3)))
    a = oracle.exact(prob, rows)
    b = oracle.method(prob, rows, oracle.Q_LOSSLESS, oracle.P_U8, tile=64)
    assert norm_err(b, a).max() < 1e-12


def test_f16_p_rounding_is_exact_on_dyadic_values():
    prob, rows = _constant_p_case(lambda tile: 2.0 ** -(4 + (tile % 3)))
    a = oracle.exact(prob, rows)
    b = oracle.method(prob, rows, oracle.Q_LOSSLESS, oracle.P_F16, tile=64)
    assert norm_err(b, a).max() < 1e-12


def _fp16_grid_values(rng):
    """fp32 values over the binary16 normal range [2^-14, 65504]: grid points,
    exact half-way points between neighbours (even and odd lower neighbour),
    the fp32 values either side of each half-way point, and random fp32
    values of every binade."""
    vals = []
    for e in range(-14, 16):
        ulp = 2.0 ** (e - 10)
        m = rng.integers(1024, 2048, size=24)
        m[:2] = (1024, 2046)  # an even and (with +1 below) odd lower neighbour at the binade's ends
        grid = m * ulp
        half = grid + ulp / 2
        vals += [grid, half, (m + 1) * ulp + ulp / 2]
        h32 = half.astype(np.float32)
        vals += [np.nextafter(h32, np.float32(np.inf)), np.nextafter(h32, np.float32(0))]
        vals.append(rng.uniform(2.0 ** e, 2.0 ** (e + 1), size=24))
    v = np.concatenate(vals).astype(np.float32)
    return v[(v >= np.float32(2.0 ** -14)) & (v <= np.float32(65504.0))]


def test_f16_p_rounding_is_ieee_binary16_nearest_even():
    """The method's fp16 container for P' (P_F16) against IEEE binary16
    round-to-nearest-even (numpy's float32 -> float16 cast) over the fp16
    normal range, through the whole P_F16 path: one-token sequences see one
    key, so p = 1 and P' = v_scale, and a V code of 1 (-1) in dim 0 (1) puts
    the rounded P' in the output.  Ties must go to the even neighbour: 10
    significant bits, truncation or ties-away each fail."""
    rng = np.random.default_rng(16)
    vs = _fp16_grid_values(rng)
    n = vs.shape[0]
    D = 256
    q = np.full((n, 1, D), 0x3F80, dtype=np.uint16)  # bf16 1.0
    kp = np.ones((n, 16, 1, D), dtype=np.int8)
    vp = np.zeros((n, 16, 1, D), dtype=np.int8)
    vp[:, :, 0, 0] = 1
    vp[:, :, 0, 1] = -1
    ks = np.full((n, 16, 1), 0.01, dtype=np.float32)
    v_scale = np.zeros((n, 16, 1), dtype=np.float32)
    v_scale[:, 0, 0] = vs
    bt = np.arange(n, dtype=np.int32)[:, None]
    seqs = np.stack([np.arange(n), np.zeros(n), np.ones(n), np.ones(n)], 1).astype(np.int32)
    prob = oracle.Problem(q, kp, vp, ks, v_scale, bt, seqs, 0, 0, 1.0 / 16)
    rows = np.stack([np.arange(n), np.zeros(n)], 1).astype(np.int32)
    out = oracle.method(prob, rows, oracle.Q_LOSSLESS, oracle.P_F16, tile=64)
    want = vs.astype(np.float16).astype(np.float64)
    assert np.isfinite(want).all()
    assert np.array_equal(out[:, 0], want)
    assert np.array_equal(out[:, 1], -want)
    # the grid really holds cases that tell the roundings apart
    assert (want != vs.astype(np.float64)).sum() > n // 3


def test_gate_against_library_sigmoid_and_special_values():
    """The output gate (out * sigmoid(g)) against scipy's logistic function on
    random values and on the special points: sigmoid(0) = 1/2 exactly, the
    saturated ends, and sigmoid(x) + sigmoid(-x) = 1."""
    rng = np.random.default_rng(5)
    out = rng.normal(size=(64, 256))
    g = rng.normal(0.0, 3.0, size=(64, 256))
    np.testing.assert_allclose(oracle.gate(out, g), out * scipy.special.expit(g), rtol=1e-14, atol=0)
    assert np.array_equal(oracle.gate(out, np.zeros_like(g)), out * 0.5)
    np.testing.assert_allclose(oracle.gate(out, np.full_like(g, 40.0)), out, rtol=1e-15)
    assert np.all(np.abs(oracle.gate(out, np.full_like(g, -800.0))) == 0.0)
    np.testing.assert_allclose(oracle.gate(out, g) + oracle.gate(out, -g), out, rtol=1e-13, atol=1e-15)


def _bf16_bits(x):
    x = np.asarray(x, dtype=np.float32)
    b = x.view(np.uint32)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)  # round to nearest even


def test_kv_quantize_golden_row():
    """A hand-derived row (scale 2 exactly, values on and between the code
    grid, half-way cases rounded to even) gives the codes written out by hand."""
    with open(os.path.join(GOLDEN, "kv_codes.json")) as f:
        gold = json.load(f)
    codes, scale = oracle.kv_quantize(_bf16_bits(gold["values"])[None, :])
    assert scale[0] == np.float32(gold["scale"])
    assert codes[0, :16].tolist() == gold["codes_first16"]
    assert not codes[0, 16:].any()


def test_kv_quantize_properties():
    """On random rows: the largest magnitude maps to +-127, every value is
    reconstructed within half a step (up to the fp32 rounding of x / scale, in
    which a value a hair above a half-way point can round to the tie), an
    all-zero row gets scale 0 and codes 0."""
    rng = np.random.default_rng(9)
    x = rng.normal(size=(500, 256)).astype(np.float32) * rng.uniform(0.01, 50, size=(500, 1)).astype(np.float32)
    x[7] = 0.0
    bits = _bf16_bits(x)
    xf = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    codes, scale = oracle.kv_quantize(bits)
    assert scale[7] == 0 and not codes[7].any()
    live = np.arange(500) != 7
    s = scale[live].astype(np.float64)[:, None]
    # half a step, plus the fp32 rounding of the quotient x / scale (<= 127 * 2^-24 steps)
    assert np.all(np.abs(xf[live] - codes[live] * s) <= (0.5 + 1e-5) * s)
    top = np.abs(xf[live]).argmax(axis=1)
    assert np.all(np.abs(codes[live][np.arange(live.sum()), top]) == 127)


def test_kv_append_places_rows_through_the_block_table():
    """Rows land at page bt[t // 16], slot t % 16; every other slot is untouched."""
    rng = np.random.default_rng(10)
    n_pool, hkv = 9, 2
    kp = rng.integers(-127, 128, size=(n_pool, 16, hkv, 256), dtype=np.int8)
    vp = rng.integers(-127, 128, size=(n_pool, 16, hkv, 256), dtype=np.int8)
    ks = rng.uniform(0.1, 1, size=(n_pool, 16, hkv)).astype(np.float32)
    vs = rng.uniform(0.1, 1, size=(n_pool, 16, hkv)).astype(np.float32)
    bt = np.array([4, 0, 7, 2], dtype=np.int32)
    tok_start, n_new = 13, 30  # tokens 13..42: pages bt[0..2], slots 13.. and 0..10
    kn = _bf16_bits(rng.normal(size=(n_new, hkv, 256)))
    vn = _bf16_bits(rng.normal(size=(n_new, hkv, 256)))
    k2, v2, ks2, vs2 = oracle.kv_append(kp, vp, ks, vs, bt, tok_start, kn, vn)
    kc, kq = oracle.kv_quantize(kn)
    vc, vq = oracle.kv_quantize(vn)
    touched = np.zeros((n_pool, 16), dtype=bool)
    for i in range(n_new):
        t = tok_start + i
        page, slot = bt[t // 16], t % 16
        touched[page, slot] = True
        assert np.array_equal(k2[page, slot], kc[i]) and np.array_equal(v2[page, slot], vc[i])
        assert np.array_equal(ks2[page, slot], kq[i]) and np.array_equal(vs2[page, slot], vq[i])
    assert np.array_equal(k2[~touched], kp[~touched]) and np.array_equal(vs2[~touched], vs[~touched])
