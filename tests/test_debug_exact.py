"""GPU: gather, mask-set and page indexing equal the oracle's enumerations bit
for bit.  The exports run the same device geometry code the attention kernel
uses (pa_tiles.cuh) and the same widening kernel."""
import numpy as np
import pytest

import oracle
from pa_testutil import to_device
from synth import CONFIGS, make_inputs
from synth.workloads import Workload

pytestmark = pytest.mark.gpu

GATHER_CASES = {
    "4k": CONFIGS["4k"],
    "chunked_ragged": CONFIGS["chunked_ragged"],
    "window_small": Workload("gw", 16, 2, ((700, 900),), 2, 5, seed=51),
    "window_off": Workload("goff", 8, 2, ((33, 500),), 1, 0, seed=52),
}


@pytest.mark.parametrize("case", list(GATHER_CASES))
def test_gather_is_bit_exact_and_skips_invisible_blocks(case):
    import windowed_prefill_attention_gb300 as pa
    wl = GATHER_CASES[case]
    inp = make_inputs(wl)
    d = to_device(inp)
    prob = oracle.Problem.from_inputs(inp)
    h = pa.pa_create(wl.n_q_heads, wl.n_kv_heads, inp.k_pool.shape[0], inp.block_table.shape[1])
    try:
        for s, (q_off, q_start, n_q, n_ctx) in enumerate(inp.seq_desc.tolist()):
            k, v, ks, vs, tok = pa.pa_debug_gather(h, inp.seq_desc, d["k_pool"], d["v_pool"], d["k_scale"],
                                                   d["v_scale"], d["block_table"], wl.n_sink_blk, wl.n_win_blk, s,
                                                   cap=70000)
            k, v, ks, vs, tok = (x.cpu().numpy() for x in (k, v, ks, vs, tok))
            ok_rows = tok >= 0
            t = tok[ok_rows]
            # stored tokens: exactly the blocks some query of the call can see
            lists = oracle.block_lists(q_start, n_q, wl.n_sink_blk, wl.n_win_blk, cap=8192)
            want_blocks = sorted(set(lists[lists >= 0].tolist()))
            assert sorted(set((tok[tok >= 0] // 16).tolist())) == want_blocks
            assert np.all(np.diff(t) > 0), "rows in logical order"
            ok_, ov_, oks, ovs = oracle.gather(prob, s, 0, n_ctx)
            for g in range(wl.n_kv_heads):
                ok_, ov_, oks, ovs = oracle.gather(prob, s, g, n_ctx)
                assert np.array_equal(k[g][ok_rows], ok_[t])
                assert np.array_equal(v[g][ok_rows], ov_[t])
                assert np.array_equal(ks[g][ok_rows], oks[t])
                assert np.array_equal(vs[g][ok_rows], ovs[t])
                # rows past n_ctx are zero (never NaN from the pool)
                assert not k[g][~ok_rows].any() and not v[g][~ok_rows].any()
                assert not ks[g][~ok_rows].any() and not vs[g][~ok_rows].any()
    finally:
        pa.pa_destroy(h)


MASK_CASES = {
    "tiny": CONFIGS["tiny"],
    "4k": CONFIGS["4k"],
    "chunked_ragged": CONFIGS["chunked_ragged"],
    "g4_window": Workload("m4", 8, 2, ((37, 700),), 2, 3, seed=53),
    "g1_window": Workload("m1", 4, 4, ((5, 400),), 1, 2, seed=54),
    "g16_window": Workload("m16", 32, 2, ((3, 300),), 1, 4, seed=55),
    "window_off": Workload("moff", 16, 2, ((21, 700),), 1, 0, seed=56),
    "sink_over_window": Workload("mso", 16, 2, ((0, 900),), 30, 4, seed=57),
}


@pytest.mark.parametrize("case", list(MASK_CASES))
def test_maskset_is_bit_exact(case):
    import windowed_prefill_attention_gb300 as pa
    wl = MASK_CASES[case]
    G = wl.n_q_heads // wl.n_kv_heads
    TQ = pa.UNIT_ROWS // G  # tokens per unit
    seq_desc = make_inputs(wl).seq_desc if wl.total_q < 20000 else None
    if seq_desc is None:
        seq_desc = np.array([(0, qs, nq, qs + nq) for qs, nq in wl.seqs], np.int32)
        off = 0
        for i, (qs, nq) in enumerate(wl.seqs):
            seq_desc[i, 0] = off
            off += nq
    h = pa.pa_create(wl.n_q_heads, wl.n_kv_heads, 8, max(wl.pages_per_seq))
    try:
        units, counts, blocks = pa.pa_debug_maskset(h, seq_desc, wl.n_sink_blk, wl.n_win_blk, units_cap=20000,
                                                    cap=600)
    finally:
        pa.pa_destroy(h)
    counts, blocks = counts.cpu().numpy(), blocks.cpu().numpy()
    lists = {s: oracle.block_lists(qs, nq, wl.n_sink_blk, wl.n_win_blk, cap=8192)
             for s, (_, qs, nq, _) in enumerate(seq_desc.tolist())}
    for u, (s, g, t0, n_tiles) in enumerate(units.tolist()):
        q_off, q_start, n_q, _ = seq_desc[s].tolist()
        toks = [t for t in range(t0, t0 + TQ) if q_start <= t < q_start + n_q]
        union = set()
        for qb in {t // 16 for t in toks}:
            row = lists[s][qb - q_start // 16]
            union.update(row[row >= 0].tolist())
        visited = blocks[u][blocks[u] >= 0].tolist()
        assert sorted(visited) == sorted(union), (case, u)
        assert len(visited) == len(set(visited)), "a block visited twice"
        for r in range(pa.UNIT_ROWS):
            t = t0 + r // G
            if q_start <= t < q_start + n_q:
                assert counts[u, r] == oracle.visible_count(t, wl.n_sink_blk, wl.n_win_blk), (case, u, r)


def _bf16_bits(x):
    b = np.asarray(x, dtype=np.float32).view(np.uint32)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)  # round to nearest even


def _qcode_rows():
    """bf16 query rows (bit patterns [n, 256]) that exercise the per-row int8
    grid: random normal rows and rows with outliers; rows whose quotients
    q * 127/absmax fall exactly on half-integers (absmax 127 gives 127/absmax
    = 1, absmax 63.5 gives 2: ties to even, both signs, even and odd
    integer parts); an all-zero row; rows holding +absmax and -absmax; a row
    with one non-zero value; tiny and huge magnitudes."""
    rng = np.random.default_rng(61)
    rows = [rng.normal(size=(200, 256)).astype(np.float32)]
    o = rng.normal(size=(40, 256)).astype(np.float32)
    o[np.arange(40), rng.integers(0, 256, 40)] *= 40.0
    rows.append(o)
    k = rng.integers(0, 127, size=(8, 256)).astype(np.float32) + 0.5
    k *= rng.choice([-1.0, 1.0], size=k.shape).astype(np.float32)
    k[:, 0] = 127.0
    rows.append(k)                                      # quotient = q exactly: k + 0.5 ties
    rows.append(k / np.float32(2.0))                    # absmax 63.5: quotient 2 q, again k + 0.5
    rows.append(np.zeros((1, 256), np.float32))         # all zero
    pm = rng.normal(size=(2, 256)).astype(np.float32)
    pm[:, 3], pm[:, 9] = 5.0, -5.0                      # +absmax and -absmax in one row
    rows.append(pm)
    one = np.zeros((2, 256), np.float32)
    one[0, 17], one[1, 200] = -0.7, 3e-3
    rows.append(one)
    rows.append(rng.normal(size=(3, 256)).astype(np.float32) * np.float32([[1e-30], [1e30], [1e-3]]))
    return _bf16_bits(np.concatenate(rows))


def test_q_int8_codes_are_bit_exact():
    """The attention prologue's int8 query grid (PA_Q_INT8), run by the kernel's
    own quantiser, gives the oracle's codes and scales bit for bit: both decide
    in fp32 with IEEE divisions.  More than 128 rows, so several CTAs and a
    ragged last one."""
    import torch

    import windowed_prefill_attention_gb300 as pa
    bits = _qcode_rows()
    q = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    codes, scales = pa.pa_debug_qcodes(q)
    codes, scales = codes.cpu().numpy(), scales.cpu().numpy()
    for i in range(bits.shape[0]):
        want_c, want_s = oracle.quantize_q_row(bits[i])
        assert np.array_equal(codes[i], want_c), i
        assert scales[i].view(np.uint32) == np.float32(want_s).view(np.uint32), i
    # the half-way rows really are ties, decided to even
    tie = bits[240:248]
    assert np.all(np.abs(codes[240:248, 1:]) % 2 == 0)
    assert np.all(np.abs(codes[248:256, 1:]) % 2 == 0)
    assert tie.shape[0] == 8
    assert not codes[256].any() and scales[256] == 0.0
