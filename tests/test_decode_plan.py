"""CPU: the decode's work split (pa_decode_plan, the host half of pa_decode).

The launch's (sequence, kv head) pairs laid end to end give one list of
visible blocks; each CTA computes a run of it.  These invariants hold for any
split the kernel can compute correctly: the runs cover the list once, in
order; a run is at most 128 blocks (32 per warp); each run's first sequence is
the one its first block belongs to; the CTAs that meet a pair hold the
partial slots 0, 1, ... in order; a one-wave split fits the slots it was given
and its runs stay within the cost budget (blocks + 16 per extra pair).
"""
import numpy as np
import pytest

import windowed_prefill_attention_gb300 as pa

SEG_COST = 16


def _n_vis(n_ctx, S, W):
    last = (n_ctx - 1) // 16
    lo = max(0, last + 1 - W) if W > 0 else 0
    ns = min(max(S, 0), lo) if W > 0 else 0
    return ns + (last - lo + 1)


def _seqs(ctxs):
    return np.array([(i, c - 1, 1, c) for i, c in enumerate(ctxs)], dtype=np.int32)


def _check(ctxs, hkv, slots, S, W):
    runs, per_cta, max_slots, listed, total = pa.pa_decode_plan(hkv, slots, _seqs(ctxs), S, W)
    n = min(len(ctxs), 512)
    nv = [_n_vis(c, S, W) for c in ctxs[:n]]
    starts = np.concatenate([[0], np.cumsum(np.repeat(nv, hkv))])  # pair starts, sequence-major
    assert total == starts[-1]
    x0 = runs[:, 0].astype(np.int64)
    ends = np.append(x0[1:], total)
    assert x0[0] == 0 and np.all(ends > x0) and np.all(ends - x0 <= 128)
    # each run's sequence holds its first block
    pair_of = np.searchsorted(starts, x0, side="right") - 1
    assert np.array_equal(runs[:, 1], pair_of // hkv)
    # partial slots: the CTAs meeting a pair, in order, hold 0, 1, 2, ...
    met = {}
    for c in range(len(runs)):
        p = pair_of[c]
        first = True
        while p < len(starts) - 1 and starts[p] < ends[c]:
            slot = runs[c, 2] if first and x0[c] > starts[p] else 0
            met.setdefault(p, []).append(int(slot))
            first = False
            p += 1
    for p, slots_ in met.items():
        assert slots_ == list(range(len(slots_))), (p, slots_)
    assert max_slots >= max(len(v) for v in met.values())
    if listed:
        assert len(runs) <= min(slots, 512) and per_cta <= 128
        for c in range(len(runs)):
            n_pairs = int(np.searchsorted(starts, ends[c], side="left") - pair_of[c])
            assert (ends[c] - x0[c]) + SEG_COST * (n_pairs - 1) <= per_cta
    else:
        assert per_cta <= 128 and np.array_equal(x0, np.arange(len(runs)) * per_cta)
    return runs, per_cta, max_slots, listed, total


def test_bench_workload_is_one_balanced_wave():
    runs, per_cta, max_slots, listed, total = _check([32768] * 64, 2, 304, 1, 256)
    assert listed and total == 64 * 2 * 257 and len(runs) <= 304
    # equal cost: every run but the last is within one pair-crossing of the budget
    lens = np.diff(np.append(runs[:, 0], total))
    assert lens[:-1].min() >= per_cta - SEG_COST


@pytest.mark.parametrize("ctxs,hkv,S,W", [
    ([4096, 32000, 17, 1, 12005, 256, 257, 4112, 65536], 2, 1, 256),
    ([5000, 129, 70000], 8, 1, 256),
    ([300, 5000, 16, 4097], 2, 1, 0),
    (list(np.random.default_rng(7).integers(1, 300, 600)), 2, 1, 8),  # two launches: the first is planned
    ([40000, 36001, 1], 2, 1, 0),
])
def test_split_invariants(ctxs, hkv, S, W):
    _check([int(c) for c in ctxs], hkv, 304, S, W)


def test_more_than_one_wave_falls_back_to_equal_runs():
    runs, per_cta, _, listed, total = _check([70000] * 9 + [69999], 1, 304, 1, 0)
    assert not listed and total > 304 * 128
    assert len(runs) == -(-total // per_cta)


def test_few_slots_and_tiny_contexts():
    _check([1, 2, 15, 16, 17, 33], 4, 1, 1, 2)
    _check([1] * 40, 2, 10, 0, 4)


def test_rejects_non_decode_queries_and_bad_shapes():
    bad = _seqs([100, 200])
    bad[1, 2] = 2  # two query tokens
    with pytest.raises(pa.PAError):
        pa.pa_decode_plan(2, 304, bad, 1, 8)
    with pytest.raises(pa.PAError):
        pa.pa_decode_plan(2, 0, _seqs([100]), 1, 8)
    with pytest.raises(pa.PAError):
        pa.pa_decode_plan(9, 304, _seqs([100]), 1, 8)
