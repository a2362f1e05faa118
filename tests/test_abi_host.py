"""Host-side checks of the C-ABI library (no GPU): it loads, exports every
symbol include/pa.h declares, validates arguments, and its work planner
covers every query row once with the tiles the mask implies."""
import ctypes as C
import os
import re
import subprocess
import sys

import numpy as np
import pytest

import oracle
from synth import CONFIGS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB = os.path.join(ROOT, "windowed_prefill_attention_gb300", "libpa.so")


@pytest.fixture(scope="module")
def pa():
    subprocess.run([sys.executable, os.path.join(ROOT, "windowed_prefill_attention_gb300", "build.py")], check=True,
                   capture_output=True)
    import windowed_prefill_attention_gb300 as mod
    return mod


def header_symbols(header="pa.h"):
    text = open(os.path.join(ROOT, "include", header)).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_0-9]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(pa):
    lib = C.CDLL(LIB)
    names = header_symbols()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
    assert set(pa.EXPORTED) == set(names)


def test_peak_probe_library_exports_its_header(pa):
    """libpa_peak.so (the tensor-core throughput probe the benchmark's int8
    roofline uses) loads and exports what include/pa_peak.h declares."""
    lib = C.CDLL(os.path.join(os.path.dirname(LIB), "libpa_peak.so"))
    names = header_symbols("pa_peak.h")
    assert names == ["pa_peak_mma_sync"]
    for n in names:
        assert hasattr(lib, n), n
    # bad arguments are rejected before any CUDA call (no GPU needed)
    lib.pa_peak_mma_sync.argtypes = [C.c_int, C.c_int, C.c_longlong, C.c_void_p, C.c_void_p]
    t = C.c_double()
    assert lib.pa_peak_mma_sync(7, 1, 10, C.byref(t), None) == -1
    assert lib.pa_peak_mma_sync(0, 0, 10, C.byref(t), None) == -1
    assert lib.pa_peak_mma_sync(0, 1, 10, None, None) == -1


def test_binding_constants_match_the_header(pa):
    text = open(os.path.join(ROOT, "include", "pa.h")).read()
    assert int(re.search(r"#define PA_UNIT_ROWS (\d+)", text).group(1)) == pa.UNIT_ROWS
    csrc = open(os.path.join(ROOT, "windowed_prefill_attention_gb300", "csrc", "pa_tiles.cuh")).read()
    assert "constexpr int kUnitRows = 2 * kRows;" in csrc and "constexpr int kRows = 128;" in csrc
    assert pa.UNIT_ROWS == 2 * 128


def test_strerror_and_defaults(pa):
    assert pa.pa_strerror(0) == "ok"
    assert "timed out" in pa.pa_strerror(pa.PA_ETIMEOUT)
    o = pa.pa_default_options()
    assert (o.q_mode, o.p_mode, o.wait_timeout_ms, o.record_timing, o.debug_stall) == (0, 0, 2000, 0, 0)


def test_null_handle_and_bad_arguments_are_rejected(pa):
    lib = pa._lib
    null = C.c_void_p()
    assert lib.pa_prefill(null, *([None] * 6), 0, 16, 16, 1, 4, C.c_float(0.1), None, None) == pa.PA_EINVAL
    assert lib.pa_last_error(null, None) == pa.PA_EINVAL
    h = C.c_void_p()
    # head_dim other than 256, page size other than 16, GQA ratio not dividing 128
    assert lib.pa_create(C.byref(h), 16, 2, 128, 16, 10, 10, None) == pa.PA_EINVAL
    assert lib.pa_create(C.byref(h), 16, 2, 256, 32, 10, 10, None) == pa.PA_EINVAL
    assert lib.pa_create(C.byref(h), 12, 4, 256, 16, 10, 10, None) == pa.PA_EINVAL


@pytest.mark.skipif(os.path.exists("/dev/nvidia0"), reason="checks the no-GPU path")
def test_create_without_gpu_fails_cleanly(pa):
    h = C.c_void_p()
    rc = pa._lib.pa_create(C.byref(h), 16, 2, 256, 16, 10, 10, None)
    assert rc in (pa.PA_ECUDA, pa.PA_EARCH)
    assert not h.value


def test_plan_rejects_empty_and_inconsistent_sequences(pa):
    with pytest.raises(pa.PAError):
        pa.pa_plan(16, 2, [(0, 0, 0, 16)], 1, 256)          # n_q = 0
    with pytest.raises(pa.PAError):
        pa.pa_plan(16, 2, [(0, 10, 20, 25)], 1, 256)        # q_start + n_q > n_ctx
    with pytest.raises(pa.PAError):
        pa.pa_plan(16, 2, [(0, -1, 20, 25)], 1, 256)        # negative start


def expected_tiles(block_set):
    """Tiles of a set of key blocks: maximal runs of consecutive blocks, each cut
    into pieces of at most 8 blocks (128-key tiles)."""
    blocks = sorted(block_set)
    n, i = 0, 0
    while i < len(blocks):
        j = i
        while j + 1 < len(blocks) and blocks[j + 1] == blocks[j] + 1:
            j += 1
        n += (j - i + 1 + 7) // 8
        i = j + 1
    return n


PLAN_CASES = [
    ("tiny", CONFIGS["tiny"].n_q_heads, CONFIGS["tiny"].n_kv_heads, [(0, 0, 256, 256)], 0, 16),
    ("4k", 16, 2, [(0, 0, 4096, 4096)], 1, 256),
    ("chunked_ragged", 16, 2, [(0, 1024, 2048, 3072), (2048, 6144, 2048, 8192), (4096, 30720, 2048, 32768),
                               (6144, 12005, 2048, 14053)], 1, 256),
    ("g4_window", 4, 1, [(0, 37, 300, 337)], 2, 3),
    ("g1_causal", 2, 2, [(0, 5, 100, 105)], 1, 0),
    ("g16", 32, 2, [(0, 0, 200, 200)], 1, 4),
]


@pytest.mark.parametrize("case", PLAN_CASES, ids=[c[0] for c in PLAN_CASES])
def test_plan_covers_rows_once_with_mask_tiles(pa, case):
    _, HQ, HKV, seqs, S, W = case
    units, n_tiles, n_rows = pa.pa_plan(HQ, HKV, seqs, S, W)
    G = HQ // HKV
    TQ = pa.UNIT_ROWS // G  # tokens per unit
    covered = {}
    lists_of = {s: oracle.block_lists(q_start, n_q, S, W, cap=4096)
                for s, (_, q_start, n_q, _) in enumerate(seqs)}
    for s, g, t0, tiles in units.tolist():
        q_off, q_start, n_q, n_ctx = seqs[s]
        toks = [t for t in range(t0, t0 + TQ) if q_start <= t < q_start + n_q]
        assert toks, "unit without query rows"
        for t in toks:
            key = (s, t, g)
            assert key not in covered
            covered[key] = True
        # the unit visits the union of its query blocks' visible key blocks
        lists = lists_of[s]
        qb0 = q_start // 16
        union = set()
        for qb in sorted({t // 16 for t in toks}):
            union.update(x for x in lists[qb - qb0].tolist() if x >= 0)
        assert tiles == expected_tiles(union), (s, g, t0)
    want = sum(n_q for _, _, n_q, _ in seqs) * HKV
    assert len(covered) == want
    assert n_tiles == int(units[:, 3].sum())
    assert all(units[i, 3] >= units[i + 1, 3] for i in range(len(units) - 1)), "longest units first"


def test_plan_skips_blocks_no_query_sees(pa):
    # a 2048-token chunk after a 30720-token cache: only the sink block and the
    # window blocks reachable from the chunk are widened
    units, _, rows = pa.pa_plan(16, 2, [(0, 30720, 2048, 32768)], 1, 256)
    first_lo = 30720 // 16 + 1 - 256
    assert rows == 16 * (1 + (32768 // 16 - first_lo))


def test_gloo_two_rank_reduction_and_aggregate():
    """The bench's N>1 bookkeeping: slowest rank's time, whole-job throughput."""
    code = r"""
import os, sys
sys.path.insert(0, %r)
import torch.distributed as dist
import bench
dist.init_process_group("gloo")
r = dist.get_rank()
slow = bench.max_over_ranks(10.0 + 5.0 * r)
v = bench.aggregate_tops(2e12, 10, slow, dist.get_world_size())
print("RANK", r, slow, v, flush=True)
dist.destroy_process_group()
""" % ROOT
    env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(29500 + os.getpid() % 1000), WORLD_SIZE="2")
    procs = []
    for r in range(2):
        e = dict(env, RANK=str(r), LOCAL_RANK=str(r))
        procs.append(subprocess.Popen([sys.executable, "-c", code], env=e, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=120) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e
        _, _, slow, v = o.strip().split()[-4:]
        assert float(slow) == 15.0
        assert abs(float(v) - 2 * 2e12 * 10 / 0.015 / 1e12) < 1e-6


def test_bench_ops_count_matches_oracle_enumeration():
    import bench
    for name in ("tiny", "4k", "32k", "chunked_ragged"):
        wl = CONFIGS[name]
        pairs = sum(oracle.visible_pairs(qs, nq, wl.n_sink_blk, wl.n_win_blk) for qs, nq in wl.seqs)
        assert bench.algorithmic_ops(wl) == 4 * 256 * wl.n_q_heads * pairs


def test_no_product_module_uses_the_oracle():
    pkg = os.path.join(ROOT, "windowed_prefill_attention_gb300")
    pat = re.compile(r"^\s*(import oracle|from oracle)|pa_oracle|_pa_oracle", re.M)
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                assert not pat.search(open(os.path.join(dirpath, f)).read()), f


def _chunk_cases():
    rng = np.random.default_rng(5)
    cases = []
    for name in ("32k", "chunked", "chunked_ragged", "4k"):
        wl = CONFIGS[name]
        offs = np.concatenate([[0], np.cumsum([nq for _, nq in wl.seqs])])
        desc = np.array([(o, qs, nq, qs + nq) for o, (qs, nq) in zip(offs, wl.seqs)], np.int32)
        cases.append((name, wl.n_q_heads, wl.n_kv_heads, desc, 76))
    # unaligned starts, short pieces, several GQA ratios and pair counts
    for i, (hq, hkv, pairs) in enumerate(((16, 2, 76), (8, 4, 76), (4, 4, 7), (32, 2, 1), (16, 2, 200))):
        rows, descs = 0, []
        for _ in range(int(rng.integers(1, 6))):
            q_start = int(rng.integers(0, 20000))
            n_q = int(rng.integers(1, 9000))
            descs.append((rows, q_start, n_q, q_start + n_q + int(rng.integers(0, 50))))
            rows += n_q
        cases.append(("random%d" % i, hq, hkv, np.array(descs, np.int32), pairs))
    return cases


@pytest.mark.parametrize("case", _chunk_cases(), ids=lambda c: c[0])
def test_host_chunks_cut_on_unit_boundaries_and_keep_every_unit_whole(pa, case):
    """The host-buffer path's chunks (pa_host_chunks, the schedule pa_prefill_host
    uses): increasing, ending at the total rows, at most two waves of units
    (+ one unit's rounding) each and one wave (+ the same) for the first and the
    last, a boundary inside a sequence on a multiple of
    a unit's tokens, and no work unit of the call's plan split between chunks."""
    _, hq, hkv, seqs, pairs = case
    ends = pa.pa_host_chunks(hq, hkv, seqs, pairs)
    n_q = seqs[:, 2].astype(np.int64)
    base = np.concatenate([[0], np.cumsum(n_q)])
    total = int(base[-1])
    ut = pa.UNIT_ROWS // (hq // hkv)
    wave = max(ut, pairs * ut // hkv)
    assert ends[-1] == total and np.all(np.diff(ends) > 0)
    sizes = np.diff(np.concatenate([[0], ends]))
    assert np.all(sizes <= 2 * wave + ut)
    assert sizes[0] <= wave + ut and sizes[-1] <= wave + ut
    for e in ends[:-1]:
        s = int(np.searchsorted(base, e, side="right")) - 1
        if base[s] < e < base[s + 1]:
            assert (int(seqs[s, 1]) + int(e - base[s])) % ut == 0
    units, _, _ = pa.pa_plan(hq, hkv, seqs, 1, 256)
    for s, _, t0, _ in units:
        q_start, n = int(seqs[s, 1]), int(seqs[s, 2])
        lo = base[s] + max(int(t0), q_start) - q_start
        hi = base[s] + min(int(t0) + ut, q_start + n) - q_start
        assert lo < hi and not np.any((ends > lo) & (ends < hi)), (s, t0)


def test_host_chunks_rejects_bad_shapes(pa):
    seqs = np.array([[0, 0, 100, 100]], np.int32)
    for args in ((16, 3, seqs, 76), (16, 2, seqs, 0)):
        with pytest.raises(pa.PAError):
            pa.pa_host_chunks(*args)


PAIR_CASES = [
    ("4k", 16, 2, [(0, 0, 4096, 4096)], 1, 256, 76),
    ("chunked_ragged", 16, 2, [(0, 1024, 2048, 3072), (2048, 6144, 2048, 8192), (4096, 30720, 2048, 32768),
                               (6144, 12005, 2048, 14053)], 1, 256, 76),
    ("few_units", 16, 2, [(0, 0, 100, 100)], 1, 256, 76),
    ("g1_causal", 2, 2, [(0, 5, 3000, 3005)], 1, 0, 7),
]


@pytest.mark.parametrize("case", PAIR_CASES, ids=[c[0] for c in PAIR_CASES])
def test_pair_plan_is_a_greedy_longest_first_schedule(pa, case):
    """pa_plan_pairs (how a launch hands pa_plan's units to the kernel's SM
    pairs): the same units, each once, laid out pair by pair, each pair's run
    longest first; replaying the greedy rule (each unit, longest first, to the
    least-loaded pair, ties to the lowest pair; a unit weighs its tiles + 2)
    gives the same assignment, and no pair carries more than the mean load
    plus one unit."""
    _, hq, hkv, seqs, S, W, n_pairs = case
    units, _, _ = pa.pa_plan(hq, hkv, seqs, S, W)
    by_pair, off = pa.pa_plan_pairs(hq, hkv, seqs, S, W, n_pairs)
    n = len(units)
    assert off[0] == 0 and off[-1] == n and np.all(np.diff(off) >= 0)
    assert sorted(map(tuple, by_pair.tolist())) == sorted(map(tuple, units.tolist()))
    load = np.zeros(n_pairs, np.int64)
    want = [[] for _ in range(n_pairs)]
    for u in units.tolist():
        p = int(np.argmin(load))  # argmin: the lowest pair among the least loaded
        want[p].append(tuple(u))
        load[p] += u[3] + 2
    for p in range(n_pairs):
        got = [tuple(x) for x in by_pair[off[p]:off[p + 1]].tolist()]
        assert got == want[p], p
        tiles = [x[3] for x in got]
        assert tiles == sorted(tiles, reverse=True)
    w = units[:, 3].astype(np.int64) + 2
    assert load.max() <= w.sum() / n_pairs + w.max()


def test_pair_plan_rejects_bad_arguments(pa):
    seqs = [(0, 0, 100, 100)]
    with pytest.raises(pa.PAError):
        pa.pa_plan_pairs(16, 2, seqs, 1, 256, 0)
    with pytest.raises(pa.PAError):
        pa.pa_plan_pairs(16, 3, seqs, 1, 256, 76)
