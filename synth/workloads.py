"""Workload definitions and seeded input generators.

The workloads stand in for the prompts of the pages' benchmark model (a
head_dim-256 GQA model prefilled at 4k, 32k and 64k context; "int8
tensor-core prefill attention", *Proof of speedup*).  No dataset or trained
weights are involved: queries and keys/values are drawn from N(0, 1), keys and
values get the int8 per-(token, kv-head) quantisation that the paged pool
stores ("fp16 shared-memory tiles for windowed prefill attention",
*Summary*: values "dequantized from the int8 paged KV pool"), and pages are
placed in the pool by a seeded permutation.

Recipe (all draws from ``numpy.random.default_rng(seed)``, in this order):

1. Q: float32 N(0,1) of shape [total_q, HQ, D], rounded to bf16 (nearest-even).
2. For each sequence in order: K then V as float32 N(0,1) [n_ctx, HKV, D].
   If ``outlier_frac`` > 0, ``round(outlier_frac * n_ctx)`` token positions
   (drawn without replacement, once per sequence, shared by K and V and all
   kv heads) are multiplied by 8.
3. Per (token, kv head): scale = absmax / 127 in float32, code =
   clip(rint(x / scale), -127, 127) as int8 (scale 0 and code 0 if absmax = 0).
4. Physical pages: ``rng.permutation(n_pool)`` (identity when
   ``identity_pages``); logical pages are dealt from it round-robin across
   sequences (sequence 0 page 0, sequence 1 page 0, ...), so sequences
   interleave in one shared pool.
5. Pool slots no block-table entry maps, and slots past n_ctx in a
   sequence's last page, hold random int8 codes and NaN scales (they must
   never be read).  Unused block-table entries are -1.
"""
from __future__ import annotations

import dataclasses
from typing import List, Tuple

import numpy as np

HEAD_DIM = 256
PAGE = 16


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    n_q_heads: int
    n_kv_heads: int
    seqs: Tuple[Tuple[int, int], ...]  # (q_start = cached tokens, n_q new tokens) per sequence
    n_sink_blk: int
    n_win_blk: int
    seed: int
    outlier_frac: float = 0.0
    identity_pages: bool = False
    spare_pages: int = 3
    sm_scale: float = 1.0 / 16.0
    head_dim: int = HEAD_DIM
    page_size: int = PAGE

    @property
    def n_ctx(self) -> List[int]:
        return [qs + nq for qs, nq in self.seqs]

    @property
    def total_q(self) -> int:
        return sum(nq for _, nq in self.seqs)

    @property
    def pages_per_seq(self) -> List[int]:
        return [(c + self.page_size - 1) // self.page_size for c in self.n_ctx]

    @property
    def n_pool_pages(self) -> int:
        return sum(self.pages_per_seq) + self.spare_pages

    def scaled(self, name: str, seqs, seed=None) -> "Workload":
        return dataclasses.replace(self, name=name, seqs=tuple(seqs),
                                   seed=self.seed if seed is None else seed)


# The five workloads of the benchmark, in order, plus parity-only variants.
CONFIGS = {
    # 1 sequence of 256 tokens, 4 Q / 1 KV head, window covers everything => plain causal.
    "tiny": Workload("tiny", 4, 1, ((0, 256),), n_sink_blk=0, n_win_blk=16, seed=0,
                     identity_pages=True),
    # 4096 tokens, GQA 16:2, sink 1 block + 256-block window (>= context => causal).
    "4k": Workload("4k", 16, 2, ((0, 4096),), 1, 256, seed=1),
    # 32768 tokens, 4096-token window + 16-token sink, 1% outlier tokens x8.
    "32k": Workload("32k", 16, 2, ((0, 32768),), 1, 256, seed=2, outlier_frac=0.01),
    # 65536 tokens, same distributions as 32k.
    "64k": Workload("64k", 16, 2, ((0, 65536),), 1, 256, seed=3, outlier_frac=0.01),
    # 4 sequences appending a 2048-token chunk to caches of 1024/6144/30720/12000 tokens.
    "chunked": Workload("chunked", 16, 2, ((1024, 2048), (6144, 2048), (30720, 2048), (12000, 2048)),
                        1, 256, seed=4, outlier_frac=0.01),
    # Parity-only: a cache of 12005 tokens gives a q_start off the 16-token grid
    # and a partially filled last page.
    "chunked_ragged": Workload("chunked_ragged", 16, 2,
                               ((1024, 2048), (6144, 2048), (30720, 2048), (12005, 2048)),
                               1, 256, seed=5, outlier_frac=0.01),
    # Beyond the pages' benchmark (they fall back to a token path above 64k):
    # 131072 tokens, same distributions as 32k.
    "128k": Workload("128k", 16, 2, ((0, 131072),), 1, 256, seed=6, outlier_frac=0.01),
}


@dataclasses.dataclass
class Inputs:
    wl: Workload
    q: np.ndarray            # uint16 bf16 bits [total_q, HQ, D]
    k_pool: np.ndarray       # int8 [n_pool, page, HKV, D]
    v_pool: np.ndarray       # int8 [n_pool, page, HKV, D]
    k_scale: np.ndarray      # float32 [n_pool, page, HKV]
    v_scale: np.ndarray      # float32 [n_pool, page, HKV]
    block_table: np.ndarray  # int32 [n_seq, max_pages]
    seq_desc: np.ndarray     # int32 [n_seq, 4] = (q_off, q_start, n_q, n_ctx)

    @property
    def n_seq(self) -> int:
        return self.seq_desc.shape[0]


def _to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _quantize_rows(x: np.ndarray):
    """Symmetric per-row int8: scale = absmax/127, code = clip(rint(x/scale))."""
    absmax = np.abs(x).max(axis=-1)
    scale = (absmax / np.float32(127.0)).astype(np.float32)
    safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    codes = np.clip(np.rint(x / safe[..., None]), -127, 127).astype(np.int8)
    codes[scale == 0] = 0
    return codes, scale


def make_inputs(wl: Workload) -> Inputs:
    rng = np.random.default_rng(wl.seed)
    D, PG, HQ, HKV = wl.head_dim, wl.page_size, wl.n_q_heads, wl.n_kv_heads
    q32 = rng.standard_normal((wl.total_q, HQ, D), dtype=np.float32)
    q = _to_bf16_bits(q32)
    del q32

    n_pool = wl.n_pool_pages
    k_pool = rng.integers(-127, 128, size=(n_pool, PG, HKV, D), dtype=np.int8)
    v_pool = rng.integers(-127, 128, size=(n_pool, PG, HKV, D), dtype=np.int8)
    k_scale = np.full((n_pool, PG, HKV), np.nan, dtype=np.float32)
    v_scale = np.full((n_pool, PG, HKV), np.nan, dtype=np.float32)

    kv_codes = []
    for (qs, nq) in wl.seqs:
        n_ctx = qs + nq
        k = rng.standard_normal((n_ctx, HKV, D), dtype=np.float32)
        v = rng.standard_normal((n_ctx, HKV, D), dtype=np.float32)
        if wl.outlier_frac > 0:
            n_out = int(round(wl.outlier_frac * n_ctx))
            idx = rng.choice(n_ctx, size=n_out, replace=False)
            k[idx] *= np.float32(8.0)
            v[idx] *= np.float32(8.0)
        kc, ks = _quantize_rows(k)
        vc, vs = _quantize_rows(v)
        kv_codes.append((kc, ks, vc, vs))

    perm = np.arange(n_pool) if wl.identity_pages else rng.permutation(n_pool)
    pages = wl.pages_per_seq
    max_pages = max(pages)
    bt = np.full((len(wl.seqs), max_pages), -1, dtype=np.int32)
    nxt = 0
    for lp in range(max_pages):          # deal pages round-robin across sequences
        for s in range(len(wl.seqs)):
            if lp < pages[s]:
                bt[s, lp] = perm[nxt]
                nxt += 1

    for s, (qs, nq) in enumerate(wl.seqs):
        n_ctx = qs + nq
        kc, ks, vc, vs = kv_codes[s]
        for lp in range(pages[s]):
            t0, t1 = lp * PG, min((lp + 1) * PG, n_ctx)
            p = bt[s, lp]
            k_pool[p, : t1 - t0] = kc[t0:t1]
            v_pool[p, : t1 - t0] = vc[t0:t1]
            k_scale[p, : t1 - t0] = ks[t0:t1]
            v_scale[p, : t1 - t0] = vs[t0:t1]

    desc = []
    off = 0
    for (qs, nq) in wl.seqs:
        desc.append((off, qs, nq, qs + nq))
        off += nq
    return Inputs(wl, q, k_pool, v_pool, k_scale, v_scale, bt, np.asarray(desc, dtype=np.int32))


def make_gate(inp: Inputs) -> np.ndarray:
    """Output-gate pre-activations for the gated attention output, bf16 bit
    patterns shaped like q: N(0, 2) from a generator of its own (so every other
    input is unchanged), with 0.1 % of entries at +-40 so that the sigmoid's
    saturated ends are exercised."""
    rng = np.random.default_rng(inp.wl.seed + 7919)
    g = rng.normal(0.0, 2.0, size=inp.q.shape).astype(np.float32)
    n_ext = max(1, g.size // 1000)
    idx = rng.choice(g.size, size=n_ext, replace=False)
    g.reshape(-1)[idx] = rng.choice(np.array([-40.0, 40.0], dtype=np.float32), size=n_ext)
    return _to_bf16_bits(g)
