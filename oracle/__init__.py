"""Oracle for windowed prefill attention over a paged int8 KV pool.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg may use this package; the product path never does.
It is a plain fp64 CPU implementation (``pa_oracle.c``) of

* the definition: causal + sink/window block-masked softmax attention over the
  dequantised paged int8 KV pool ("int8 tensor-core prefill attention",
  sections "Why the attention, and why tensor cores" and "Relation to open PRs";
  "fp16 shared-memory tiles for windowed prefill attention", "Summary"), and
* the pages' quantised method, step by step (int8 Q per row, integer scores,
  online softmax over key tiles, V scale folded into P, P quantised per row),
* the output gate that follows it on the pages' path, out * sigmoid(q_gate)
  ("int8 tensor-core prefill attention", section "Correctness").

It shares no code with the CUDA path.  Parity pins live in tests/.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from .build import build as _build

Q_LOSSLESS, Q_INT8 = 0, 1
P_F16, P_U8, P_EXACT = 0, 1, 2


class _Problem(C.Structure):
    _fields_ = [
        ("n_q_heads", C.c_int), ("n_kv_heads", C.c_int), ("head_dim", C.c_int), ("page_size", C.c_int),
        ("q", C.c_void_p), ("k_pool", C.c_void_p), ("v_pool", C.c_void_p),
        ("k_scale", C.c_void_p), ("v_scale", C.c_void_p),
        ("block_table", C.c_void_p), ("bt_stride", C.c_int),
        ("n_seq", C.c_int), ("seqs", C.c_void_p),
        ("n_sink_blk", C.c_int), ("n_win_blk", C.c_int), ("sm_scale", C.c_double),
    ]


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(_build())
        _lib.pa_oracle_key_visible.restype = C.c_int
        _lib.pa_oracle_key_visible.argtypes = [C.c_int] * 5
        _lib.pa_oracle_visible_count.restype = C.c_longlong
        _lib.pa_oracle_visible_count.argtypes = [C.c_int] * 4
        _lib.pa_oracle_visible_pairs.restype = C.c_longlong
        _lib.pa_oracle_visible_pairs.argtypes = [C.c_int] * 5
        _lib.pa_oracle_block_lists.restype = C.c_int
        _lib.pa_oracle_block_lists.argtypes = [C.c_int] * 6 + [C.c_void_p]
        _lib.pa_oracle_gather.restype = None
        _lib.pa_oracle_gather.argtypes = [C.POINTER(_Problem), C.c_int, C.c_int, C.c_int] + [C.c_void_p] * 4
        _lib.pa_oracle_exact.restype = C.c_int
        _lib.pa_oracle_exact.argtypes = [C.POINTER(_Problem), C.c_int, C.c_void_p, C.c_void_p, C.c_int]
        _lib.pa_oracle_quantize_q_row.restype = None
        _lib.pa_oracle_quantize_q_row.argtypes = [C.c_void_p, C.c_int, C.c_void_p, C.POINTER(C.c_float)]
        _lib.pa_oracle_quantize_p_u8.restype = C.c_double
        _lib.pa_oracle_quantize_p_u8.argtypes = [C.c_void_p, C.c_int, C.c_double, C.c_void_p]
        _lib.pa_oracle_method.restype = C.c_int
        _lib.pa_oracle_method.argtypes = [C.POINTER(_Problem), C.c_int, C.c_void_p, C.c_int, C.c_int,
                                          C.c_int, C.c_void_p, C.c_int]
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(C.c_void_p)


class Problem:
    """Host arrays of one attention call, held alive for the C oracle."""

    def __init__(self, q, k_pool, v_pool, k_scale, v_scale, block_table, seq_desc, n_sink_blk, n_win_blk,
                 sm_scale):
        self.arrays = [np.ascontiguousarray(a) for a in
                       (q, k_pool, v_pool, k_scale, v_scale, block_table, seq_desc)]
        q, kp, vp, ks, vs, bt, sd = self.arrays
        assert q.dtype == np.uint16 and kp.dtype == np.int8 and vp.dtype == np.int8
        assert ks.dtype == np.float32 and vs.dtype == np.float32
        assert bt.dtype == np.int32 and sd.dtype == np.int32
        self.head_dim = q.shape[2]
        self.s = _Problem(q.shape[1], kp.shape[2], q.shape[2], kp.shape[1],
                          _ptr(q).value, _ptr(kp).value, _ptr(vp).value, _ptr(ks).value, _ptr(vs).value,
                          _ptr(bt).value, bt.shape[1], sd.shape[0], _ptr(sd).value,
                          int(n_sink_blk), int(n_win_blk), float(sm_scale))

    @classmethod
    def from_inputs(cls, inp, **override):
        wl = inp.wl
        kw = dict(n_sink_blk=wl.n_sink_blk, n_win_blk=wl.n_win_blk, sm_scale=wl.sm_scale)
        kw.update(override)
        return cls(inp.q, inp.k_pool, inp.v_pool, inp.k_scale, inp.v_scale, inp.block_table, inp.seq_desc, **kw)


def _threads(n_threads):
    return n_threads or len(os.sched_getaffinity(0))


def exact(prob: Problem, rows: np.ndarray, n_threads: int = 0) -> np.ndarray:
    """Exact fp64 output rows; ``rows`` is int32 [n, 2] of (global q row, q head)."""
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    out = np.empty((rows.shape[0], prob.head_dim), dtype=np.float64)
    if lib().pa_oracle_exact(C.byref(prob.s), rows.shape[0], _ptr(rows), _ptr(out), _threads(n_threads)):
        raise ValueError("row outside every sequence")
    return out


def gate(out_rows: np.ndarray, gate_rows: np.ndarray) -> np.ndarray:
    """The gated attention output out * sigmoid(g), elementwise, in fp64:
    sigmoid(g) = 1 / (1 + exp(-g)).  ``gate_rows`` are the gate values of the
    same (row, head) pairs as ``out_rows`` (any float dtype)."""
    g = np.asarray(gate_rows, dtype=np.float64)
    with np.errstate(over="ignore"):  # exp(-g) = inf for g << 0 gives sigmoid 0, as it should
        return np.asarray(out_rows, dtype=np.float64) * (1.0 / (1.0 + np.exp(-g)))


def kv_quantize(x_bits: np.ndarray):
    """The pool's quantisation of K/V rows ("fp16 shared-memory tiles for
    windowed prefill attention", "Summary": int8 pages, per-token per-kv-head
    fp32 scales): for each row of 256 bf16 values (bit patterns, last axis),
    scale = absmax / 127 and code = rint(x / scale), half to even, clamped to
    [-127, 127], decided in fp32 (IEEE-rounded division); scale 0 and codes 0
    for an all-zero row.  Returns (int8 codes, float32 scales)."""
    x = (np.asarray(x_bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
    absmax = np.abs(x).max(axis=-1)
    scale = np.divide(absmax, np.float32(127.0), dtype=np.float32)
    codes = np.zeros(x.shape, dtype=np.int8)
    nz = scale > 0
    q = np.divide(x[nz], scale[nz][:, None], dtype=np.float32)
    codes[nz] = np.clip(np.rint(q), -127, 127).astype(np.int8)
    return codes, scale


def kv_append(k_pool, v_pool, k_scale, v_scale, bt_row, tok_start, k_new_bits, v_new_bits):
    """KV append on host copies of the pool: the new tokens' rows quantised
    (kv_quantize) and placed at page bt_row[t // 16], slot t % 16, kv head g.
    Returns the updated (k_pool, v_pool, k_scale, v_scale)."""
    k_pool, v_pool, k_scale, v_scale = (np.array(a, copy=True) for a in (k_pool, v_pool, k_scale, v_scale))
    kc, ks = kv_quantize(k_new_bits)
    vc, vs = kv_quantize(v_new_bits)
    for i in range(kc.shape[0]):
        t = tok_start + i
        page, slot = int(bt_row[t // 16]), t % 16
        k_pool[page, slot] = kc[i]
        v_pool[page, slot] = vc[i]
        k_scale[page, slot] = ks[i]
        v_scale[page, slot] = vs[i]
    return k_pool, v_pool, k_scale, v_scale


def method(prob: Problem, rows: np.ndarray, q_mode: int, p_mode: int, tile: int = 64,
           n_threads: int = 0) -> np.ndarray:
    """The pages' quantised steps for the given rows (see pa_oracle.c)."""
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    out = np.empty((rows.shape[0], prob.head_dim), dtype=np.float64)
    if lib().pa_oracle_method(C.byref(prob.s), rows.shape[0], _ptr(rows), q_mode, p_mode, tile, _ptr(out),
                              _threads(n_threads)):
        raise ValueError("bad rows or tile")
    return out


def quantize_q_row(q_bits: np.ndarray):
    """int8 codes and float32 scale of one bf16 query row (bit patterns)."""
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    codes = np.empty(q_bits.shape[0], np.int8)
    sc = C.c_float(0.0)
    lib().pa_oracle_quantize_q_row(_ptr(q_bits), q_bits.shape[0], _ptr(codes), C.byref(sc))
    return codes, np.float32(sc.value)


def quantize_p_u8(p: np.ndarray, prev_scale: float = 1.0):
    """u8 codes (as float64) and scale of one row's P' over one key tile."""
    p = np.ascontiguousarray(p, dtype=np.float64)
    out = np.empty_like(p)
    sp = lib().pa_oracle_quantize_p_u8(_ptr(p), p.shape[0], float(prev_scale), _ptr(out))
    return out, sp


def key_visible(t, j, n_sink_blk, n_win_blk, page=16) -> bool:
    return bool(lib().pa_oracle_key_visible(t, j, page, n_sink_blk, n_win_blk))


def visible_count(t, n_sink_blk, n_win_blk, page=16) -> int:
    return int(lib().pa_oracle_visible_count(t, page, n_sink_blk, n_win_blk))


def visible_pairs(q_start, n_q, n_sink_blk, n_win_blk, page=16) -> int:
    return int(lib().pa_oracle_visible_pairs(q_start, n_q, page, n_sink_blk, n_win_blk))


def block_lists(q_start, n_q, n_sink_blk, n_win_blk, cap, page=16) -> np.ndarray:
    n_blk = (q_start + n_q - 1) // page - q_start // page + 1
    out = np.empty((n_blk, cap), dtype=np.int32)
    if lib().pa_oracle_block_lists(q_start, n_q, page, n_sink_blk, n_win_blk, cap, _ptr(out)):
        raise ValueError("cap too small")
    return out


def gather(prob: Problem, s: int, g: int, n_tok: int):
    D = prob.head_dim
    k = np.empty((n_tok, D), np.int8)
    v = np.empty((n_tok, D), np.int8)
    ks = np.empty(n_tok, np.float32)
    vs = np.empty(n_tok, np.float32)
    lib().pa_oracle_gather(C.byref(prob.s), s, g, n_tok, _ptr(k), _ptr(v), _ptr(ks), _ptr(vs))
    return k, v, ks, vs


def all_rows(inp) -> np.ndarray:
    """Every (global q row, q head) pair of a workload."""
    n, h = inp.q.shape[0], inp.q.shape[1]
    ii, hh = np.meshgrid(np.arange(n, dtype=np.int32), np.arange(h, dtype=np.int32), indexing="ij")
    return np.stack([ii.ravel(), hh.ravel()], axis=1)
