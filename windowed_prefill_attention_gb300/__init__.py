"""GB300 (sm_103a) windowed prefill attention over a paged int8 KV pool.

A thin ctypes binding over ``libpa.so`` (C ABI in ``include/pa.h``).  The
functions keep the C names; they only marshal arguments (torch tensors for
device memory, the current torch stream) and raise on a non-zero status.
Every step of the computation runs in the library's CUDA kernels; there is no
CPU or PyTorch fallback: if the library is missing this module fails to import.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libpa.so")

if not os.path.exists(_LIB_PATH):
    raise ImportError("libpa.so is not built; run `python -c \"import __graft_entry__ as g; g.build()\"` "
                      "or `python windowed_prefill_attention_gb300/build.py`")

_lib = C.CDLL(_LIB_PATH)

PA_OK, PA_EINVAL, PA_EARCH, PA_ECUDA, PA_ETIMEOUT, PA_EBADPAGE, PA_ENOMEM, PA_ENOSCRATCH = 0, -1, -2, -3, -4, -5, -6, -7
PA_NOALLOC_SCRATCH_BYTES = 32 << 20
# query rows per work unit (PA_UNIT_ROWS in include/pa.h)
UNIT_ROWS = 256
PA_Q_BF16, PA_Q_INT8 = 0, 1
PA_P_F16, PA_P_U8 = 0, 1

EXPORTED = ("pa_default_options", "pa_create", "pa_destroy", "pa_prefill", "pa_prefill_batch",
            "pa_prefill_batch_gated", "pa_prefill_host", "pa_kv_append", "pa_decode",
            "pa_last_error", "pa_timing", "pa_strerror", "pa_plan", "pa_plan_pairs", "pa_host_chunks", "pa_decode_plan",
            "pa_debug_gather",
            "pa_debug_maskset", "pa_debug_qcodes", "pa_debug_copy_streams_idle", "pa_prefill_noalloc",
            "pa_debug_noalloc_units")


class pa_options(C.Structure):
    _fields_ = [("q_mode", C.c_int), ("p_mode", C.c_int), ("wait_timeout_ms", C.c_int), ("record_timing", C.c_int),
                ("debug_stall", C.c_int), ("debug_fail_host", C.c_int)]


class pa_seq(C.Structure):
    _fields_ = [("q_off", C.c_int), ("q_start", C.c_int), ("n_q", C.c_int), ("n_ctx", C.c_int)]


_vp, _i, _f = C.c_void_p, C.c_int, C.c_float
_lib.pa_default_options.argtypes = [C.POINTER(pa_options)]
_lib.pa_default_options.restype = None
_lib.pa_create.argtypes = [C.POINTER(_vp), _i, _i, _i, _i, _i, _i, C.POINTER(pa_options)]
_lib.pa_destroy.argtypes = [_vp]
_lib.pa_destroy.restype = None
_lib.pa_prefill.argtypes = [_vp] + [_vp] * 6 + [_i] * 5 + [_f, _vp, _vp]
_lib.pa_prefill_batch.argtypes = [_vp, _i, C.POINTER(pa_seq)] + [_vp] * 6 + [_i, _i, _f, _vp, _vp]
_lib.pa_prefill_host.argtypes = _lib.pa_prefill_batch.argtypes
_lib.pa_prefill_batch_gated.argtypes = [_vp, _i, C.POINTER(pa_seq)] + [_vp] * 7 + [_i, _i, _f, _vp, _vp]
_lib.pa_kv_append.argtypes = [_vp, _vp, _vp, _i, _i] + [_vp] * 6
_lib.pa_decode.argtypes = _lib.pa_prefill_batch.argtypes
_lib.pa_last_error.argtypes = [_vp, _vp]
_lib.pa_timing.argtypes = [_vp, _i, C.POINTER(C.c_double), C.POINTER(C.c_double), C.POINTER(_i)]
_lib.pa_strerror.argtypes = [_i]
_lib.pa_strerror.restype = C.c_char_p
_lib.pa_plan.argtypes = [_i, _i, _i, C.POINTER(pa_seq), _i, _i, _vp, _i, C.POINTER(_i), C.POINTER(C.c_longlong),
                         C.POINTER(_i)]
_lib.pa_plan_pairs.argtypes = [_i, _i, _i, C.POINTER(pa_seq), _i, _i, _i, _vp, _i, _vp, C.POINTER(_i)]
_lib.pa_host_chunks.argtypes = [_i, _i, _i, C.POINTER(pa_seq), _i, _vp, _i, C.POINTER(_i)]
_lib.pa_decode_plan.argtypes = [_i, _i, _i, C.POINTER(pa_seq), _i, _i, _vp, _i, C.POINTER(_i), C.POINTER(_i),
                                C.POINTER(_i), C.POINTER(_i), C.POINTER(C.c_longlong)]
_lib.pa_debug_gather.argtypes = ([_vp, _i, C.POINTER(pa_seq)] + [_vp] * 5 + [_i, _i, _i] + [_vp] * 5
                                 + [_i, C.POINTER(_i), _vp])
_lib.pa_debug_maskset.argtypes = [_vp, _i, C.POINTER(pa_seq), _i, _i, _vp, _vp, _i, _vp, _i, C.POINTER(_i), _vp]
_lib.pa_debug_qcodes.argtypes = [_vp, _i, _vp, _vp, _vp]
_lib.pa_debug_copy_streams_idle.argtypes = [_vp]
_lib.pa_prefill_noalloc.argtypes = [_i] * 4 + [_vp] * 6 + [_i] * 5 + [_f, _vp, _vp]
_lib.pa_debug_noalloc_units.argtypes = [_i, _vp, _vp]


class PAError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__("%s: %s (%d)" % (where, pa_strerror(code), code))
        self.code = code


def pa_strerror(code: int) -> str:
    return _lib.pa_strerror(code).decode()


def _check(code: int, where: str) -> int:
    if code != PA_OK:
        raise PAError(code, where)
    return code


def _seqs(seqs):
    """[(q_off, q_start, n_q, n_ctx), ...] or an int array [n, 4] -> ctypes array."""
    arr = np.asarray(seqs, dtype=np.int64).reshape(-1, 4)
    if arr.size and (int(arr.min()) < -2**31 or int(arr.max()) >= 2**31):
        raise ValueError("sequence fields must fit int32")
    return (pa_seq * arr.shape[0]).from_buffer_copy(np.ascontiguousarray(arr, dtype=np.int32))


def _dev(t, dtype, name):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return C.c_void_p(t.data_ptr())


def _host(a, name):
    import torch
    if isinstance(a, torch.Tensor):
        if a.is_cuda or not a.is_contiguous():
            raise TypeError("%s must be a contiguous host tensor" % name)
        return C.c_void_p(a.data_ptr())
    a = np.asarray(a)
    if not a.flags["C_CONTIGUOUS"]:
        raise ValueError("%s must be contiguous" % name)
    return a.ctypes.data_as(C.c_void_p)


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def pa_default_options() -> pa_options:
    o = pa_options()
    _lib.pa_default_options(C.byref(o))
    return o


def pa_create(n_q_heads, n_kv_heads, n_pool_pages, max_pages_per_seq, head_dim=256, page_size=16,
              q_mode=PA_Q_BF16, p_mode=PA_P_F16, wait_timeout_ms=2000, record_timing=False, debug_stall=False,
              debug_fail_host=False):
    o = pa_options(q_mode, p_mode, wait_timeout_ms, 1 if record_timing else 0, 1 if debug_stall else 0,
                   1 if debug_fail_host else 0)
    h = C.c_void_p()
    _check(_lib.pa_create(C.byref(h), n_q_heads, n_kv_heads, head_dim, page_size, n_pool_pages, max_pages_per_seq,
                          C.byref(o)), "pa_create")
    return h


def pa_destroy(h) -> None:
    _lib.pa_destroy(h)


def _dev_inputs(q, k_pool, v_pool, k_scale, v_scale, block_table):
    import torch
    return [_dev(q, torch.bfloat16, "q"), _dev(k_pool, torch.int8, "k_pool"), _dev(v_pool, torch.int8, "v_pool"),
            _dev(k_scale, torch.float32, "k_scale"), _dev(v_scale, torch.float32, "v_scale"),
            _dev(block_table, torch.int32, "block_table")]


def pa_prefill(h, q, k_pool, v_pool, k_scale, v_scale, block_table, q_start, n_q, n_ctx, n_sink_blk, n_win_blk,
               sm_scale, out, stream=None) -> None:
    import torch
    args = _dev_inputs(q, k_pool, v_pool, k_scale, v_scale, block_table)
    _check(_lib.pa_prefill(h, *args, q_start, n_q, n_ctx, n_sink_blk, n_win_blk, float(sm_scale),
                           _dev(out, torch.bfloat16, "out"), _stream(stream)), "pa_prefill")


def pa_prefill_batch(h, seqs, q, k_pool, v_pool, k_scale, v_scale, block_table, n_sink_blk, n_win_blk, sm_scale,
                     out, stream=None, q_gate=None) -> None:
    """q_gate (bf16, shaped like out) selects pa_prefill_batch_gated."""
    import torch
    s = _seqs(seqs)
    args = _dev_inputs(q, k_pool, v_pool, k_scale, v_scale, block_table)
    if q_gate is None:
        _check(_lib.pa_prefill_batch(h, len(s), s, *args, n_sink_blk, n_win_blk, float(sm_scale),
                                     _dev(out, torch.bfloat16, "out"), _stream(stream)), "pa_prefill_batch")
    else:
        _check(_lib.pa_prefill_batch_gated(h, len(s), s, args[0], _dev(q_gate, torch.bfloat16, "q_gate"), *args[1:],
                                           n_sink_blk, n_win_blk, float(sm_scale), _dev(out, torch.bfloat16, "out"),
                                           _stream(stream)), "pa_prefill_batch_gated")


def pa_decode(h, seqs, q, k_pool, v_pool, k_scale, v_scale, block_table, n_sink_blk, n_win_blk, sm_scale, out,
              stream=None) -> None:
    """One new token per sequence (seqs rows (q_off, n_ctx - 1, 1, n_ctx))."""
    import torch
    s = _seqs(seqs)
    args = _dev_inputs(q, k_pool, v_pool, k_scale, v_scale, block_table)
    _check(_lib.pa_decode(h, len(s), s, *args, n_sink_blk, n_win_blk, float(sm_scale),
                          _dev(out, torch.bfloat16, "out"), _stream(stream)), "pa_decode")


def pa_kv_append(h, k_new, v_new, tok_start, block_table_row, k_pool, v_pool, k_scale, v_scale,
                 stream=None) -> None:
    """Quantise the new tokens' K/V rows (bf16 [n_new, HKV, 256]) into the pool."""
    import torch
    n_new = int(k_new.shape[0])
    _check(_lib.pa_kv_append(h, _dev(k_new, torch.bfloat16, "k_new"), _dev(v_new, torch.bfloat16, "v_new"), n_new,
                             int(tok_start), _dev(block_table_row, torch.int32, "block_table_row"),
                             _dev(k_pool, torch.int8, "k_pool"), _dev(v_pool, torch.int8, "v_pool"),
                             _dev(k_scale, torch.float32, "k_scale"), _dev(v_scale, torch.float32, "v_scale"),
                             _stream(stream)), "pa_kv_append")


def pa_prefill_host(h, seqs, q, k_pool, v_pool, k_scale, v_scale, block_table, n_sink_blk, n_win_blk, sm_scale,
                    out, stream=None) -> None:
    """Host buffers (numpy arrays or CPU tensors; pinned is fastest); synchronous."""
    s = _seqs(seqs)
    args = [_host(a, n) for a, n in ((q, "q"), (k_pool, "k_pool"), (v_pool, "v_pool"), (k_scale, "k_scale"),
                                     (v_scale, "v_scale"), (block_table, "block_table"))]
    _check(_lib.pa_prefill_host(h, len(s), s, *args, n_sink_blk, n_win_blk, float(sm_scale), _host(out, "out"),
                                _stream(stream)), "pa_prefill_host")


def pa_prefill_noalloc(n_q_heads, n_kv_heads, n_pool_pages, max_pages_per_seq, q, k_pool, v_pool, k_scale, v_scale,
                       block_table, q_start, n_q, n_ctx, n_sink_blk, n_win_blk, sm_scale, out, stream=None) -> None:
    """Handle-free pa_prefill whose scratch is a static device array (no allocation); synchronous."""
    import torch
    args = _dev_inputs(q, k_pool, v_pool, k_scale, v_scale, block_table)
    _check(_lib.pa_prefill_noalloc(n_q_heads, n_kv_heads, n_pool_pages, max_pages_per_seq, *args, q_start, n_q, n_ctx,
                                   n_sink_blk, n_win_blk, float(sm_scale), _dev(out, torch.bfloat16, "out"),
                                   _stream(stream)), "pa_prefill_noalloc")


def pa_debug_noalloc_units(n_units, stream=None):
    """The work list (int32 [n_units, 4]) the last pa_prefill_noalloc call on the current device built."""
    units = np.zeros((n_units, 4), dtype=np.int32)
    _check(_lib.pa_debug_noalloc_units(n_units, units.ctypes.data_as(C.c_void_p), _stream(stream)),
           "pa_debug_noalloc_units")
    return units


def pa_debug_copy_streams_idle(h) -> bool:
    """True if the handle's host-path copy streams have no work pending (does not wait)."""
    r = _lib.pa_debug_copy_streams_idle(h)
    if r < 0:
        raise PAError(r, "pa_debug_copy_streams_idle")
    return r == 1


def pa_last_error(h, stream=None) -> int:
    """Synchronise and return the first device-side status since the last call (0 = fine)."""
    return _lib.pa_last_error(h, _stream(stream))


def pa_timing(h, reset=False):
    w, a, n = C.c_double(), C.c_double(), C.c_int()
    _check(_lib.pa_timing(h, 1 if reset else 0, C.byref(w), C.byref(a), C.byref(n)), "pa_timing")
    return w.value, a.value, n.value


def pa_plan(n_q_heads, n_kv_heads, seqs, n_sink_blk, n_win_blk):
    """Host-only work plan: (units int32 [n, 4] = seq, kv head, first token, tiles; total tiles; widened rows)."""
    s = _seqs(seqs)
    n_units, n_tiles, n_rows = C.c_int(), C.c_longlong(), C.c_int()
    _check(_lib.pa_plan(n_q_heads, n_kv_heads, len(s), s, n_sink_blk, n_win_blk, None, 0, C.byref(n_units),
                        C.byref(n_tiles), C.byref(n_rows)), "pa_plan")
    units = np.zeros((n_units.value, 4), dtype=np.int32)
    _check(_lib.pa_plan(n_q_heads, n_kv_heads, len(s), s, n_sink_blk, n_win_blk, units.ctypes.data_as(C.c_void_p),
                        n_units.value, C.byref(n_units), C.byref(n_tiles), C.byref(n_rows)), "pa_plan")
    return units, n_tiles.value, n_rows.value


def pa_plan_pairs(n_q_heads, n_kv_heads, seqs, n_sink_blk, n_win_blk, n_pairs):
    """Host-only: pa_plan's units as a launch hands them to n_pairs SM pairs.  Returns
    (units int32 [n, 4] laid out pair by pair, pair_off int32 [n_pairs + 1])."""
    s = _seqs(seqs)
    n = C.c_int()
    off = np.zeros(n_pairs + 1, dtype=np.int32)
    _check(_lib.pa_plan_pairs(n_q_heads, n_kv_heads, len(s), s, n_sink_blk, n_win_blk, n_pairs, None, 0,
                              off.ctypes.data_as(C.c_void_p), C.byref(n)), "pa_plan_pairs")
    units = np.zeros((n.value, 4), dtype=np.int32)
    _check(_lib.pa_plan_pairs(n_q_heads, n_kv_heads, len(s), s, n_sink_blk, n_win_blk, n_pairs,
                              units.ctypes.data_as(C.c_void_p), n.value, off.ctypes.data_as(C.c_void_p),
                              C.byref(n)), "pa_plan_pairs")
    return units, off


def pa_host_chunks(n_q_heads, n_kv_heads, seqs, n_pairs):
    """Host-only: the chunk ends (rows of the sequences laid end to end) of pa_prefill_host."""
    s = _seqs(seqs)
    n = C.c_int()
    _check(_lib.pa_host_chunks(n_q_heads, n_kv_heads, len(s), s, n_pairs, None, 0, C.byref(n)), "pa_host_chunks")
    ends = np.zeros(n.value, dtype=np.int64)
    _check(_lib.pa_host_chunks(n_q_heads, n_kv_heads, len(s), s, n_pairs, ends.ctypes.data_as(C.c_void_p), n.value,
                               C.byref(n)), "pa_host_chunks")
    return ends


def pa_decode_plan(n_kv_heads, slots, seqs, n_sink_blk, n_win_blk):
    """Host-only: pa_decode's work split of one launch.  Returns (runs int32 [n_cta, 3] =
    first block, sequence, partial slot; per_cta; max_slots; listed; total blocks)."""
    s = _seqs(seqs)
    n_cta, per_cta, max_slots, listed, total = C.c_int(), C.c_int(), C.c_int(), C.c_int(), C.c_longlong()
    args = lambda buf, cap: (n_kv_heads, slots, len(s), s, n_sink_blk, n_win_blk, buf, cap, C.byref(n_cta),  # noqa: E731
                             C.byref(per_cta), C.byref(max_slots), C.byref(listed), C.byref(total))
    _check(_lib.pa_decode_plan(*args(None, 0)), "pa_decode_plan")
    runs = np.zeros((n_cta.value, 3), dtype=np.int32)
    _check(_lib.pa_decode_plan(*args(runs.ctypes.data_as(C.c_void_p), n_cta.value)), "pa_decode_plan")
    return runs, per_cta.value, max_slots.value, bool(listed.value), total.value


def pa_debug_gather(h, seqs, k_pool, v_pool, k_scale, v_scale, block_table, n_sink_blk, n_win_blk, seq, cap,
                    stream=None):
    """Widened rows of sequence `seq` as the kernels see them (int8 codes, scales, logical token of each row)."""
    import torch
    s = _seqs(seqs)
    dev = k_pool.device
    hkv = k_pool.shape[2]
    k_out = torch.empty((hkv, cap, 256), dtype=torch.int8, device=dev)
    v_out = torch.empty_like(k_out)
    ks_out = torch.empty((hkv, cap), dtype=torch.float32, device=dev)
    vs_out = torch.empty_like(ks_out)
    tok = torch.empty((cap,), dtype=torch.int32, device=dev)
    n = C.c_int()
    _check(_lib.pa_debug_gather(h, len(s), s, _dev(k_pool, torch.int8, "k_pool"), _dev(v_pool, torch.int8, "v_pool"),
                                _dev(k_scale, torch.float32, "k_scale"), _dev(v_scale, torch.float32, "v_scale"),
                                _dev(block_table, torch.int32, "block_table"), n_sink_blk, n_win_blk, seq,
                                C.c_void_p(k_out.data_ptr()), C.c_void_p(v_out.data_ptr()),
                                C.c_void_p(ks_out.data_ptr()), C.c_void_p(vs_out.data_ptr()),
                                C.c_void_p(tok.data_ptr()), cap, C.byref(n), _stream(stream)), "pa_debug_gather")
    r = n.value
    # the export packs rows densely as [HKV][n_rows]
    k_flat = k_out.reshape(-1)[: hkv * r * 256].reshape(hkv, r, 256)
    v_flat = v_out.reshape(-1)[: hkv * r * 256].reshape(hkv, r, 256)
    ks = ks_out.reshape(-1)[: hkv * r].reshape(hkv, r)
    vs = vs_out.reshape(-1)[: hkv * r].reshape(hkv, r)
    return k_flat, v_flat, ks, vs, tok[:r]


def pa_debug_maskset(h, seqs, n_sink_blk, n_win_blk, units_cap, cap, stream=None):
    """Per unit: visited key blocks and per-row admitted key counts (see include/pa.h)."""
    import torch
    s = _seqs(seqs)
    counts = torch.empty((units_cap, UNIT_ROWS), dtype=torch.int32, device="cuda")
    blocks = torch.empty((units_cap, cap), dtype=torch.int32, device="cuda")
    units = np.zeros((units_cap, 4), dtype=np.int32)
    n = C.c_int()
    _check(_lib.pa_debug_maskset(h, len(s), s, n_sink_blk, n_win_blk, C.c_void_p(counts.data_ptr()),
                                 C.c_void_p(blocks.data_ptr()), cap, units.ctypes.data_as(C.c_void_p), units_cap,
                                 C.byref(n), _stream(stream)), "pa_debug_maskset")
    k = n.value
    return units[:k], counts[:k], blocks[:k]


def pa_debug_qcodes(q_rows, stream=None):
    """The attention prologue's int8 query grid on bf16 rows [n, 256]: (int8 codes [n, 256], fp32 scales [n])."""
    import torch
    n = int(q_rows.shape[0])
    codes = torch.empty((n, 256), dtype=torch.int8, device=q_rows.device)
    scales = torch.empty((n,), dtype=torch.float32, device=q_rows.device)
    _check(_lib.pa_debug_qcodes(_dev(q_rows, torch.bfloat16, "q_rows"), n, C.c_void_p(codes.data_ptr()),
                                C.c_void_p(scales.data_ptr()), _stream(stream)), "pa_debug_qcodes")
    return codes, scales


class Handle:
    """Owns a pa_handle; ``close()`` (or garbage collection) destroys it."""

    def __init__(self, n_q_heads, n_kv_heads, n_pool_pages, max_pages_per_seq, **opts):
        self.h = pa_create(n_q_heads, n_kv_heads, n_pool_pages, max_pages_per_seq, **opts)
        self.n_q_heads, self.n_kv_heads = n_q_heads, n_kv_heads

    def close(self):
        if self.h is not None:
            pa_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
