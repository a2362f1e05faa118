"""Shared helpers for the tests: device upload, a call through the C ABI, and
the parity measures (normalised by max(1, |ref|) as the tolerance states)."""
import numpy as np

import oracle

# Tolerance of the path against the fp64 definition: max |err| <= 3e-2 * max(1, |ref|)
# and mean |err| / max(1, |ref|) <= 1e-2.
TOL_MAX = 3e-2
TOL_MEAN = 1e-2


def to_device(inp, device="cuda"):
    import torch
    return dict(q=torch.from_numpy(inp.q.view(np.int16)).view(torch.bfloat16).to(device),
                k_pool=torch.from_numpy(inp.k_pool).to(device), v_pool=torch.from_numpy(inp.v_pool).to(device),
                k_scale=torch.from_numpy(inp.k_scale).to(device), v_scale=torch.from_numpy(inp.v_scale).to(device),
                block_table=torch.from_numpy(inp.block_table).to(device))


def run_gpu(inp, S=None, W=None, sm_scale=None, gate_bits=None, **opts):
    """One pa_prefill_batch call (pa_prefill_batch_gated when gate_bits, bf16 bit
    patterns shaped like q, is given); returns (out as float32 numpy [total_q,
    HQ, D], device status)."""
    import torch

    import windowed_prefill_attention_gb300 as pa
    wl = inp.wl
    S = wl.n_sink_blk if S is None else S
    W = wl.n_win_blk if W is None else W
    sm_scale = wl.sm_scale if sm_scale is None else sm_scale
    d = to_device(inp)
    out = torch.full_like(d["q"], float("nan"))
    h = pa.pa_create(wl.n_q_heads, wl.n_kv_heads, inp.k_pool.shape[0], inp.block_table.shape[1], **opts)
    try:
        q_gate = None
        if gate_bits is not None:
            q_gate = torch.from_numpy(np.ascontiguousarray(gate_bits).view(np.int16)).view(torch.bfloat16).cuda()
        pa.pa_prefill_batch(h, inp.seq_desc, d["q"], d["k_pool"], d["v_pool"], d["k_scale"], d["v_scale"],
                            d["block_table"], S, W, sm_scale, out, q_gate=q_gate)
        rc = pa.pa_last_error(h)
    finally:
        pa.pa_destroy(h)
    return out.float().cpu().numpy(), rc


def sample_rows(inp, n_tokens, seed=0, edge=20):
    """(global row, head) pairs: every head of `n_tokens` random tokens plus the
    first and last `edge` tokens of each sequence and tokens around 16-blocks."""
    rng = np.random.default_rng(seed)
    toks = set()
    for q_off, q_start, n_q, _ in inp.seq_desc.tolist():
        toks.update(range(q_off, q_off + min(edge, n_q)))
        toks.update(range(q_off + max(0, n_q - edge), q_off + n_q))
        for b in (q_off + 4096 - q_start, q_off + 4112 - q_start, q_off + 16 - q_start % 16):
            toks.update(t for t in range(b - 2, b + 2) if q_off <= t < q_off + n_q)
    total = inp.q.shape[0]
    toks.update(rng.choice(total, size=min(n_tokens, total), replace=False).tolist())
    toks = np.array(sorted(toks), dtype=np.int32)
    heads = np.arange(inp.q.shape[1], dtype=np.int32)
    return np.stack(np.meshgrid(toks, heads, indexing="ij"), -1).reshape(-1, 2)


def norm_errors(got, ref):
    e = np.abs(got - ref) / np.maximum(1.0, np.abs(ref))
    return float(e.max()), float(e.mean())


def compare(out, inp, rows, **prob_kw):
    """Normalised max / mean error of the GPU rows against the exact oracle."""
    prob = oracle.Problem.from_inputs(inp, **prob_kw)
    ref = oracle.exact(prob, rows)
    got = out[rows[:, 0], rows[:, 1]].astype(np.float64)
    assert np.isfinite(got).all()
    return norm_errors(got, ref)
