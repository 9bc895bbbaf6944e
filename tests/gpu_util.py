"""Helpers for the GPU parity tests: run a case through the C ABI and
compare with the fp64 oracle at the stated tolerances."""
from __future__ import annotations

import numpy as np

# Tolerances against the fp64 oracle: O max-abs and relative L2 over the
# compared entries, LSE max-abs.
O_MAX_ABS = 2e-3
O_REL_L2 = 1e-3
LSE_MAX_ABS = 1e-4


def run_gpu(case, num_splits=None, flags=0, device="cuda", status_out=None):
    import torch

    import speculative_decoding_verify_kv_gb300 as va
    p, kv, mode = va.upload(case, device, num_splits=num_splits, flags=flags)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    o, lse = va.verify_attn(p, kv, mode, status=status)
    torch.cuda.synchronize()
    st = int(status.item())
    if status_out is not None:
        status_out.append(st)
    else:
        assert st == 0, f"device status {st:#x}"
    return o.cpu().numpy(), lse.cpu().numpy()


FP16_UNIT_ROUNDOFF = 2.0 ** -11


def q8_lse_bound(case):
    """Per (row, head) bound on the LSE error of the Q8 tensor-core path.

    That path rounds each dequantised K element once to fp16 (relative error
    at most u = 2^-11) and keeps Q exact, so every score moves by at most
    scale * u * sum_d |q_d k_td|, and LSE (a smooth maximum of the scores)
    by at most the largest such move over the visible tokens.  Returns an
    array [total_rows, H] (NaN where no bound was needed)."""
    import oracle.verify_oracle as orc
    H, KVH, D = case.num_heads, case.num_kv_heads, case.head_dim
    G = H // KVH
    Q = orc.decode_q(case.q, case.q_dtype)
    out = np.full((case.total_rows, H), np.nan)
    for s in range(case.num_seqs):
        lo, hi = int(case.cu_rows[s]), int(case.cu_rows[s + 1])
        if hi == lo:
            continue
        ctx = int(case.ctx_len[s])
        kind = orc.seq_kind_of(s, case.seq_kind, case.mode)
        draft = getattr(case, "draft_k", None) if kind == 1 else None
        for kvh in range(KVH):
            K = orc.decode_rows(orc.span_rows(case.k, draft, s, kvh, ctx, hi - lo, lo,
                                              page_size=case.page_size, capacity=case.capacity,
                                              num_kv_heads=KVH, block_table=case.block_table),
                                case.kv_dtype)
            for r in range(lo, hi):
                pos = orc.visible_positions(ctx, hi - lo, kind, case.parent[lo:hi], r - lo)
                for h in range(kvh * G, (kvh + 1) * G):
                    out[r, h] = case.scale * FP16_UNIT_ROUNDOFF * float(
                        (np.abs(K[pos]) @ np.abs(Q[r, h])).max())
    return out


def compare(o, lse, O, L, what="", lse_tol=None):
    """Compare GPU (o, lse) with oracle (O, L) on the entries the oracle
    computed (non-NaN LSE).  ``lse_tol`` (per entry) replaces the LSE bound
    where the arithmetic of the path under test fixes a different one."""
    sel = ~np.isnan(L)
    assert sel.any(), "nothing to compare"
    go, ro = o[sel].astype(np.float64), O[sel]
    gl, rl = lse[sel].astype(np.float64), L[sel]
    assert np.isfinite(go).all() and np.isfinite(gl).all(), f"{what}: non-finite GPU output"
    d = go - ro
    max_abs = float(np.abs(d).max())
    rel = float(np.linalg.norm(d) / max(np.linalg.norm(ro), 1e-30))
    lerr = np.abs(gl - rl)
    lse_err = float(lerr.max())
    tol = LSE_MAX_ABS if lse_tol is None else np.maximum(LSE_MAX_ABS, lse_tol[sel])
    msg = f"{what}: max|dO|={max_abs:.3e} relL2={rel:.3e} max|dLSE|={lse_err:.3e}"
    assert max_abs <= O_MAX_ABS and rel <= O_REL_L2 and bool(np.all(lerr <= tol)), msg
    return max_abs, rel, lse_err


def sample_rows_heads(case):
    """Rows {first, middle, last} of each sequence and heads at the edges
    of the first and last GQA groups."""
    rows = set()
    for s in range(case.num_seqs):
        lo, hi = int(case.cu_rows[s]), int(case.cu_rows[s + 1])
        if hi > lo:
            rows |= {lo, (lo + hi - 1) // 2, hi - 1}
    G = case.num_heads // case.num_kv_heads
    heads = sorted({0, G - 1, G, case.num_heads - 1} & set(range(case.num_heads)))
    return sorted(rows), heads
