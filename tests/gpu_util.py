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


def compare(o, lse, O, L, what=""):
    """Compare GPU (o, lse) with oracle (O, L) on the entries the oracle
    computed (non-NaN LSE), at the flat tolerances above."""
    sel = ~np.isnan(L)
    assert sel.any(), "nothing to compare"
    go, ro = o[sel].astype(np.float64), O[sel]
    gl, rl = lse[sel].astype(np.float64), L[sel]
    assert np.isfinite(go).all() and np.isfinite(gl).all(), f"{what}: non-finite GPU output"
    d = go - ro
    max_abs = float(np.abs(d).max())
    rel = float(np.linalg.norm(d) / max(np.linalg.norm(ro), 1e-30))
    lse_err = float(np.abs(gl - rl).max())
    msg = f"{what}: max|dO|={max_abs:.3e} relL2={rel:.3e} max|dLSE|={lse_err:.3e}"
    assert max_abs <= O_MAX_ABS and rel <= O_REL_L2 and lse_err <= LSE_MAX_ABS, msg
    return max_abs, rel, lse_err


