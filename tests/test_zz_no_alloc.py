"""The verify entry point that runs on library-held scratch
(``verify_attn_noalloc``: no workspace argument, no allocation on the call
path), checked against the entry points that take a caller workspace.

Collected last on purpose: it must pass alone and after every other test
(the scratch is shared by all calls on a device and holds no state)."""
import ctypes
import os
import re

import numpy as np
import pytest

import speculative_decoding_verify_kv_gb300 as va
import synthetic as sy

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "verify_attn.h")


def test_static_limit_matches_header():
    text = open(HEADER).read()
    m = re.search(r"#define VA_STATIC_WORKSPACE_BYTES \((\d+)u \* (\d+)u \* (\d+)u\)", text)
    assert m, "VA_STATIC_WORKSPACE_BYTES not found"
    assert int(m.group(1)) * int(m.group(2)) * int(m.group(3)) == va.STATIC_WORKSPACE_BYTES


def _host_problem(case):
    """The case's arrays as host tensors: enough for the host-side checks,
    which run before any device access."""
    return va.upload(case, "cpu")


def test_oversized_problem_is_rejected_before_launch():
    # 2 x 16 chain rows, H24/KV4/D256, S=8: 32 slots x 32 rows x 24 heads x
    # (256 + 2) x 4 B of partials = 25 MB > 16 MiB.
    case = sy.make_case("oversized", num_heads=24, num_kv_heads=4, head_dim=256,
                        kv_dtype=sy.Q8_0, q_dtype=sy.BF16, ctx=[64, 64], rows=[16, 16],
                        seed=11, num_splits=8)
    p, kv, mode = _host_problem(case)
    assert va.workspace_size(p, kv) > va.STATIC_WORKSPACE_BYTES
    import torch
    o = torch.empty((case.total_rows, case.num_heads, case.head_dim), dtype=torch.float32)
    lse = torch.empty((case.total_rows, case.num_heads), dtype=torch.float32)
    # Straight through the C ABI with the default stream: the size check
    # comes before any CUDA call, so this runs without a GPU.
    st = va.lib.verify_attn_noalloc(ctypes.byref(p.c()), ctypes.byref(kv.c()), mode,
                                    o.data_ptr(), lse.data_ptr(), None, None)
    assert st == 4  # VA_ERR_WORKSPACE_TOO_SMALL


def test_headline_problem_fits():
    p, kv, _ = _host_problem(sy.long_q8(ctx=256))
    assert 0 < va.workspace_size(p, kv) <= va.STATIC_WORKSPACE_BYTES


CASES = {
    # the benchmark's call: 1 x 16 chain rows, H24/KV4/D256, Q8_0, S = 8
    "long-q8-ctx32768": lambda: sy.long_q8(ctx=32768),
    # direct rows and tree suffixes in one launch over a paged Q8_0 cache
    "mixed-small": lambda: sy.mixed_tree_direct(ctx=[40, 300, 17, 130], direct=(0, 2),
                                                num_splits=2, seed=7),
}


@pytest.mark.gpu
@pytest.mark.parametrize("name", sorted(CASES))
def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row(name):
    import torch
    case = CASES[name]()
    p, kv, mode = va.upload(case, "cuda")
    assert va.workspace_size(p, kv) <= va.STATIC_WORKSPACE_BYTES
    st_ref = torch.zeros(1, dtype=torch.int32, device="cuda")
    o_ref, l_ref = va.verify_attn(p, kv, mode, status=st_ref)
    torch.cuda.synchronize()
    assert int(st_ref.item()) == 0
    o_ref, l_ref = o_ref.cpu().numpy(), l_ref.cpu().numpy()

    o = torch.empty((case.total_rows, case.num_heads, case.head_dim), dtype=torch.float32,
                    device="cuda")
    lse = torch.empty((case.total_rows, case.num_heads), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    free = []
    for call in range(2):
        o.fill_(float("nan"))
        lse.fill_(float("nan"))
        torch.cuda.synchronize()
        va.verify_attn_noalloc(p, kv, mode, o, lse, status=status)
        torch.cuda.synchronize()
        free.append(torch.cuda.mem_get_info()[0])
        assert int(status.item()) == 0, f"call {call}: device status {int(status.item()):#x}"
        go, gl = o.cpu().numpy(), lse.cpu().numpy()
        assert np.isfinite(go).all() and np.isfinite(gl).all(), f"call {call}: unwritten output"
        # Same plan, same kernels, same arithmetic: only the scratch address
        # differs, so the outputs are the same bits.
        assert np.array_equal(go.view(np.uint32), o_ref.view(np.uint32)), (
            f"call {call}: O differs from the workspace entry point in "
            f"{int((go.view(np.uint32) != o_ref.view(np.uint32)).sum())} elements")
        assert np.array_equal(gl.view(np.uint32), l_ref.view(np.uint32)), (
            f"call {call}: LSE differs from the workspace entry point")
    # The second call allocated no device memory.
    assert free[1] == free[0]
