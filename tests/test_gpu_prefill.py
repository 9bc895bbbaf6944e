"""Chain sequences longer than a tree's 32-row limit (prefill segments) in
the same launch as direct rows and tree suffixes: parity with the fp64
oracle, bit-exact invariance of the direct rows, and the device-side limit
on tree sequences (lucebox PR #686, section "Mechanism": the
[prefill][direct/AR][tree] lowering of one verify call)."""
import numpy as np
import pytest

import oracle
import synthetic as sy
from gpu_util import compare, run_gpu
from oracle_parallel import oracle_full

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import speculative_decoding_verify_kv_gb300 as va  # noqa: E402

KERNELS = [0, va.FLAG_CUDA_CORES]


def _full(case, S, flags):
    o, lse = run_gpu(case, num_splits=S, flags=flags)
    O, L = oracle.verify_case(case)
    return compare(o, lse, O, L, f"{case.name} S={S} flags={flags}")


@pytest.mark.parametrize("flags", KERNELS)
def test_prefill_segment_q8_paged_mixed(flags):
    """A 100-row chain (5 row blocks of 128 MMA rows at G = 6), a 40-row
    chain, a direct row and a tree suffix; ragged contexts across tiles."""
    c = sy.make_case("prefill-q8-mixed", num_heads=24, num_kv_heads=4, head_dim=256,
                     kv_dtype=sy.Q8_0, q_dtype=sy.BF16, ctx=[200, 1030, 64, 517],
                     rows=[100, 1, 8, 40], kinds=[0, 0, 1, 0], mode="mixed", paged=True,
                     seed=301)
    _full(c, 3, flags)


@pytest.mark.parametrize("flags", KERNELS)
def test_prefill_chain_bf16_d128(flags):
    """A 200-row chain alone (chain mode), G = 4: 7 row blocks."""
    c = sy.make_case("prefill-bf16-d128", num_heads=32, num_kv_heads=8, head_dim=128,
                     kv_dtype=sy.BF16, q_dtype=sy.BF16, ctx=[700], rows=[200], seed=302)
    _full(c, 2, flags)


def test_direct_rows_invariant_with_prefill_segment():
    c = sy.make_case("prefill-inv", num_heads=24, num_kv_heads=4, head_dim=256,
                     kv_dtype=sy.Q8_0, q_dtype=sy.BF16, ctx=[1016, 1024, 900, 2000],
                     rows=[1, 1, 96, 8], kinds=[0, 0, 0, 1], mode="mixed", paged=True,
                     seed=303)
    o, lse = run_gpu(c, num_splits=8)
    d = sy.subset_sequences(c, [0, 1])
    od, ld = run_gpu(d, num_splits=8)
    assert np.array_equal(o[:2], od) and np.array_equal(lse[:2], ld)


def test_tree_longer_than_mask_is_flagged():
    """A 33-row tree in a mixed launch: VA_DEV_BAD_ROWS, the other sequence
    still correct."""
    c = sy.make_case("tree33", num_heads=8, num_kv_heads=2, head_dim=128, kv_dtype=sy.BF16,
                     q_dtype=sy.BF16, ctx=[40, 50], rows=[4, 33], kinds=[0, 1], mode="mixed",
                     seed=304)
    st = []
    o, lse = run_gpu(c, num_splits=2, status_out=st)
    assert st[0] & va.DEV_BAD_ROWS
    O, L = oracle.verify_case(c, rows=range(4))
    compare(o[:4], lse[:4], O[:4], L[:4], "tree33: chain sequence")
    # The flagged sequence's rows are NaN: the partial kernel writes none of
    # its slots, so whatever the scratch held must not reach O.
    assert np.isnan(o[4:]).all() and np.isnan(lse[4:]).all()


def test_workload_mixed_prefill():
    """The bench's prefill workload (256-row chain at ctx 8192 beside direct
    rows and trees up to ctx 32768) in the bench's configuration, every
    (row, head) against the oracle."""
    c = sy.mixed_prefill()
    o, lse = run_gpu(c, num_splits=8)
    O, L = oracle_full(("mixed_prefill", {}), c)
    assert not np.isnan(L).any()
    compare(o, lse, O, L, f"{c.name} S=8 (every row and head)")


@pytest.mark.parametrize("flags", KERNELS)
def test_prefill_at_the_row_limit(flags):
    """A chain of VA_MAX_ROWS_PER_SEQ (1,024) rows: 32 row blocks of 128
    MMA rows at G = 4, ragged context."""
    assert va.MAX_ROWS_PER_SEQ == 1024
    c = sy.make_case("prefill-1024", num_heads=4, num_kv_heads=1, head_dim=64,
                     kv_dtype=sy.BF16, q_dtype=sy.BF16, ctx=[77], rows=[1024], seed=305)
    _full(c, 2, flags)


def test_prefill_chain_q8_contiguous_g8():
    """A 100-row chain at G = 8 (7 row blocks) over a contiguous Q8_0 cache
    with a multi-tile context, beside a direct row."""
    c = sy.make_case("prefill-q8-g8", num_heads=16, num_kv_heads=2, head_dim=128,
                     kv_dtype=sy.Q8_0, q_dtype=sy.BF16, ctx=[700, 300], rows=[100, 1],
                     seed=306)
    _full(c, 3, 0)
