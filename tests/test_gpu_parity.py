"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Small cases (several tiles, ragged tails, every dtype, layout and mask kind)
compare every output; the five full-size verify workloads compare sampled
(row, head) outputs the oracle computes one by one, in the launch
configuration the bench times.
"""
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


def full(case, flags=0, num_splits=None, what=""):
    """Every output against the oracle."""
    S = num_splits or case.num_splits
    o, lse = run_gpu(case, num_splits=S, flags=flags)
    O, L = oracle.verify_case(case)
    return compare(o, lse, O, L, what or f"{case.name} S={S} flags={flags}")


# --------------------------------------------------------------------------
# Small cases, every output compared.

@pytest.mark.parametrize("S", [1, 2])
@pytest.mark.parametrize("flags", KERNELS)
def test_tiny_chain_f32(S, flags):
    full(sy.tiny_chain(num_splits=S), flags)


@pytest.mark.parametrize("S", [1, 3])
@pytest.mark.parametrize("flags", KERNELS)
def test_bf16_d256_ragged(S, flags):
    c = sy.make_case("bf16-ragged", num_heads=24, num_kv_heads=4, head_dim=256, kv_dtype=sy.BF16,
                     q_dtype=sy.BF16, ctx=[300], rows=[16], seed=201, q_sigma=0.5, kv_sigma=0.5)
    full(c, flags, S)


@pytest.mark.parametrize("S", [1, 8])
@pytest.mark.parametrize("flags", KERNELS)
def test_q8_d256_ragged(S, flags):
    c = sy.make_case("q8-ragged", num_heads=24, num_kv_heads=4, head_dim=256, kv_dtype=sy.Q8_0,
                     q_dtype=sy.BF16, ctx=[1000], rows=[16], seed=202)
    full(c, flags, S)


@pytest.mark.parametrize("flags", KERNELS)
def test_paged_d128_bf16_small(flags):
    c = sy.make_case("paged-d128-small", num_heads=32, num_kv_heads=8, head_dim=128,
                     kv_dtype=sy.BF16, q_dtype=sy.BF16, ctx=[100, 517, 33], rows=[16, 16, 16],
                     paged=True, seed=203, extra_blocks=5)
    full(c, flags, 2)


@pytest.mark.parametrize("flags", KERNELS)
def test_mixed_small(flags):
    c = sy.mixed_tree_direct(ctx=[100, 130, 70, 33, 48, 16, 1, 64], num_splits=2, seed=204)
    full(c, flags)


@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("kv_dtype", [sy.BF16, sy.Q8_0])
@pytest.mark.parametrize("D", [64, 128])
def test_other_head_dims(kv_dtype, D, paged):
    c = sy.make_case(f"d{D}", num_heads=8, num_kv_heads=2, head_dim=D, kv_dtype=kv_dtype,
                     q_dtype=sy.BF16, ctx=[200, 7], rows=[5, 3], kinds=[1, 0], mode="mixed",
                     paged=paged, seed=205 + D)
    full(c, 0, 3)


@pytest.mark.parametrize("D", [64, 128, 256])
def test_q8_paged_equals_contiguous_bitwise_multi_tile(D):
    """The paged Q8 kernel loads raw rows itself while the contiguous one
    lands them by bulk copy and dequantises in place: same arithmetic, so
    the same bits, over several tiles and a ragged tail."""
    kw = dict(num_heads=8, num_kv_heads=2, head_dim=D, kv_dtype=sy.Q8_0, q_dtype=sy.BF16,
              ctx=[700, 333], rows=[7, 2], seed=230 + D)
    cp = sy.make_case(f"q8-paged-d{D}", paged=True, extra_blocks=3, **kw)
    cc = sy.to_contiguous(cp)
    op, lp = _gpu(cp, 2)
    oc, lc = _gpu(cc, 2)
    assert np.array_equal(op, oc) and np.array_equal(lp, lc)
    full(cp, 0, 2)


def test_f32_cache_bf16_query():
    c = sy.make_case("f32-bf16q", num_heads=4, num_kv_heads=1, head_dim=64, kv_dtype=sy.F32,
                     q_dtype=sy.BF16, ctx=[90], rows=[4], seed=206)
    full(c, 0, 2)


# --------------------------------------------------------------------------
# Edge cases.

@pytest.mark.parametrize("flags", KERNELS)
def test_zero_context(flags):
    c = sy.make_case("ctx0", num_heads=24, num_kv_heads=4, head_dim=256, kv_dtype=sy.Q8_0,
                     q_dtype=sy.BF16, ctx=[0, 0], rows=[1, 16], seed=210)
    full(c, flags, 4)


@pytest.mark.parametrize("flags", KERNELS)
def test_more_splits_than_chunks(flags):
    c = sy.make_case("many-splits", num_heads=8, num_kv_heads=2, head_dim=128, kv_dtype=sy.BF16,
                     q_dtype=sy.BF16, ctx=[20, 300], rows=[2, 4], seed=211)
    full(c, flags, 64)


@pytest.mark.parametrize("flags", KERNELS)
def test_max_rows_and_group(flags):
    """32 rows x G=8 = 256 query rows per KV head (two row blocks)."""
    c = sy.make_case("rows256", num_heads=16, num_kv_heads=2, head_dim=128, kv_dtype=sy.Q8_0,
                     q_dtype=sy.BF16, ctx=[150], rows=[32], mode="tree", seed=212)
    full(c, flags, 2)


@pytest.mark.parametrize("flags", KERNELS)
def test_empty_sequences_in_mixed(flags):
    c = sy.make_case("empty-seqs", num_heads=24, num_kv_heads=4, head_dim=256, kv_dtype=sy.Q8_0,
                     q_dtype=sy.BF16, ctx=[64, 10, 90, 0], rows=[0, 8, 0, 1], kinds=[1, 1, 0, 0],
                     mode="mixed", paged=True, seed=213)
    full(c, flags, 2)


def test_tail_is_never_read():
    """Slots past each span hold NaN bit patterns (the generator's default);
    a finite, correct result shows the kernels mask and never use them."""
    c = sy.make_case("nan-tail", num_heads=24, num_kv_heads=4, head_dim=256, kv_dtype=sy.BF16,
                     q_dtype=sy.BF16, ctx=[77], rows=[9], seed=214, capacity=256)
    full(c, 0, 1)


# --------------------------------------------------------------------------
# Bit-exact structural properties.

def _gpu(case, S, flags=0):
    return run_gpu(case, num_splits=S, flags=flags)


@pytest.mark.parametrize("flags", KERNELS)
def test_paged_equals_contiguous_bitwise(flags):
    c = sy.make_case("pg", num_heads=24, num_kv_heads=4, head_dim=256, kv_dtype=sy.Q8_0,
                     q_dtype=sy.BF16, ctx=[400, 37, 1024], rows=[8, 1, 8], kinds=[1, 0, 1],
                     mode="mixed", paged=True, seed=220, extra_blocks=4)
    a = _gpu(c, 3, flags)
    b = _gpu(sy.to_contiguous(c), 3, flags)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("flags", KERNELS)
def test_tree_with_chain_parents_equals_chain_bitwise(flags):
    c = sy.make_case("ct", num_heads=24, num_kv_heads=4, head_dim=256, kv_dtype=sy.BF16,
                     q_dtype=sy.BF16, ctx=[500], rows=[16], seed=221)
    t = sy.VerifyCase(**{**c.__dict__, "mode": "tree"})
    a, b = _gpu(c, 2, flags), _gpu(t, 2, flags)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("flags", KERNELS)
def test_repeatable_bitwise(flags):
    c = sy.mixed_tree_direct(ctx=[1016, 1024, 1025, 300, 20, 600, 90, 1], seed=222)
    a, b = _gpu(c, 8, flags), _gpu(c, 8, flags)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("flags", KERNELS)
def test_direct_rows_invariant_to_launch_composition(flags):
    """The direct rows of the mixed launch equal, bit for bit, a launch of
    the direct sequences alone (lucebox PR #686: the 1,024-token partition
    boundary changed direct rows when a W8 tree joined the launch)."""
    c = sy.mixed_tree_direct(num_splits=8, seed=223, ctx=[1016, 1024, 1025, 1032, 2048, 3000, 900, 1100])
    o, lse = _gpu(c, 8, flags)
    d = sy.subset_sequences(c, [0, 1])
    od, ld = _gpu(d, 8, flags)
    assert np.array_equal(o[:2], od) and np.array_equal(lse[:2], ld)


def test_direct_rows_invariant_for_every_choice_of_direct_pair():
    ctx = [1016, 1024, 1025, 1032, 300, 1008, 64, 2000]
    for a in range(8):
        for b in range(a + 1, 8):
            c = sy.mixed_tree_direct(num_splits=8, seed=224, ctx=ctx, direct=(a, b))
            o, lse = _gpu(c, 8)
            d = sy.subset_sequences(c, [a, b])
            od, ld = _gpu(d, 8)
            ra, rb = int(c.cu_rows[a]), int(c.cu_rows[b])
            assert np.array_equal(o[[ra, rb]], od) and np.array_equal(lse[[ra, rb]], ld), (a, b)


def test_debug_row_map_matches_oracle():
    c = sy.mixed_tree_direct(ctx=[10, 20, 30, 40, 50, 60, 70, 80], seed=225)
    p, kv, mode = va.upload(c, "cuda")
    row_seq, anc = va.debug_row_map(p, mode)
    ref_seq, ref_anc = oracle.row_map(c.cu_rows, c.parent, c.seq_kind, c.mode)
    assert np.array_equal(row_seq.cpu().numpy(), ref_seq)
    assert np.array_equal(anc.cpu().numpy().view(np.uint32), ref_anc)


@pytest.mark.parametrize("paged", [False, True])
def test_debug_gather_matches_oracle(paged):
    c = sy.make_case("gather", num_heads=8, num_kv_heads=2, head_dim=128, kv_dtype=sy.Q8_0,
                     q_dtype=sy.BF16, ctx=[33, 200, 16], rows=[3, 1, 8], paged=paged, seed=226,
                     extra_blocks=7)
    p, kv, mode = va.upload(c, "cuda")
    max_len = int(c.kv_len.max()) + 5
    for kvh in range(2):
        got = va.debug_gather_index(p, kv, kvh, max_len).cpu().numpy()
        for s in range(c.num_seqs):
            L = int(c.kv_len[s])
            ref = oracle.gather_index(s, kvh, np.arange(L), page_size=c.page_size,
                                      capacity=c.capacity, num_kv_heads=2,
                                      block_table=c.block_table)
            assert np.array_equal(got[s, :L], ref)
            assert (got[s, L:] == -1).all()


# --------------------------------------------------------------------------
# Device-detected data errors: flagged, rows NaN, no fault.

def _status_of(case, S=2):
    st = []
    o, lse = run_gpu(case, num_splits=S, status_out=st)
    return st[0], o, lse


def test_bad_parent_is_flagged():
    c = sy.make_case("badp", num_heads=8, num_kv_heads=2, head_dim=128, kv_dtype=sy.BF16,
                     q_dtype=sy.BF16, ctx=[50, 60], rows=[4, 4], mode="tree", seed=230)
    c.parent[5] = 3  # row 1 of sequence 1 points at a later node
    st, o, lse = _status_of(c)
    assert st & va.DEV_BAD_PARENT
    assert np.isnan(lse[4:]).all() and np.isfinite(lse[:4]).all()


def test_bad_block_is_flagged():
    c = sy.make_case("badb", num_heads=8, num_kv_heads=2, head_dim=128, kv_dtype=sy.Q8_0,
                     q_dtype=sy.BF16, ctx=[50, 60], rows=[4, 4], paged=True, seed=231)
    c.block_table[1, 1] = 10_000
    st, o, lse = _status_of(c)
    assert st & va.DEV_BAD_BLOCK
    assert np.isfinite(lse[:4]).all()


def test_context_overflow_is_flagged():
    c = sy.make_case("ovf", num_heads=8, num_kv_heads=2, head_dim=128, kv_dtype=sy.BF16,
                     q_dtype=sy.BF16, ctx=[50, 60], rows=[4, 4], seed=232)
    c.ctx_len[1] = 70  # 70 + 4 > capacity 64
    st, o, lse = _status_of(c)
    assert st & va.DEV_CTX_OVERFLOW
    assert np.isnan(lse[4:]).all() and np.isfinite(lse[:4]).all()


# --------------------------------------------------------------------------
# The five verify workloads at full size, in the bench's launch configuration,
# every (row, head) against the oracle (run over the host's cores).

def full_size(recipe, S, flags=0):
    case = getattr(sy, recipe[0])(**recipe[1])
    o, lse = run_gpu(case, num_splits=S, flags=flags)
    O, L = oracle_full(recipe, case)
    assert not np.isnan(L).any()
    return compare(o, lse, O, L, f"{case.name} S={S} (every row and head)")


@pytest.mark.parametrize("S", [1, 8])
def test_workload_dflash_bf16_ctx4096_full(S):
    full(sy.dflash_bf16(ctx=4096), 0, S)


@pytest.mark.parametrize("S", [1, 8])
def test_workload_dflash_bf16_ctx8192(S):
    full_size(("dflash_bf16", {"ctx": 8192}), S)


@pytest.mark.parametrize("ctx", [8192, 20676, 32768])
def test_workload_long_q8(ctx):
    full_size(("long_q8", {"ctx": ctx}), 8)


def test_workload_paged_d128():
    full_size(("paged_d128", {}), 8)


def test_workload_paged_d128_q8():
    """The batched D=128 shape over a paged Q8_0 cache (the Q8 D=128 path)."""
    full_size(("paged_d128", {"kv_dtype": sy.Q8_0}), 8)


def test_workload_mixed_tree_direct():
    c = sy.mixed_tree_direct()
    full_size(("mixed_tree_direct", {}), 8)
    o, lse = _gpu(c, 8)
    d = sy.subset_sequences(c, [0, 1])
    od, ld = _gpu(d, 8)
    assert np.array_equal(o[:2], od) and np.array_equal(lse[:2], ld)
