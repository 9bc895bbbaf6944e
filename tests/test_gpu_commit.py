"""Tree scratch KV and the tree commit of the KV on the GPU (lucebox PR
#686, "State and commit invariants": tree rows write scratch KV; the commit
promotes only the accepted prefix and preflights before any mutation)."""
import numpy as np
import pytest

import oracle
import oracle.verify_oracle as orc
import synthetic as sy
from gpu_util import compare, run_gpu

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import speculative_decoding_verify_kv_gb300 as va  # noqa: E402

KERNELS = [0, va.FLAG_CUDA_CORES]


def _mixed_q8_paged(seed=401):
    return sy.make_case("scratch-q8", num_heads=24, num_kv_heads=4, head_dim=256,
                        kv_dtype=sy.Q8_0, q_dtype=sy.BF16, ctx=[1016, 300, 77, 1030, 0],
                        rows=[8, 1, 8, 40, 8], kinds=[1, 0, 1, 0, 1], mode="mixed",
                        paged=True, seed=seed)


@pytest.mark.parametrize("flags", KERNELS)
def test_scratch_equals_drafts_in_cache_bitwise(flags):
    """Moving the tree drafts into the scratch KV (and NaN-filling their old
    cache rows) changes no output bit."""
    c = _mixed_q8_paged()
    a = run_gpu(c, num_splits=8, flags=flags)
    b = run_gpu(sy.with_tree_scratch(c), num_splits=8, flags=flags)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_scratch_q8_paged_runs_on_tensor_cores_and_matches_oracle():
    c = sy.with_tree_scratch(_mixed_q8_paged(402))
    p, kv, mode = va.upload(c, "cuda", num_splits=3)
    assert va.plan(p, kv, mode)["kernel"] == va.KERNEL_TENSOR
    o, lse = run_gpu(c, num_splits=3)
    O, L = oracle.verify_case(c)
    compare(o, lse, O, L, "scratch q8 paged")


def test_scratch_q8_contiguous_runs_on_the_transposed_kernel_and_matches_oracle():
    """A contiguous Q8_0 cache with a tree scratch KV runs on the transposed
    tensor-core kernel (tokens on M); every output against the oracle."""
    base = sy.to_contiguous(_mixed_q8_paged(403))
    c = sy.with_tree_scratch(base)
    p, kv, mode = va.upload(c, "cuda", num_splits=3)
    assert va.plan(p, kv, mode)["kernel"] == va.KERNEL_TENSOR_Q8
    o, lse = run_gpu(c, num_splits=3)
    O, L = oracle.verify_case(c)
    compare(o, lse, O, L, "scratch q8 contiguous")


@pytest.mark.parametrize("paged", [False, True])
def test_scratch_bf16_uses_cuda_cores_and_matches_oracle(paged):
    c = sy.with_tree_scratch(sy.make_case(
        "scratch-bf16", num_heads=8, num_kv_heads=2, head_dim=128, kv_dtype=sy.BF16,
        q_dtype=sy.BF16, ctx=[130, 64, 9], rows=[8, 3, 5], kinds=[1, 0, 1], mode="mixed",
        paged=paged, seed=403))
    p, kv, mode = va.upload(c, "cuda", num_splits=2)
    assert va.plan(p, kv, mode)["kernel"] == 0
    o, lse = run_gpu(c, num_splits=2)
    O, L = oracle.verify_case(c)
    compare(o, lse, O, L, f"scratch bf16 paged={paged}")


def _storage(t, like):
    a = t.cpu().numpy()
    return a.view(like.dtype) if a.dtype != like.dtype else a


def _promote_gpu(c, acc, nodes):
    p, kv, mode = va.upload(c, "cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    va.verify_attn_promote(p, kv, mode, torch.from_numpy(acc).cuda(),
                           torch.from_numpy(nodes).cuda(), status)
    torch.cuda.synchronize()
    return _storage(kv.k, c.k), _storage(kv.v, c.v), int(status.item())


def _promote_oracle(c, acc, nodes):
    return orc.promote(c.k, c.v, c.draft_k, c.draft_v, ctx_len=c.ctx_len, cu_rows=c.cu_rows,
                       parent=c.parent, seq_kind=c.seq_kind, mode=c.mode, accepted_len=acc,
                       accepted_nodes=nodes, page_size=c.page_size, capacity=c.capacity,
                       num_kv_heads=c.num_kv_heads, block_table=c.block_table)


@pytest.mark.parametrize("kv_dtype,D,paged", [(sy.Q8_0, 256, True), (sy.Q8_0, 128, False),
                                              (sy.BF16, 128, True), (sy.F32, 64, False)])
def test_promote_matches_oracle_bitwise(kv_dtype, D, paged):
    c = sy.with_tree_scratch(sy.make_case(
        "commit", num_heads=8, num_kv_heads=2, head_dim=D, kv_dtype=kv_dtype,
        q_dtype=sy.F32 if kv_dtype == sy.F32 else sy.BF16, ctx=[14, 40, 3, 100],
        rows=[8, 1, 8, 8], kinds=[1, 0, 1, 1], mode="mixed", paged=paged, seed=404))
    acc, nodes = sy.accepted_paths(c, 405)
    assert acc.sum() > 0
    k, v, st = _promote_gpu(c, acc, nodes)
    k2, v2, bad = _promote_oracle(c, acc, nodes)
    assert st == 0 and not bad
    # byte for byte (the NaN patterns of unused rows included)
    assert np.array_equal(k.view(np.uint8), k2.view(np.uint8))
    assert np.array_equal(v.view(np.uint8), v2.view(np.uint8))


def test_promote_preflight_failure_writes_nothing():
    c = sy.with_tree_scratch(sy.make_case(
        "commit-bad", num_heads=8, num_kv_heads=2, head_dim=128, kv_dtype=sy.Q8_0,
        q_dtype=sy.BF16, ctx=[20, 30], rows=[8, 8], kinds=[1, 1], mode="mixed", paged=True,
        seed=406))
    acc, nodes = sy.accepted_paths(c, 407)
    # Sequence 1: a path that skips a tree level (not a root path).
    lo = int(c.cu_rows[1])
    deep = [j for j in range(8) if int(c.parent[lo + j]) >= 0]
    acc[1], nodes[lo:lo + 8] = 1, [deep[0]] + [-1] * 7
    k, v, st = _promote_gpu(c, acc, nodes)
    assert st & va.DEV_BAD_PARENT
    assert np.array_equal(k.view(np.uint8), c.k.view(np.uint8))
    assert np.array_equal(v.view(np.uint8), c.v.view(np.uint8))


def test_accepted_rows_as_chain_over_committed_cache():
    """Commit on the GPU, then verify the accepted paths as chains over the
    committed cache on the GPU: matches the oracle (which shows, exactly,
    that these equal the tree rows of the scratch launch)."""
    c = sy.with_tree_scratch(_mixed_q8_paged(408))
    acc, nodes = sy.accepted_paths(c, 409)
    k, v, st = _promote_gpu(c, acc, nodes)
    assert st == 0
    ch = sy.accepted_as_chains(c, k, v, acc, nodes)
    o, lse = run_gpu(ch, num_splits=8)
    O, L = oracle.verify_case(ch)
    compare(o, lse, O, L, "accepted paths as chains")
