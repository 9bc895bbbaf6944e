"""Host-only checks of the C ABI: the library loads, exports every symbol
the header declares, and rejects bad arguments before touching a GPU."""
import ctypes
import os
import re
import subprocess

import pytest

import speculative_decoding_verify_kv_gb300 as va

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "verify_attn.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n not in ("defined",)))


def test_header_declares_the_api():
    names = declared_functions()
    for n in ["verify_attn_chain", "verify_attn_tree", "verify_attn_mixed", "va_workspace_size",
              "va_validate", "va_status_string", "va_debug_row_map", "va_debug_gather_index"]:
        assert n in names


def test_library_exports_every_declared_symbol():
    for n in declared_functions():
        assert hasattr(va.lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", va.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line.strip())
    for n in declared_functions():
        assert n in exported, n


def test_binding_lists_every_export():
    assert sorted(va.EXPORTED) == declared_functions()


def test_status_strings():
    for code in range(6):
        assert va.lib.va_status_string(code)
    assert va.lib.va_status_string(99) == b"unknown status"
    assert va.lib.va_version() >= 100


FAKE = 1 << 20  # a 16-byte aligned address that is never dereferenced on the host path


def _problem(**kw):
    d = dict(num_seqs=1, num_heads=24, q_dtype=va.BF16, q=FAKE, cu_rows=FAKE, ctx_len=FAKE,
             parent=FAKE, seq_kind=FAKE, total_rows=16, max_rows_per_seq=16, scale=0.0,
             num_splits=8, flags=0)
    d.update(kw)
    return va.VaProblem(d["num_seqs"], d["num_heads"], d["q_dtype"], d["q"], d["cu_rows"],
                        d["ctx_len"], d["parent"], d["seq_kind"], d["total_rows"],
                        d["max_rows_per_seq"], d["scale"], d["num_splits"], d["flags"])


def _kv(**kw):
    d = dict(dtype=va.Q8_0, num_kv_heads=4, head_dim=256, k=FAKE, v=FAKE, page_size=0,
             capacity=32784, block_table=None, max_blocks_per_seq=0, num_blocks=0,
             draft_k=None, draft_v=None)
    d.update(kw)
    return va.VaKV(d["dtype"], d["num_kv_heads"], d["head_dim"], d["k"], d["v"],
                   d["page_size"], d["capacity"], d["block_table"], d["max_blocks_per_seq"],
                   d["num_blocks"], d["draft_k"], d["draft_v"])


def validate(p, kv, mode=va.MODE_CHAIN, ws=1 << 40):
    return va.lib.va_validate(ctypes.byref(p), ctypes.byref(kv), mode, ws)


def test_validate_ok():
    assert validate(_problem(), _kv()) == 0
    assert validate(_problem(), _kv(page_size=16, capacity=0, block_table=FAKE,
                                    max_blocks_per_seq=2050, num_blocks=2050)) == 0
    assert validate(_problem(q_dtype=va.F32, num_heads=4), _kv(dtype=va.F32, head_dim=64, num_kv_heads=1),
                    ) == 0


@pytest.mark.parametrize("bad,code", [
    (dict(p=dict(num_seqs=0)), 1), (dict(p=dict(num_heads=0)), 1),
    (dict(p=dict(num_splits=0)), 1), (dict(p=dict(max_rows_per_seq=0)), 1),
    (dict(p=dict(q=None)), 1), (dict(p=dict(cu_rows=None)), 1), (dict(p=dict(ctx_len=None)), 1),
    (dict(p=dict(scale=-1.0)), 1), (dict(p=dict(flags=0x80)), 1), (dict(p=dict(q_dtype=7)), 1),
    (dict(kv=dict(k=None)), 1), (dict(kv=dict(dtype=9)), 1), (dict(kv=dict(capacity=0)), 1),
    (dict(kv=dict(page_size=16, block_table=None, max_blocks_per_seq=4, num_blocks=4)), 1),
    (dict(p=dict(num_heads=25)), 2), (dict(kv=dict(head_dim=96)), 2),
    (dict(p=dict(max_rows_per_seq=1025)), 2), (dict(kv=dict(page_size=32)), 2),
    (dict(kv=dict(capacity=100)), 2), (dict(p=dict(num_heads=72)), 2),
    (dict(p=dict(q_dtype=va.F32)), 2), (dict(p=dict(num_splits=1000)), 2),
    (dict(kv=dict(k=FAKE + 8)), 3), (dict(kv=dict(v=FAKE + 2)), 3), (dict(p=dict(q=FAKE + 4)), 3),
])
def test_validate_rejects(bad, code):
    p = _problem(**bad.get("p", {}))
    kv = _kv(**bad.get("kv", {}))
    assert validate(p, kv) == code


def test_row_limits_by_sequence_kind():
    # Chain sequences (prefill segments, draft chains) take up to 1024 rows;
    # a tree launch is limited to 32 rows per sequence (the ancestor mask);
    # a mixed launch defers the tree limit to the device (VA_DEV_BAD_ROWS).
    assert va.MAX_ROWS_PER_SEQ == 1024 and va.MAX_TREE_ROWS == 32
    text = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                             "include", "verify_attn.h")).read()
    assert "#define VA_MAX_ROWS_PER_SEQ 1024" in text and "#define VA_MAX_TREE_ROWS 32" in text
    for mode in (va.MODE_CHAIN, va.MODE_MIXED):
        assert validate(_problem(max_rows_per_seq=1024), _kv(), mode) == 0
        assert validate(_problem(max_rows_per_seq=1025), _kv(), mode) == 2
    assert validate(_problem(max_rows_per_seq=32), _kv(), va.MODE_TREE) == 0
    assert validate(_problem(max_rows_per_seq=33), _kv(), va.MODE_TREE) == 2


def test_tree_and_mixed_need_metadata():
    assert validate(_problem(parent=None), _kv(), va.MODE_TREE) == 1
    assert validate(_problem(parent=None), _kv(), va.MODE_CHAIN) == 0
    assert validate(_problem(seq_kind=None), _kv(), va.MODE_MIXED) == 1
    assert validate(_problem(), _kv(), 3) == 1


def test_workspace_size_and_undersized_workspace():
    p, kv = _problem(), _kv()
    need = va.lib.va_workspace_size(ctypes.byref(p), ctypes.byref(kv))
    info = va.VaPlanInfo()
    assert va.lib.va_plan(ctypes.byref(p), ctypes.byref(kv), 0, ctypes.byref(info)) == 0
    items = info.slots * 16 * 24
    rnd = lambda x: (x + 255) // 256 * 256
    assert need == rnd(items * 256 * 4) + rnd(items * 2 * 4)
    assert validate(p, kv, ws=need) == 0
    assert validate(p, kv, ws=need - 1) == 4
    # the verify entry points refuse an undersized workspace before any launch
    rc = va.lib.verify_attn_chain(ctypes.byref(p), ctypes.byref(kv), FAKE, need - 1, FAKE, FAKE,
                                  None, None)
    assert rc == 4
    assert va.lib.va_workspace_size(None, ctypes.byref(kv)) == 0


def test_plan_does_not_depend_on_other_sequences():
    """Sub-chunk count and slot count come from S, KVH and the SM count only:
    the same sequence planned alone or inside a bigger launch gets the same
    split structure (lucebox PR #686: partitioning that follows launch
    composition changed direct rows)."""
    def info(**kw):
        p = _problem(**kw)
        out = va.VaPlanInfo()
        assert va.lib.va_plan(ctypes.byref(p), ctypes.byref(_kv()), 2, ctypes.byref(out)) == 0
        return out.sub_splits, out.slots

    assert info(num_seqs=2, total_rows=2, max_rows_per_seq=1) == \
        info(num_seqs=8, total_rows=50, max_rows_per_seq=8)


def test_promote_host_checks():
    """verify_attn_promote rejects missing arguments before any device
    access: the tree scratch KV, accepted_len and the status word are
    required, and the usual problem checks apply."""
    P = ctypes.c_void_p
    fn = va.lib.verify_attn_promote

    def call(p, kv, acc=FAKE, nodes=FAKE, status=FAKE):
        return fn(ctypes.byref(p), ctypes.byref(kv), va.MODE_MIXED, P(acc), P(nodes), P(status),
                  None)

    scratch = dict(draft_k=FAKE, draft_v=FAKE)
    assert call(_problem(), _kv()) == 1                                   # no scratch KV
    assert call(_problem(), _kv(**scratch), acc=None) == 1               # no accepted_len
    assert call(_problem(), _kv(**scratch), status=None) == 1            # no status word
    assert call(_problem(), _kv(**scratch), nodes=None) == 1             # rows but no nodes
    assert call(_problem(num_heads=25), _kv(**scratch)) == 2             # problem checks
    assert call(_problem(), _kv(draft_k=FAKE, draft_v=None)) == 1        # half a scratch KV
    assert call(_problem(), _kv(draft_k=FAKE + 8, draft_v=FAKE)) == 3    # unaligned scratch


def _sms():
    """SMs the library plans for: the device's count, or its fallback of
    148 when no GPU is present."""
    try:
        import torch
        if torch.cuda.is_available():
            return torch.cuda.get_device_properties(0).multi_processor_count
    except Exception:
        pass
    return 148


def test_plan_rule():
    """Kernel choice and grid of va_plan (host logic only).  Kernel: the
    row-major tensor-core kernel for bf16 caches without a tree scratch KV
    and for Q8_0 caches except contiguous ones with a scratch KV, which take
    the transposed tensor-core kernel; bf16 with a scratch KV, fp32 caches
    or the flag -> CUDA cores.  Chunk count T = clamp(floor(k * SMs / KVH),
    S, 16 S) with k = 1 (tensor cores) or 2 (CUDA cores); row blocks of 128
    (row-major), 96 (transposed) or 16 (CUDA cores) query rows; one grid z
    per sequence."""
    import numpy as np
    import synthetic as sy
    sms = _sms()

    def plan(case, **kw):
        p, kv, mode = va.upload(case, "cpu", **{k: v for k, v in kw.items() if k != "scratch"})
        if kw.get("scratch"):
            kv.draft_k = kv.draft_v = kv.k
        return va.plan(p, kv, mode)

    def clamp(x, lo, hi):
        return max(lo, min(x, hi))

    q8 = sy.long_q8(ctx=256)                              # H24/KV4/D256, 16 rows, S = 8
    pl = plan(q8)
    T = clamp(sms // 4, 8, 128)
    assert (pl["kernel"], pl["threads"], pl["slots"]) == (va.KERNEL_TENSOR, 640, T)
    assert (pl["grid_x"], pl["grid_y"], pl["grid_z"]) == (T, 4, 1)   # 96 rows: one block
    assert plan(q8, num_splits=1)["slots"] == clamp(sms // 4, 1, 16)
    simt = plan(q8, flags=va.FLAG_CUDA_CORES)
    assert simt["kernel"] == va.KERNEL_CUDA_CORES and simt["slots"] == clamp(2 * sms // 4, 8, 128)
    # grid x: a sequence's row blocks times its chunks, at most max(T, S * blocks)
    assert simt["grid_x"] == max(simt["slots"], 8 * -(-16 * 6 // 16))   # 16-row blocks
    d128 = sy.make_case("p", num_heads=32, num_kv_heads=8, head_dim=128, kv_dtype=sy.BF16,
                        q_dtype=sy.BF16, ctx=[40, 50], rows=[16, 16], paged=True, seed=1)
    pl = plan(d128, num_splits=8)
    assert (pl["kernel"], pl["threads"], pl["slots"], pl["grid_z"]) == \
        (va.KERNEL_TENSOR, 384, clamp(sms // 8, 8, 128), 2)
    long_chain = sy.make_case("c", num_heads=24, num_kv_heads=4, head_dim=256, kv_dtype=sy.Q8_0,
                              q_dtype=sy.BF16, ctx=[40], rows=[100], seed=2)
    pl = plan(long_chain, num_splits=8)
    assert pl["grid_x"] == max(pl["slots"], 8 * 5)         # 600 query rows: 5 blocks of 128
    bf_chain = sy.make_case("c", num_heads=24, num_kv_heads=4, head_dim=256, kv_dtype=sy.BF16,
                            q_dtype=sy.BF16, ctx=[40], rows=[100], seed=2)
    assert plan(bf_chain, num_splits=8)["grid_x"] == max(pl["slots"], 8 * 5)   # blocks of 128
    f32 = sy.tiny_chain()
    assert plan(f32)["kernel"] == va.KERNEL_CUDA_CORES
    mixed = sy.mixed_tree_direct(ctx=[40, 300, 17, 130], direct=(0, 2), num_splits=2, seed=7)
    assert plan(mixed, scratch=True)["kernel"] == va.KERNEL_TENSOR
    tq = plan(sy.to_contiguous(mixed), scratch=True)
    assert (tq["kernel"], tq["threads"]) == (va.KERNEL_TENSOR_Q8, 512)
    assert tq["grid_x"] == tq["slots"]          # 8 rows x G 6 = 48: one 96-row block
    assert plan(d128, num_splits=8, scratch=True)["kernel"] == va.KERNEL_CUDA_CORES
    assert np.isfinite(T)
