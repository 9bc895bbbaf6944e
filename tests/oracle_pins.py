"""Pins for the fp64 oracle: checks that tie it to something other than
itself (hand-worked fixtures, library routines, brute force, closed forms and
invariants).  Each ``check_*`` raises AssertionError on a mismatch; the
oracle tests call them directly and the mutation tests call them on an
oracle with a planted mistake, expecting a failure.
"""
from __future__ import annotations

import json
import math
import os
import struct

import numpy as np

import oracle.verify_oracle as orc
import synthetic as sy

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _val(x):
    if isinstance(x, list) and x and x[0] == "ln":
        return math.log(x[1])
    if x == "inf":
        return math.inf
    if x == "-inf":
        return -math.inf
    return float(x)


# ---------------------------------------------------------------------------
# Storage decoding.

def check_fp16_golden():
    d = load("fp16_bits.json")
    for b, v in d["cases"]:
        got = float(orc.decode_fp16(np.array([int(b, 16)], dtype=np.uint16))[0])
        want = _val(v)
        assert got == want and math.copysign(1, got) == math.copysign(1, want), (b, got, want)


def check_fp16_all_patterns():
    """Every non-NaN binary16 pattern against numpy's own float16 type."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = orc.decode_fp16(bits)
    ok = np.isnan(ref) == np.isnan(got)
    fin = ~np.isnan(ref)
    assert ok.all()
    assert np.array_equal(got[fin], ref[fin])


def check_bf16_decode():
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 65536, size=4096).astype(np.uint16)
    got = orc.decode_bf16(bits)
    ref = np.array([struct.unpack("<f", struct.pack("<I", int(b) << 16))[0] for b in bits])
    fin = ~np.isnan(ref)
    assert np.array_equal(np.isnan(got), ~fin)
    assert np.array_equal(got[fin], ref[fin])
    assert orc.decode_bf16(np.array([0x3F80]))[0] == 1.0
    assert orc.decode_bf16(np.array([0xC040]))[0] == -3.0


def check_q8_golden():
    d = load("q8_0_blocks.json")
    for blk in d["blocks"]:
        sb = int(blk["scale_bits"], 16)
        raw = np.zeros(34, dtype=np.uint8)
        raw[0], raw[1] = sb & 0xFF, sb >> 8
        raw[2:] = np.asarray(blk["codes"], dtype=np.int8).view(np.uint8)
        got = orc.dequant_q8_0(raw)
        assert np.array_equal(got, np.asarray(blk["values"], dtype=np.float64)), (blk["scale_bits"], got)
    # two blocks in one row, each with its own scale
    raw = np.zeros(68, dtype=np.uint8)
    for i, blk in enumerate(d["blocks"][:2]):
        sb = int(blk["scale_bits"], 16)
        raw[34 * i], raw[34 * i + 1] = sb & 0xFF, sb >> 8
        raw[34 * i + 2:34 * i + 34] = np.asarray(blk["codes"], dtype=np.int8).view(np.uint8)
    got = orc.dequant_q8_0(raw)
    want = np.concatenate([d["blocks"][0]["values"], d["blocks"][1]["values"]])
    assert np.array_equal(got, want)


# ---------------------------------------------------------------------------
# Masks, row map, split rule and page addressing.

def check_tree_masks_golden():
    d = load("tree_masks.json")
    for c in d["cases"]:
        masks = orc.row_masks(len(c["parent"]), c["kind"], np.asarray(c["parent"]))
        if "masks" in c:
            assert masks == c["masks"], (c["name"], masks)
        else:
            assert masks[-1] == c["masks_last"], (c["name"], masks[-1])


def check_row_map_mixed():
    parent = np.array([-1, -1, 0, 0, 1, 1, 2, -1, 6, -1, 0, 1], dtype=np.int32)
    cu = np.array([0, 1, 9, 9, 12], dtype=np.int32)     # direct, tree of 8, empty, chain of 3
    kind = np.array([0, 1, 0, 0], dtype=np.uint8)
    row_seq, masks = orc.row_map(cu, parent, kind, "mixed")
    assert row_seq.tolist() == [0, 1, 1, 1, 1, 1, 1, 1, 1, 3, 3, 3]
    # tree part: parent [-1,0,0,1,1,2,-1,6] -> masks by hand 1,3,5,11,19,37,64,192
    assert masks.tolist() == [1, 1, 3, 5, 11, 19, 37, 64, 192, 1, 3, 7]


def check_split_golden():
    d = load("split_plan.json")
    for c in d["cases"]:
        got = [list(r) for r in orc.split_ranges(c["L"], c["S"])]
        assert got == c["ranges"], (c["L"], c["S"], got)


def check_device_split_golden():
    """The GPU library's chunk count and chunks against hand-worked cases."""
    d = load("device_split_plan.json")
    for c in d["cases"]:
        T = orc.device_chunk_count(c["S"], c["KVH"], c["sms"], c["ctas_per_sm"])
        assert T == c["T"], (c["work"], T)
        Ts = T
        if "rows" in c:
            Ts = orc.device_seq_chunks(T, c["S"], c["rows"], c["G"], c["rows_per_block"])
            assert Ts == c["Ts"], (c["work"], Ts)
        want = [(j * c["c"], (j + 1) * c["c"]) for j in range(c["full"])]
        if c["tail"] is not None:
            want.append(tuple(c["tail"]))
        want += [(c["L"], c["L"])] * c["empty"]
        got = orc.device_chunk_ranges(c["L"], Ts)
        got += [(c["L"], c["L"])] * (T - Ts)
        assert got == want, (c["work"], got[:3], got[-3:])


def check_device_split_properties():
    """Chunks tile [0, L) in order; every chunk but the last non-empty one is
    a whole number of 64-token tiles and at least 128 tokens."""
    for L in [1, 63, 64, 127, 128, 129, 1000, 1024, 1032, 4097, 20676, 32784, 100000]:
        for T in [1, 2, 8, 16, 37, 38, 76, 128]:
            rs = orc.device_chunk_ranges(L, T)
            assert len(rs) == T and rs[0][0] == 0 and rs[-1][1] == L
            for (a, b), (c, _) in zip(rs, rs[1:]):
                assert b == c and a <= b
            live = [(a, b) for a, b in rs if b > a]
            for a, b in live[:-1]:
                assert (b - a) % 64 == 0 and b - a >= 128, (L, T, a, b)
            assert live[-1][1] - live[-1][0] <= live[0][1] - live[0][0]


def check_split_rule_properties():
    for L in [1, 2, 15, 16, 17, 255, 1024, 1025, 1032, 4097, 20676, 32784]:
        for S in [1, 2, 3, 5, 8, 13, 64]:
            rs = orc.split_ranges(L, S)
            assert len(rs) == S
            assert rs[0][0] == 0 and rs[-1][1] == L
            for (a, b), (c, _) in zip(rs, rs[1:]):
                assert b == c and a <= b
            for a, _ in rs:
                assert a % 16 == 0 or a == L


def check_gather_golden():
    # block_table [[2, 0]], KVH = 2: token 3 of KV head 0 lives on page 2,
    # slot 3 -> row (2*2+0)*16+3 = 67; token 17 of KV head 1 lives on page 0,
    # slot 1 -> row (0*2+1)*16+1 = 17.  Contiguous capacity 32: token 5 of
    # sequence 1, KV head 1 -> (1*2+1)*32+5 = 101.
    bt = np.array([[2, 0]], dtype=np.int32)
    assert int(orc.gather_index(0, 0, 3, page_size=16, capacity=0, num_kv_heads=2, block_table=bt)) == 67
    assert int(orc.gather_index(0, 1, 17, page_size=16, capacity=0, num_kv_heads=2, block_table=bt)) == 17
    assert int(orc.gather_index(1, 1, 5, page_size=0, capacity=32, num_kv_heads=2)) == 101


def check_paged_equals_contiguous():
    c = sy.make_case("pg", num_heads=4, num_kv_heads=2, head_dim=32, kv_dtype=sy.Q8_0,
                     q_dtype=sy.BF16, ctx=[37, 5, 16], rows=[3, 1, 4], kinds=[1, 0, 1],
                     mode="mixed", paged=True, seed=11, extra_blocks=3)
    c2 = sy.to_contiguous(c)
    O1, L1 = orc.verify_case(c)
    O2, L2 = orc.verify_case(c2)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)
    assert np.isfinite(O1).all()


# ---------------------------------------------------------------------------
# Attention values.

def _golden_args(c, scale):
    H, KVH, D = c["H"], c["KVH"], c["D"]
    K = np.asarray(c["K"], dtype=np.float32)
    V = np.asarray(c["V"], dtype=np.float32)
    if K.ndim == 2:
        K, V = K[None], V[None]
    L = K.shape[1]
    k = K.reshape(1, KVH, L, D)
    v = V.reshape(1, KVH, L, D)
    q = np.asarray(c["Q"], dtype=np.float32).reshape(-1, H, D)
    n = q.shape[0]
    return dict(q=q, k=k, v=v, kv_dtype="f32", q_dtype="f32", num_heads=H,
                num_kv_heads=KVH, head_dim=D, ctx_len=[c["ctx"]], cu_rows=[0, n],
                parent=np.asarray(c["parent"], dtype=np.int32),
                seq_kind=np.array([c["kind"]], dtype=np.uint8),
                mode="tree" if c["kind"] else "chain", capacity=L, scale=scale)


def check_golden_attention(num_splits=None):
    d = load("tiny_attention.json")
    scale = math.log(2.0)
    for c in d["cases"]:
        O, LSE = orc.verify_attention(**_golden_args(c, scale), num_splits=num_splits)
        want_o = np.asarray(c["O"], dtype=np.float64)
        want_l = np.array([[_val(row)] if row[0] == "ln" else [_val(x) for x in row]
                           for row in c["LSE"]])
        assert np.allclose(O, want_o, rtol=0, atol=1e-13), (c["name"], O, want_o)
        assert np.allclose(LSE, want_l, rtol=0, atol=1e-13), (c["name"], LSE, want_l)
    # the Q8 case: one 32-element block per row, scale 0.5
    qc = d["q8_case"]
    sb = int(qc["scale_bits"], 16)

    def rows_of(codes_list):
        out = np.zeros((len(codes_list), 34), dtype=np.uint8)
        for t, codes in enumerate(codes_list):
            out[t, 0], out[t, 1] = sb & 0xFF, sb >> 8
            cc = np.zeros(32, dtype=np.int8)
            cc[:len(codes)] = codes
            out[t, 2:] = cc.view(np.uint8)
        return out

    k = rows_of(qc["K_codes"]).reshape(1, 1, 2, 34)
    v = rows_of(qc["V_codes"]).reshape(1, 1, 2, 34)
    qv = np.zeros(32, dtype=np.float32)
    qv[:len(qc["Q"])] = qc["Q"]
    q = sy.f32_to_bf16_bits(qv).reshape(1, 1, 32)
    O, LSE = orc.verify_attention(q, k, v, kv_dtype="q8_0", q_dtype="bf16", num_heads=1,
                                  num_kv_heads=1, head_dim=32, ctx_len=[qc["ctx"]],
                                  cu_rows=[0, 1], capacity=2, scale=scale,
                                  num_splits=num_splits)
    want = np.zeros(32)
    want[:2] = qc["O_head"]
    assert np.allclose(O[0, 0], want, rtol=0, atol=1e-13), O[0, 0]
    assert abs(LSE[0, 0] - _val(qc["LSE"])) < 1e-13


def _bf_decode(kind, row):
    if kind == "f32":
        return [float(x) for x in row]
    if kind == "bf16":
        return [struct.unpack("<f", struct.pack("<I", int(b) << 16))[0] for b in row]
    out = []
    for b in range(len(row) // 34):
        blk = [int(x) for x in row[34 * b:34 * b + 34]]
        d = struct.unpack("<e", bytes(blk[:2]))[0]
        out += [d * (c - 256 if c > 127 else c) for c in blk[2:]]
    return out


def _bf_visible(t, ctx, j, kind, parent):
    if t < ctx:
        return True
    a = t - ctx
    if kind == 0:
        return a <= j

    def anc_or_self(x, y):
        if x == y:
            return True
        p = int(parent[y])
        return p >= 0 and anc_or_self(x, p)

    return anc_or_self(a, j)


def brute_force(case):
    """Pure-Python verify attention: explicit visibility predicate, plain
    exp without max subtraction, library decodes (struct)."""
    H, KVH, D = case.num_heads, case.num_kv_heads, case.head_dim
    G = H // KVH
    total = case.total_rows
    O = np.zeros((total, H, D))
    LSE = np.zeros((total, H))
    kflat = case.k.reshape(-1, case.k.shape[-1])
    vflat = case.v.reshape(-1, case.v.shape[-1])
    for s in range(case.num_seqs):
        lo, hi = int(case.cu_rows[s]), int(case.cu_rows[s + 1])
        ctx = int(case.ctx_len[s])
        L = ctx + hi - lo
        kind = 0 if case.mode == "chain" else (1 if case.mode == "tree" else int(case.seq_kind[s]))
        par = case.parent[lo:hi]
        for r in range(lo, hi):
            j = r - lo
            for h in range(H):
                kvh = h // G
                qv = _bf_decode(case.q_dtype, case.q[r, h])
                num = [0.0] * D
                den = 0.0
                for t in range(L):
                    if not _bf_visible(t, ctx, j, kind, par):
                        continue
                    if getattr(case, "draft_k", None) is not None and kind == 1 and t >= ctx:
                        # tree scratch KV: row lo + (t - ctx), this KV head
                        kv = _bf_decode(case.kv_dtype, case.draft_k[lo + t - ctx][kvh])
                        vv = _bf_decode(case.kv_dtype, case.draft_v[lo + t - ctx][kvh])
                    else:
                        if case.page_size:
                            blk = int(case.block_table[s][t // 16])
                            idx = (blk * KVH + kvh) * 16 + t % 16
                        else:
                            idx = (s * KVH + kvh) * case.capacity + t
                        kv = _bf_decode(case.kv_dtype, kflat[idx])
                        vv = _bf_decode(case.kv_dtype, vflat[idx])
                    z = case.scale * sum(a * b for a, b in zip(qv, kv))
                    w = math.exp(z)
                    den += w
                    for d in range(D):
                        num[d] += w * vv[d]
                O[r, h] = [x / den for x in num]
                LSE[r, h] = math.log(den)
    return O, LSE


def brute_cases():
    return [
        sy.make_case("bf-f32-chain", num_heads=4, num_kv_heads=2, head_dim=8, kv_dtype=sy.F32,
                     q_dtype=sy.F32, ctx=[0, 5], rows=[3, 4], seed=21),
        sy.make_case("bf-bf16-tree", num_heads=2, num_kv_heads=1, head_dim=8, kv_dtype=sy.BF16,
                     q_dtype=sy.BF16, ctx=[9], rows=[6], mode="tree", seed=22),
        sy.make_case("bf-q8-mixed-paged", num_heads=4, num_kv_heads=2, head_dim=32,
                     kv_dtype=sy.Q8_0, q_dtype=sy.BF16, ctx=[17, 1, 0], rows=[5, 1, 3],
                     kinds=[1, 0, 1], mode="mixed", paged=True, seed=23, extra_blocks=2),
        sy.make_case("bf-q8-chain", num_heads=6, num_kv_heads=3, head_dim=64, kv_dtype=sy.Q8_0,
                     q_dtype=sy.F32, ctx=[20], rows=[2], seed=24),
        # A 40-row chain (a prefill segment: more rows than a 32-bit
        # ancestor mask holds) beside a tree suffix in one mixed launch.
        sy.make_case("bf-f32-prefill-mixed", num_heads=2, num_kv_heads=1, head_dim=8,
                     kv_dtype=sy.F32, q_dtype=sy.F32, ctx=[3, 6], rows=[40, 5], kinds=[0, 1],
                     mode="mixed", seed=25),
        # Tree drafts in a tree scratch KV (their cache rows NaN).
        sy.with_tree_scratch(sy.make_case(
            "bf-q8-mixed-paged-scratch", num_heads=4, num_kv_heads=2, head_dim=32,
            kv_dtype=sy.Q8_0, q_dtype=sy.BF16, ctx=[17, 1, 0, 9], rows=[5, 1, 3, 6],
            kinds=[1, 0, 1, 0], mode="mixed", paged=True, seed=26, extra_blocks=2)),
    ]


def check_brute_force():
    for c in brute_cases():
        O, LSE = orc.verify_case(c)
        Ob, Lb = brute_force(c)
        assert np.allclose(O, Ob, rtol=1e-12, atol=1e-12), c.name
        assert np.allclose(LSE, Lb, rtol=1e-12, atol=1e-12), c.name


def check_weights_sum_to_one():
    c = brute_cases()[2]
    _, _, W = orc.verify_case(c, return_weights=True)
    for (r, h), (pos, w) in W.items():
        assert abs(w.sum() - 1.0) < 1e-12
        assert (w > 0).all()


def check_closed_forms():
    c = sy.make_case("cf", num_heads=4, num_kv_heads=2, head_dim=32, kv_dtype=sy.F32,
                     q_dtype=sy.F32, ctx=[11, 0], rows=[4, 3], kinds=[1, 0], mode="mixed",
                     seed=31)
    # (a) all keys zero -> uniform weights: O = mean of the visible V and
    #     LSE = ln |visible set|.
    c0 = sy.VerifyCase(**{**c.__dict__, "k": np.zeros_like(c.k)})
    O, LSE = orc.verify_case(c0)
    for s in range(c.num_seqs):
        lo, hi = c.cu_rows[s], c.cu_rows[s + 1]
        ctx = int(c.ctx_len[s])
        for r in range(lo, hi):
            j = r - lo
            if c.seq_kind[s] == 0:
                drafts = list(range(j + 1))
            else:
                drafts, p = [j], int(c.parent[lo + j])
                while p >= 0:
                    drafts.append(p)
                    p = int(c.parent[lo + p])
            vis = list(range(ctx)) + [ctx + a for a in drafts]
            for h in range(c.num_heads):
                mean = c.v[s, h // 2, vis].astype(np.float64).mean(axis=0)
                assert np.allclose(O[r, h], mean, rtol=0, atol=1e-12)
                assert abs(LSE[r, h] - math.log(len(vis))) < 1e-12
    # (b) every value row equal to c -> O = c.
    cv = np.broadcast_to(np.linspace(-2, 3, 32, dtype=np.float32), c.v.shape).copy()
    O, _ = orc.verify_case(sy.VerifyCase(**{**c.__dict__, "v": cv}))
    assert np.allclose(O, np.linspace(-2, 3, 32, dtype=np.float32).astype(np.float64),
                       rtol=0, atol=1e-12)
    # (c) ctx = 0, row 0 sees only itself -> O = v_0, LSE = scale q.k_0.
    O, LSE = orc.verify_case(c)
    s, r = 1, int(c.cu_rows[1])
    for h in range(c.num_heads):
        k0 = c.k[s, h // 2, 0].astype(np.float64)
        assert np.array_equal(O[r, h], c.v[s, h // 2, 0].astype(np.float64))
        assert abs(LSE[r, h] - c.scale * float(np.dot(c.q[r, h].astype(np.float64), k0))) < 1e-12


def check_split_invariance():
    for c in [sy.tiny_chain(), brute_cases()[2],
              sy.make_case("sp", num_heads=2, num_kv_heads=1, head_dim=32, kv_dtype=sy.BF16,
                           q_dtype=sy.BF16, ctx=[1030, 3], rows=[8, 2], kinds=[1, 0],
                           mode="mixed", seed=41)]:
        O, LSE = orc.verify_case(c)
        for S in [1, 2, 3, 8, 64]:
            Os, Ls = orc.verify_case(c, num_splits=S)
            assert np.allclose(Os, O, rtol=1e-12, atol=1e-13), (c.name, S)
            assert np.allclose(Ls, LSE, rtol=1e-12, atol=1e-13), (c.name, S)


def check_chain_is_tree_with_chain_parents():
    c = sy.make_case("ct", num_heads=4, num_kv_heads=1, head_dim=32, kv_dtype=sy.Q8_0,
                     q_dtype=sy.BF16, ctx=[40], rows=[7], seed=51)
    O1, L1 = orc.verify_case(c)
    t = sy.VerifyCase(**{**c.__dict__, "mode": "tree",
                         "parent": np.arange(-1, 6, dtype=np.int32)})
    O2, L2 = orc.verify_case(t)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


def check_direct_rows_independent_of_launch():
    c = sy.mixed_tree_direct(ctx=[100, 130, 70, 33, 48, 16, 1, 64], seed=61)
    O, LSE = orc.verify_case(c)
    d = sy.subset_sequences(c, [0, 1])
    Od, Ld = orc.verify_case(d)
    assert np.array_equal(O[:2], Od) and np.array_equal(LSE[:2], Ld)


# ---------------------------------------------------------------------------
# Tree commit of the KV (lucebox PR #686, "State and commit invariants").

def _commit_args(ctx, parent, path, kind=1):
    n = len(parent)
    nodes = np.full(n, -1, dtype=np.int32)
    nodes[:len(path)] = path
    return dict(ctx_len=np.array([ctx]), cu_rows=np.array([0, n]),
                parent=np.asarray(parent, dtype=np.int32), seq_kind=np.array([kind], np.uint8),
                mode="mixed", accepted_len=np.array([len(path)], dtype=np.int32),
                accepted_nodes=nodes)


def check_tree_commit_golden():
    g = load("tree_commit.json")
    c = g["contiguous"]
    scratch = np.asarray(c["scratch"], dtype=np.float32)[:, None, :]
    for case in c["cases"]:
        cap = case["capacity"]
        cache = np.asarray(c["cache"][:cap], dtype=np.float32)[None, None]
        k2, v2, bad = orc.promote(cache, cache, scratch, scratch, page_size=0, capacity=cap,
                                  num_kv_heads=1, **_commit_args(c["ctx"], c["parent"],
                                                                 case["path"]))
        if "reason" in case:
            assert bad == {case["reason"]}, (case["name"], bad)
            assert np.array_equal(k2, cache) and np.array_equal(v2, cache), case["name"]
        else:
            assert not bad, (case["name"], bad)
            assert np.array_equal(k2[0, 0], np.asarray(case["after"], np.float32)), case["name"]
    pg = g["paged"]
    pool = np.zeros((pg["num_blocks"], 1, 16, 2), dtype=np.float32)
    scratch = np.asarray(pg["scratch"], dtype=np.float32)[:, None, :]
    bt = np.asarray([pg["block_table"]], dtype=np.int32)
    k2, _, bad = orc.promote(pool, pool, scratch, scratch, page_size=16, capacity=0,
                             num_kv_heads=1, block_table=bt,
                             **_commit_args(pg["ctx"], pg["parent"], pg["path"]))
    assert not bad
    want = np.zeros_like(pool)
    for blk, slot, row in pg["written"]:
        want[blk, 0, slot] = row
    assert np.array_equal(k2, want)


def check_commit_then_chain():
    """Each accepted tree row (its drafts in the scratch KV) equals, exactly,
    the same query as a chain row over the committed cache: the chain row
    at position ctx + i sees the path's first i + 1 nodes, which are the
    tree row's ancestors and itself, in the same order."""
    base = sy.make_case("commit-chain", num_heads=4, num_kv_heads=2, head_dim=16,
                        kv_dtype=sy.BF16, q_dtype=sy.BF16, ctx=[5, 12, 3], rows=[8, 1, 8],
                        kinds=[1, 0, 1], mode="mixed", paged=True, seed=27)
    c = sy.with_tree_scratch(base)
    acc, nodes = sy.accepted_paths(c, 28)
    O, L = orc.verify_case(c)
    k2, v2, bad = orc.promote(c.k, c.v, c.draft_k, c.draft_v, ctx_len=c.ctx_len,
                              cu_rows=c.cu_rows, parent=c.parent, seq_kind=c.seq_kind,
                              mode=c.mode, accepted_len=acc, accepted_nodes=nodes,
                              page_size=c.page_size, capacity=c.capacity,
                              num_kv_heads=c.num_kv_heads, block_table=c.block_table)
    assert not bad
    ch = sy.accepted_as_chains(c, k2, v2, acc, nodes)
    Oc, Lc = orc.verify_case(ch)
    rows = [int(c.cu_rows[s]) + int(a) for s in range(c.num_seqs)
            for a in nodes[int(c.cu_rows[s]):int(c.cu_rows[s]) + int(acc[s])]]
    assert len(rows) == ch.total_rows > 0
    assert np.array_equal(O[rows], Oc) and np.array_equal(L[rows], Lc)

