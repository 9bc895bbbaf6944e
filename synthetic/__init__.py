"""Seeded synthetic inputs for speculative-decoding verify attention.

This module is shared by the tests, ``bench.py`` and ``__graft_entry__.smoke``.
It feeds both the fp64 oracle and the CUDA path, so it deliberately holds none
of the method's arithmetic: only random draws, storage-format packing
(round-to-nearest-even to bf16 / fp16, Q8_0 block packing) and the cache
layout (contiguous or 16-token pages with a shuffled block table).

Storage formats (what both sides consume, bit for bit):

* ``q``: ``[total_rows][H][D]``; float32, or uint16 holding bf16 bits.
* contiguous cache: ``[num_seqs][KVH][capacity][row]``; paged pool:
  ``[num_blocks][KVH][16][row]`` with ``block_table[num_seqs][max_blocks]``.
  A row is D float32, D uint16 (bf16 bits) or, for Q8_0, D/32 blocks of
  34 bytes: a little-endian fp16 scale followed by 32 int8 codes.
* the K/V of the draft rows sit at positions ctx..ctx+n-1 of the same cache.
* cache slots past a sequence's end are filled with NaN bit patterns by
  default, so that a kernel that reads past the live span shows it.

Workload recipes follow the five verify shapes of the speculative-decoding
pages (tiny chain, H24/KV4/D256 bf16 chain, long-context Q8, paged D128
batch, mixed tree + direct over paged Q8).
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np

F32, BF16, Q8_0 = "f32", "bf16", "q8_0"
PAGE = 16
Q8_BLOCK = 32
Q8_BLOCK_BYTES = 34

BF16_NAN = 0x7FC0
F16_NAN = 0x7E00


def rng_for(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def f32_to_bf16_bits(x) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even)."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    nan = np.isnan(a)
    if nan.any():
        r[nan] = BF16_NAN
    return r


def f64_to_f16_bits(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


def pack_q8_0(codes: np.ndarray, scale_bits: np.ndarray) -> np.ndarray:
    """Pack int8 codes ``[..., D]`` and fp16 scale bits ``[..., D/32]`` into
    Q8_0 rows ``[..., D/32*34]`` (uint8)."""
    codes = np.asarray(codes, dtype=np.int8)
    d = codes.shape[-1]
    nb = d // Q8_BLOCK
    lead = codes.shape[:-1]
    out = np.empty(lead + (nb, Q8_BLOCK_BYTES), dtype=np.uint8)
    sb = np.asarray(scale_bits, dtype=np.uint16).reshape(lead + (nb,))
    out[..., 0] = (sb & 0xFF).astype(np.uint8)
    out[..., 1] = (sb >> 8).astype(np.uint8)
    out[..., 2:] = codes.reshape(lead + (nb, Q8_BLOCK)).view(np.uint8)
    return out.reshape(lead + (nb * Q8_BLOCK_BYTES,))


def row_elems(kv_dtype: str, head_dim: int) -> int:
    """Storage elements per (token, KV head) row."""
    if kv_dtype == Q8_0:
        return head_dim // Q8_BLOCK * Q8_BLOCK_BYTES
    return head_dim


def row_bytes(kv_dtype: str, head_dim: int) -> int:
    return {F32: 4 * head_dim, BF16: 2 * head_dim,
            Q8_0: head_dim // Q8_BLOCK * Q8_BLOCK_BYTES}[kv_dtype]


def storage_dtype(kind: str):
    return {F32: np.float32, BF16: np.uint16, Q8_0: np.uint8}[kind]


@dataclass
class VerifyCase:
    """One verify-attention problem in storage form."""

    name: str
    num_heads: int
    num_kv_heads: int
    head_dim: int
    kv_dtype: str
    q_dtype: str
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    ctx_len: np.ndarray
    cu_rows: np.ndarray
    parent: np.ndarray
    seq_kind: np.ndarray
    mode: str = "chain"
    page_size: int = 0
    capacity: int = 0
    block_table: Optional[np.ndarray] = None
    # Optional tree scratch KV: [total_rows][KVH][row] storage rows.
    draft_k: Optional[np.ndarray] = None
    draft_v: Optional[np.ndarray] = None
    scale: float = 0.0
    num_splits: int = 1
    seed: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.ctx_len.shape[0])

    @property
    def total_rows(self) -> int:
        return int(self.cu_rows[-1])

    @property
    def rows_per_seq(self) -> np.ndarray:
        return np.diff(self.cu_rows)

    @property
    def max_rows_per_seq(self) -> int:
        r = self.rows_per_seq
        return int(r.max()) if r.size else 0

    @property
    def kv_len(self) -> np.ndarray:
        return self.ctx_len.astype(np.int64) + self.rows_per_seq

    @property
    def kv_bytes(self) -> int:
        """Algorithmic KV bytes one call reads: every live (token, KV head)
        row of K and of V once."""
        return int(self.kv_len.sum()) * self.num_kv_heads * 2 * row_bytes(
            self.kv_dtype, self.head_dim)

    @property
    def flops(self) -> int:
        """4*D flops per visible (row, head, token): Q.K and P.V."""
        tot = 0
        for s in range(self.num_seqs):
            n = int(self.rows_per_seq[s])
            ctx = int(self.ctx_len[s])
            for j in range(n):
                if self.seq_kind[s] == 1:
                    vis = 1
                    p = int(self.parent[self.cu_rows[s] + j])
                    while p >= 0:
                        vis += 1
                        p = int(self.parent[self.cu_rows[s] + p])
                else:
                    vis = j + 1
                tot += (ctx + vis) * self.num_heads * 4 * self.head_dim
        return tot

    def with_splits(self, s: int) -> "VerifyCase":
        return replace(self, num_splits=s)


def _values(rng, kind, shape, sigma=1.0):
    """Random K/V/Q storage for float dtypes: N(0, sigma^2)."""
    x = rng.standard_normal(size=shape, dtype=np.float32) * np.float32(sigma)
    if kind == F32:
        return x
    return f32_to_bf16_bits(x)


def _q8_values(rng, shape, scale_lo=0.002, scale_hi=0.02):
    """Q8_0 rows: codes uniform in [-127, 127], fp16 scales ~ U(lo, hi)."""
    *lead, d = shape
    codes = rng.integers(-127, 128, size=tuple(lead) + (d,), dtype=np.int8)
    sc = rng.uniform(scale_lo, scale_hi, size=tuple(lead) + (d // Q8_BLOCK,))
    return pack_q8_0(codes, f64_to_f16_bits(sc))


def _poison_row(kind, relems):
    if kind == F32:
        return np.full(relems, np.nan, dtype=np.float32)
    if kind == BF16:
        return np.full(relems, BF16_NAN, dtype=np.uint16)
    row = np.zeros(relems, dtype=np.uint8)
    nb = relems // Q8_BLOCK_BYTES
    for b in range(nb):
        row[b * Q8_BLOCK_BYTES] = F16_NAN & 0xFF
        row[b * Q8_BLOCK_BYTES + 1] = F16_NAN >> 8
    return row


def random_tree_parents(rng, n: int) -> np.ndarray:
    """A seeded random tree over n draft nodes in topological order:
    parent[0] = -1 and parent[j] ~ U{0..j-1}."""
    p = np.empty(n, dtype=np.int32)
    if n:
        p[0] = -1
    for j in range(1, n):
        p[j] = int(rng.integers(0, j))
    return p


def make_case(name: str, *, num_heads: int, num_kv_heads: int, head_dim: int,
              kv_dtype: str, q_dtype: str, ctx: list[int], rows: list[int],
              kinds: Optional[list[int]] = None, parents: Optional[list] = None,
              mode: str = "chain", paged: bool = False, seed: int = 0,
              num_splits: int = 1, scale: float = 0.0, q_sigma: float = 1.0,
              kv_sigma: float = 1.0, capacity: Optional[int] = None,
              tail_fill: str = "nan", extra_blocks: int = 0,
              q8_scale_range=(0.002, 0.02)) -> VerifyCase:
    """Build a case. ``ctx[s]`` prior tokens and ``rows[s]`` draft rows per
    sequence; ``kinds[s]`` is 0 (chain / direct) or 1 (tree)."""
    rng = rng_for(seed)
    ns = len(ctx)
    assert len(rows) == ns
    if kinds is None:
        kinds = [1 if mode == "tree" else 0] * ns
    ctx_a = np.asarray(ctx, dtype=np.int32)
    rows_a = np.asarray(rows, dtype=np.int32)
    cu = np.zeros(ns + 1, dtype=np.int32)
    cu[1:] = np.cumsum(rows_a)
    total = int(cu[-1])
    parent = np.empty(total, dtype=np.int32)
    for s in range(ns):
        n = int(rows_a[s])
        if kinds[s] == 1:
            if parents is not None and parents[s] is not None:
                ps = np.asarray(parents[s], dtype=np.int32)
            else:
                ps = random_tree_parents(rng, n)
        else:
            ps = np.arange(-1, n - 1, dtype=np.int32)
        parent[cu[s]:cu[s + 1]] = ps
    seq_kind = np.asarray(kinds, dtype=np.uint8)

    d = head_dim
    if q_dtype == F32:
        q = _values(rng, F32, (total, num_heads, d), q_sigma)
    else:
        q = _values(rng, BF16, (total, num_heads, d), q_sigma)

    relems = row_elems(kv_dtype, d)
    L = ctx_a.astype(np.int64) + rows_a
    sdt = storage_dtype(kv_dtype)

    def gen_rows(count):
        if kv_dtype == Q8_0:
            return _q8_values(rng, (count, d), *q8_scale_range)
        return _values(rng, kv_dtype, (count, d), kv_sigma)

    poison = _poison_row(kv_dtype, relems) if tail_fill == "nan" else np.zeros(relems, dtype=sdt)
    block_table = None
    if not paged:
        cap = int(capacity) if capacity is not None else int(-(-int(L.max()) // PAGE) * PAGE)
        k = np.empty((ns, num_kv_heads, cap, relems), dtype=sdt)
        v = np.empty_like(k)
        for s in range(ns):
            for h in range(num_kv_heads):
                ls = int(L[s])
                k[s, h, :ls] = gen_rows(ls)
                v[s, h, :ls] = gen_rows(ls)
                k[s, h, ls:] = poison
                v[s, h, ls:] = poison
        page_size = 0
    else:
        cap = 0
        nblk = [int(-(-int(l) // PAGE)) for l in L]
        total_blocks = sum(nblk) + extra_blocks
        perm = rng.permutation(total_blocks).astype(np.int32)
        max_blocks = max(nblk) if nblk else 1
        block_table = np.full((ns, max_blocks), -1, dtype=np.int32)
        k = np.empty((total_blocks, num_kv_heads, PAGE, relems), dtype=sdt)
        v = np.empty_like(k)
        k[:] = poison
        v[:] = poison
        pos = 0
        for s in range(ns):
            ls = int(L[s])
            for h in range(num_kv_heads):
                kr = gen_rows(ls)
                vr = gen_rows(ls)
                for b in range(nblk[s]):
                    pid = int(perm[pos + b])
                    lo, hi = b * PAGE, min(ls, (b + 1) * PAGE)
                    k[pid, h, :hi - lo] = kr[lo:hi]
                    v[pid, h, :hi - lo] = vr[lo:hi]
            for b in range(nblk[s]):
                block_table[s, b] = perm[pos + b]
            pos += nblk[s]
        page_size = PAGE
    if scale == 0.0:
        scale = 1.0 / float(np.sqrt(d))
    return VerifyCase(name=name, num_heads=num_heads, num_kv_heads=num_kv_heads,
                      head_dim=d, kv_dtype=kv_dtype, q_dtype=q_dtype, q=q, k=k, v=v,
                      ctx_len=ctx_a, cu_rows=cu, parent=parent, seq_kind=seq_kind,
                      mode=mode, page_size=page_size, capacity=cap,
                      block_table=block_table, scale=scale, num_splits=num_splits,
                      seed=seed)


def to_contiguous(case: VerifyCase) -> VerifyCase:
    """The same values laid out contiguously (capacity = max span rounded
    up to 16); used to check paged == contiguous."""
    assert case.page_size == PAGE
    L = case.kv_len
    cap = int(-(-int(L.max()) // PAGE) * PAGE)
    relems = case.k.shape[-1]
    ns, kvh = case.num_seqs, case.num_kv_heads
    k = np.zeros((ns, kvh, cap, relems), dtype=case.k.dtype)
    v = np.zeros_like(k)
    for s in range(ns):
        for b in range(int(-(-int(L[s]) // PAGE))):
            pid = int(case.block_table[s, b])
            k[s, :, b * PAGE:(b + 1) * PAGE] = case.k[pid]
            v[s, :, b * PAGE:(b + 1) * PAGE] = case.v[pid]
    return replace(case, k=k, v=v, page_size=0, capacity=cap, block_table=None)


# ---------------------------------------------------------------------------
# The five verify workloads (seed = 1000 + workload number).

def tiny_chain(num_splits: int = 1, seed: int = 1001) -> VerifyCase:
    """1 sequence, H4/KV1/D64, ctx 256 + 4 chain rows, fp32 N(0,1), scale 1/8."""
    return make_case("tiny-chain-f32", num_heads=4, num_kv_heads=1, head_dim=64,
                     kv_dtype=F32, q_dtype=F32, ctx=[256], rows=[4], seed=seed,
                     num_splits=num_splits, scale=1.0 / 8.0)


def dflash_bf16(ctx: int = 4096, num_splits: int = 1, seed: int = 1002) -> VerifyCase:
    """H24/KV4/D256, 16 chain rows, bf16 Q/K/V = 0.5 N(0,1), contiguous."""
    return make_case(f"dflash-bf16-ctx{ctx}", num_heads=24, num_kv_heads=4,
                     head_dim=256, kv_dtype=BF16, q_dtype=BF16, ctx=[ctx], rows=[16],
                     seed=seed, num_splits=num_splits, q_sigma=0.5, kv_sigma=0.5)


def long_q8(ctx: int = 32768, num_splits: int = 8, seed: int = 1003) -> VerifyCase:
    """H24/KV4/D256, 16 chain rows, Q bf16 N(0,1), Q8_0 cache, contiguous."""
    return make_case(f"long-q8-ctx{ctx}", num_heads=24, num_kv_heads=4, head_dim=256,
                     kv_dtype=Q8_0, q_dtype=BF16, ctx=[ctx], rows=[16], seed=seed,
                     num_splits=num_splits)


def paged_d128(num_splits: int = 8, seed: int = 1004, ctx=None,
               kv_dtype: str = BF16) -> VerifyCase:
    """4 sequences, ctx ~ U{28000..30000}, H32/KV8/D128, 16 chain rows each,
    bf16 N(0,1) (or Q8_0 with kv_dtype), 16-token pages under a shuffled
    block table."""
    if ctx is None:
        r = rng_for(seed + 7)
        ctx = [int(c) for c in r.integers(28000, 30001, size=4)]
    return make_case("paged-d128-" + kv_dtype, num_heads=32, num_kv_heads=8, head_dim=128,
                     kv_dtype=kv_dtype, q_dtype=BF16, ctx=list(ctx), rows=[16] * len(ctx),
                     paged=True, seed=seed, num_splits=num_splits)


MIXED_CTX = [1016, 1024, 1025, 4097, 8192, 16383, 20676, 32768]


def mixed_tree_direct(num_splits: int = 8, seed: int = 1005, ctx=None,
                      direct=(0, 1), width: int = 8) -> VerifyCase:
    """8 sequences over paged Q8_0: the ``direct`` ones contribute one direct
    row, the rest a width-8 seeded random tree suffix. H24/KV4/D256."""
    if ctx is None:
        ctx = MIXED_CTX
    kinds = [0 if s in direct else 1 for s in range(len(ctx))]
    rows = [1 if s in direct else width for s in range(len(ctx))]
    return make_case("mixed-tree-direct-q8", num_heads=24, num_kv_heads=4,
                     head_dim=256, kv_dtype=Q8_0, q_dtype=BF16, ctx=list(ctx),
                     rows=rows, kinds=kinds, mode="mixed", paged=True, seed=seed,
                     num_splits=num_splits)


def mixed_prefill(num_splits: int = 8, seed: int = 1006, ctx=(8192, 16383, 20676, 4097, 32768),
                  rows=(256, 1, 1, 8, 8), kinds=(0, 0, 0, 1, 1)) -> VerifyCase:
    """A mixed launch with a prefill segment: sequence 0 is a 256-row chain
    (causal among its own rows, more rows than a tree's 32-bit ancestor
    mask holds), two sequences contribute one direct row and two a width-8
    seeded random tree suffix.  H24/KV4/D256 over paged Q8_0."""
    return make_case("mixed-prefill-q8", num_heads=24, num_kv_heads=4, head_dim=256,
                     kv_dtype=Q8_0, q_dtype=BF16, ctx=list(ctx), rows=list(rows),
                     kinds=list(kinds), mode="mixed", paged=True, seed=seed,
                     num_splits=num_splits)


def _cache_index(case: VerifyCase, s: int, kvh: int, t: int):
    """Index tuple of token t of (s, kvh) in the case's cache array."""
    if case.page_size == 0:
        return (s, kvh, t)
    return (int(case.block_table[s, t // PAGE]), kvh, t % PAGE)


def with_tree_scratch(case: VerifyCase) -> VerifyCase:
    """The same launch with the tree sequences' draft K/V moved into a tree
    scratch KV [total_rows][KVH][row] (row r of the launch), their old cache
    rows overwritten with NaN patterns, and the scratch rows of the other
    sequences NaN too: a correct reader sees the same values as before and
    never touches a NaN."""
    relems = case.k.shape[-1]
    poison = _poison_row(case.kv_dtype, relems)
    k, v = case.k.copy(), case.v.copy()
    dk = np.empty((case.total_rows, case.num_kv_heads, relems), dtype=case.k.dtype)
    dv = np.empty_like(dk)
    dk[:] = poison
    dv[:] = poison
    for s in range(case.num_seqs):
        if case.seq_kind[s] != 1 and case.mode != "tree":
            continue
        lo, hi = int(case.cu_rows[s]), int(case.cu_rows[s + 1])
        ctx = int(case.ctx_len[s])
        for a in range(hi - lo):
            for kvh in range(case.num_kv_heads):
                idx = _cache_index(case, s, kvh, ctx + a)
                dk[lo + a, kvh] = k[idx]
                dv[lo + a, kvh] = v[idx]
                k[idx] = poison
                v[idx] = poison
    return replace(case, k=k, v=v, draft_k=dk, draft_v=dv, name=case.name + "-scratch")


def accepted_paths(case: VerifyCase, seed: int):
    """Seeded accepted prefixes: for each tree sequence a root path ending
    at a random node (or empty), none for chain sequences.  Returns int32
    accepted_len [num_seqs] and accepted_nodes [total_rows] (root first,
    -1 past each path)."""
    rng = rng_for(seed)
    acc_len = np.zeros(case.num_seqs, dtype=np.int32)
    nodes = np.full(case.total_rows, -1, dtype=np.int32)
    for s in range(case.num_seqs):
        lo, hi = int(case.cu_rows[s]), int(case.cu_rows[s + 1])
        tree = case.seq_kind[s] == 1 or case.mode == "tree"
        if not tree or hi == lo:
            continue
        end = int(rng.integers(-1, hi - lo))  # -1: nothing accepted
        path = []
        while end >= 0:
            path.append(end)
            end = int(case.parent[lo + end])
        path.reverse()
        acc_len[s] = len(path)
        nodes[lo:lo + len(path)] = path
    return acc_len, nodes


def accepted_as_chains(case: VerifyCase, k, v, acc_len, nodes) -> VerifyCase:
    """A chain launch over a committed cache (k, v): one sequence per tree
    sequence with an accepted path, its rows the path's query rows at
    positions ctx .. ctx+m-1 (where the commit put their K/V)."""
    seqs = [s for s in range(case.num_seqs) if acc_len[s] > 0]
    qrows, ctx, rows = [], [], []
    for s in seqs:
        lo = int(case.cu_rows[s])
        m = int(acc_len[s])
        qrows += [lo + int(a) for a in nodes[lo:lo + m]]
        ctx.append(int(case.ctx_len[s]))
        rows.append(m)
    cu = np.zeros(len(seqs) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(rows)
    parent = np.concatenate([np.arange(-1, m - 1, dtype=np.int32) for m in rows])
    if case.page_size:
        bt = case.block_table[seqs]
        kk, vv = k, v
    else:
        bt = None
        kk, vv = k[seqs], v[seqs]
    return replace(case, q=case.q[qrows], k=kk, v=vv, ctx_len=np.asarray(ctx, dtype=np.int32),
                   cu_rows=cu, parent=parent, seq_kind=np.zeros(len(seqs), dtype=np.uint8),
                   mode="chain", block_table=bt, draft_k=None, draft_v=None,
                   name=case.name + "-accepted")


def subset_sequences(case: VerifyCase, seqs) -> VerifyCase:
    """A launch holding only the given sequences (same cache/pool, same
    values): used for the launch-composition invariance check."""
    seqs = list(seqs)
    rows = case.rows_per_seq
    cu = np.zeros(len(seqs) + 1, dtype=np.int32)
    cu[1:] = np.cumsum([rows[s] for s in seqs])
    q = np.concatenate([case.q[case.cu_rows[s]:case.cu_rows[s + 1]] for s in seqs])
    parent = np.concatenate([case.parent[case.cu_rows[s]:case.cu_rows[s + 1]] for s in seqs])
    if case.page_size:
        bt = case.block_table[seqs]
        k, v = case.k, case.v
    else:
        bt = None
        k, v = case.k[seqs], case.v[seqs]
    return replace(case, q=q, k=k, v=v, ctx_len=case.ctx_len[seqs].copy(), cu_rows=cu,
                   parent=parent, seq_kind=case.seq_kind[seqs].copy(), block_table=bt,
                   name=case.name + f"-subset{seqs}")
