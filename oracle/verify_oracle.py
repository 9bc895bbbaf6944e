"""fp64 CPU oracle for speculative-decoding verify attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  The library under
``speculative_decoding_verify_kv_gb300`` never imports it, and this module
imports nothing from the library: the two share no code.

What it computes (plain definition, float64, no blocking or fusion):

For sequence s, local draft row j and query head h of a verify launch:

1. KV head ``kvh = h // G`` with ``G = H / KVH`` (contiguous head groups).
2. The KV span holds ``L = ctx + n`` tokens; the draft rows' own K/V sit at
   positions ``ctx .. ctx+n-1`` of the same cache.
3. Visible set ``V = {0..ctx-1} ∪ {ctx + a : a == j or a is an ancestor of j}``.
   A chain (and a one-row direct / AR row) has ``parent[j] = j-1``; a tree
   suffix follows its parent array to -1.  Sources: lucebox PR #686 "retain
   speculation during paged prefill", section "State and commit invariants"
   (tree rows carry ancestry metadata over a fixed-width suffix; prompt and AR
   rows stay positioned causal reads) and section "Mechanism" (the
   [prefill][direct/AR][tree] lowering).
4. Decode storage exactly to float64: bf16 by bit shift, fp16 by explicit bit
   decode, Q8_0 as ``double(fp16 scale) * double(int8 code)`` per 32-element
   block (hipfire PR #695, alpineQ comments: the ``attention_flash_q8_0_*``
   kernels read a Q8 KV cache; Q8_0's 32-element blocks with one fp16 scale).
5. ``z_t = scale * sum_d q_d k_{t,d}``, ``M = max z``, ``w_t = exp(z_t - M)``,
   ``l = sum w``, ``O = sum_t w_t v_t / l``, ``LSE = M + ln l``.

The split variant follows the FA2 split-KV design of hipfire PR #817
("speed up long-context DFlash verify 13.4% with FA2 split-KV", sections
"Summary" and "Performance": S chunks write online-softmax partials that a
merge pass combines): each chunk yields ``(m_s, l_s, acc_s)`` in float64 and
the merge takes ``M = max m_s``, ``l = sum e^{m_s-M} l_s``,
``O = sum e^{m_s-M} acc_s / l``.  The chunk rule depends only on the
sequence's own span L and the split count S, never on what else shares the
launch (lucebox PR #686, section "Correctness failure found during
qualification": the 1,024-token partition boundary).

Optional tree scratch KV and the tree commit (lucebox PR #686, "State and
commit invariants": tree rows write scratch KV; the commit transaction
promotes only the accepted prefix after checking every domain): with
``draft_k``/``draft_v`` a tree sequence's draft position a reads scratch row
``cu_rows[s] + a``; ``promote`` copies each tree's accepted root path to
positions ``ctx ..`` of the cache, or nothing at all if any check fails.

Parity status: every function below is pinned by ``tests/test_oracle.py``
(brute force, closed forms, library special cases, invariants and hand-worked
fixtures under ``tests/golden/``).
"""
from __future__ import annotations

import math
from typing import Optional

import numpy as np

PAGE = 16
Q8_BLOCK = 32
Q8_BLOCK_BYTES = 34


# ---------------------------------------------------------------------------
# Exact decoding of the storage formats.

def decode_bf16(bits) -> np.ndarray:
    """bf16 bits -> float64: the bf16 pattern is the top half of an fp32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def decode_fp16(bits) -> np.ndarray:
    """IEEE binary16 bits -> float64, decoded field by field."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    sign = np.where((b >> 15) & 1, -1.0, 1.0)
    exp = (b >> 10) & 0x1F
    man = (b & 0x3FF).astype(np.float64)
    normal = sign * (1024.0 + man) * np.exp2(exp.astype(np.float64) - 25.0)
    subnormal = sign * man * 2.0 ** -24
    special = np.where(man == 0, sign * np.inf, np.nan)
    return np.where(exp == 0, subnormal, np.where(exp == 31, special, normal))


def dequant_q8_0(raw) -> np.ndarray:
    """Q8_0 rows ``[..., nb*34]`` (uint8) -> float64 ``[..., nb*32]``.

    Each 34-byte block is a little-endian fp16 scale d followed by 32 int8
    codes q; element i of the block is d * q[i].
    """
    raw = np.asarray(raw, dtype=np.uint8)
    nb = raw.shape[-1] // Q8_BLOCK_BYTES
    blk = raw.reshape(raw.shape[:-1] + (nb, Q8_BLOCK_BYTES))
    sbits = blk[..., 0].astype(np.uint16) | (blk[..., 1].astype(np.uint16) << 8)
    d = decode_fp16(sbits)
    q = blk[..., 2:].copy().view(np.int8).astype(np.float64)
    return (d[..., None] * q).reshape(raw.shape[:-1] + (nb * Q8_BLOCK,))


def decode_rows(rows, kv_dtype: str) -> np.ndarray:
    if kv_dtype == "f32":
        return np.asarray(rows, dtype=np.float32).astype(np.float64)
    if kv_dtype == "bf16":
        return decode_bf16(rows)
    if kv_dtype == "q8_0":
        return dequant_q8_0(rows)
    raise ValueError(kv_dtype)


def decode_q(q, q_dtype: str) -> np.ndarray:
    return decode_rows(q, q_dtype)


# ---------------------------------------------------------------------------
# Row map, masks and KV addressing.

def ancestors(parent_local, j: int) -> list[int]:
    """Ancestors of draft node j: follow parent links until -1."""
    out = []
    p = int(parent_local[j])
    while p >= 0:
        if p >= j or p in out:
            raise ValueError(f"parent array is not topological at node {j}")
        out.append(p)
        p = int(parent_local[p])
    return out


def row_masks(n: int, kind: int, parent_local) -> list[int]:
    """Per local row j: bit a set iff draft position a is visible to row j
    (a == j or a is an ancestor).  kind 0 = chain / direct, 1 = tree."""
    masks = []
    for j in range(n):
        if kind == 0:
            vis = range(j + 1)
        else:
            vis = [j] + ancestors(parent_local, j)
        m = 0
        for a in vis:
            m |= 1 << a
        masks.append(m)
    return masks


def row_map(cu_rows, parent, seq_kind, mode: str):
    """Global row -> (sequence, ancestor mask).  Returns int32 row_seq and
    uint32 masks (rows with n > 32 are not representable and rejected)."""
    cu = np.asarray(cu_rows)
    total = int(cu[-1])
    row_seq = np.empty(total, dtype=np.int32)
    masks = np.empty(total, dtype=np.uint32)
    for s in range(len(cu) - 1):
        lo, hi = int(cu[s]), int(cu[s + 1])
        if hi - lo > 32:
            raise ValueError("at most 32 rows per sequence")
        kind = seq_kind_of(s, seq_kind, mode)
        pl = None if parent is None else np.asarray(parent[lo:hi])
        for j, m in enumerate(row_masks(hi - lo, kind, pl)):
            row_seq[lo + j] = s
            masks[lo + j] = m
    return row_seq, masks


def seq_kind_of(s: int, seq_kind, mode: str) -> int:
    if mode == "chain":
        return 0
    if mode == "tree":
        return 1
    return int(seq_kind[s])


def visible_positions(ctx: int, n: int, kind: int, parent_local, j: int) -> np.ndarray:
    """Sorted KV positions visible to local row j."""
    if kind == 0:
        drafts = list(range(j + 1))
    else:
        drafts = sorted([j] + ancestors(parent_local, j))
    return np.concatenate([np.arange(ctx, dtype=np.int64),
                           np.asarray([ctx + a for a in drafts], dtype=np.int64)])


def gather_index(s: int, kvh: int, t, *, page_size: int, capacity: int,
                 num_kv_heads: int, block_table=None):
    """Physical row of token t of sequence s, KV head kvh, counted in rows of
    the cache array: contiguous ``[seq][KVH][capacity]`` or paged
    ``[block][KVH][16]`` (page ``block_table[s][t // 16]``, slot ``t % 16``)."""
    t = np.asarray(t, dtype=np.int64)
    if page_size == 0:
        return (s * num_kv_heads + kvh) * capacity + t
    blk = np.asarray(block_table)[s, t // PAGE].astype(np.int64)
    return (blk * num_kv_heads + kvh) * PAGE + t % PAGE


def kv_rows(cache, s: int, kvh: int, L: int, *, page_size: int, capacity: int,
            num_kv_heads: int, block_table=None) -> np.ndarray:
    """Storage rows of tokens 0..L-1 for (s, kvh)."""
    flat = np.asarray(cache).reshape(-1, np.asarray(cache).shape[-1])
    idx = gather_index(s, kvh, np.arange(L), page_size=page_size, capacity=capacity,
                       num_kv_heads=num_kv_heads, block_table=block_table)
    return flat[idx]


def kv_head_of(h: int, G: int) -> int:
    """Grouped-query mapping: query heads come in contiguous groups of G per
    KV head (H24/KV4 gives heads 0..5 -> KV head 0, 6..11 -> 1, ...)."""
    return h // G


# ---------------------------------------------------------------------------
# Attention of one row over its visible set.

def attend(q, K, V, scale: float):
    """Softmax attention of one query over keys K [T, D] and values V [T, D]:
    returns (o [D], lse, weights [T])."""
    z = scale * np.einsum("td,d->t", K, q)
    M = z.max()
    w = np.exp(z - M)
    l = w.sum()
    o = np.einsum("t,td->d", w, V) / l
    return o, M + math.log(l), w / l


def split_ranges(L: int, S: int) -> list[tuple[int, int]]:
    """Chunk rule of the split-KV pass: chunk = ceil(L / S) rounded up to a
    multiple of 16 tokens; chunk s covers [s*chunk, min((s+1)*chunk, L)) and
    may be empty.  Depends only on this sequence's L and S."""
    per_split = -(-L // S)                      # ceil(L / S)
    chunk = -(-per_split // PAGE) * PAGE        # rounded up to 16 tokens
    return [(min(s * chunk, L), min((s + 1) * chunk, L)) for s in range(S)]


def device_chunk_count(S: int, num_kv_heads: int, sm_count: int, ctas_per_sm: int) -> int:
    """How many chunks (T) the GPU library cuts each sequence into: one wave
    of CTAs per (sequence, KV head), i.e. ctas_per_sm * sm_count //
    num_kv_heads, kept within [S, 16 S].  ctas_per_sm is 1 for the
    tensor-core kernels and 2 for the CUDA-core kernel.  Not a rule of the
    pages (they fix only that the cut follows the sequence's own span and
    S): the library's reading of "S chunks", restated here so that tests can
    pin the chunks its kernels run."""
    T = ctas_per_sm * sm_count // num_kv_heads
    return max(S, min(T, 16 * S))


def device_seq_chunks(T: int, S: int, rows: int, group: int, rows_per_block: int) -> int:
    """How many of the T chunks the GPU library cuts a sequence with `rows`
    query rows into: T shared out among the sequence's row blocks (ceil(rows
    * group / rows_per_block) of them; each streams the span again), but at
    least S.  A sequence of one row block keeps all T.  rows_per_block is 128
    for the row-major tensor-core kernel and 16 for the CUDA-core kernel.
    Like device_chunk_count, the library's reading, not the pages': it
    depends on the sequence alone."""
    rb = max(1, -(-rows * group // rows_per_block))
    return max(S, T // rb)


def device_chunk_ranges(L: int, T: int) -> list[tuple[int, int]]:
    """The GPU library's chunks of a span of L tokens cut T ways: chunk
    length c = max(ceil(L / T), 128) rounded up to a multiple of 64 tokens
    (whole 64-token tiles, at least two of them), chunk j = [min(j c, L),
    min((j + 1) c, L)); trailing chunks may be empty.  Like split_ranges it
    depends on the sequence's own span only (lucebox PR #686, "Correctness
    failure found during qualification")."""
    c = max(-(-L // T), 128)
    c = -(-c // 64) * 64
    return [(min(j * c, L), min((j + 1) * c, L)) for j in range(T)]


def partial(q, K, V, pos, lo: int, hi: int, scale: float):
    """Online-softmax partial of one chunk: (m, l, acc) over the visible
    positions inside [lo, hi); an empty chunk gives (-inf, 0, 0)."""
    sel = (pos >= lo) & (pos < hi)
    if not sel.any():
        return -math.inf, 0.0, np.zeros(K.shape[1])
    Kc, Vc = K[pos[sel]], V[pos[sel]]
    z = scale * np.einsum("td,d->t", Kc, q)
    m = z.max()
    w = np.exp(z - m)
    return m, w.sum(), np.einsum("t,td->d", w, Vc)


def merge(parts):
    """Combine chunk partials in ascending chunk order."""
    live = [p for p in parts if p[1] > 0]
    M = max(p[0] for p in live)
    l = sum(math.exp(m - M) * ls for m, ls, _ in live)
    acc = sum(math.exp(m - M) * a for m, _, a in live)
    return acc / l, M + math.log(l)


# ---------------------------------------------------------------------------
# The whole verify launch.

def span_rows(cache, draft, s: int, kvh: int, ctx: int, n: int, lo: int, *, page_size: int,
              capacity: int, num_kv_heads: int, block_table=None) -> np.ndarray:
    """Storage rows of the span's L = ctx + n tokens for (s, kvh): all from
    the cache, or (``draft`` given: a tree scratch KV [total_rows][KVH][row])
    the ctx context rows from the cache followed by scratch rows lo .. lo+n-1
    for the draft positions (lucebox PR #686, "State and commit invariants":
    tree rows write scratch KV)."""
    if draft is None:
        return kv_rows(cache, s, kvh, ctx + n, page_size=page_size, capacity=capacity,
                       num_kv_heads=num_kv_heads, block_table=block_table)
    ctx_part = kv_rows(cache, s, kvh, ctx, page_size=page_size, capacity=capacity,
                       num_kv_heads=num_kv_heads, block_table=block_table)
    return np.concatenate([ctx_part, np.asarray(draft)[lo:lo + n, kvh]])


def verify_attention(q, k, v, *, kv_dtype: str, q_dtype: str, num_heads: int,
                     num_kv_heads: int, head_dim: int, ctx_len, cu_rows,
                     parent=None, seq_kind=None, mode: str = "chain",
                     page_size: int = 0, capacity: int = 0, block_table=None,
                     draft_k=None, draft_v=None,
                     scale: float = 0.0, num_splits: Optional[int] = None,
                     rows: Optional[list] = None, heads: Optional[list] = None,
                     return_weights: bool = False):
    """Verify attention for every (row, head) (or the ``rows`` x ``heads``
    subset).  Returns O [total_rows, H, D] and LSE [total_rows, H] in float64
    (entries outside the subset are NaN).  ``num_splits=None`` is the
    unsplit definition; an integer S takes the split-and-merge route.
    ``draft_k``/``draft_v`` (optional tree scratch KV): a tree sequence's
    draft K/V come from scratch rows cu_rows[s] + a instead of the cache."""
    H, KVH, D = num_heads, num_kv_heads, head_dim
    if H % KVH:
        raise ValueError("H must be a multiple of KVH")
    G = H // KVH
    if scale == 0.0:
        scale = 1.0 / math.sqrt(D)
    cu = np.asarray(cu_rows, dtype=np.int64)
    ctx_len = np.asarray(ctx_len, dtype=np.int64)
    total = int(cu[-1])
    O = np.full((total, H, D), np.nan)
    LSE = np.full((total, H), np.nan)
    W = {}
    rowset = set(range(total)) if rows is None else set(int(r) for r in rows)
    headset = list(range(H)) if heads is None else [int(h) for h in heads]
    Q = decode_q(np.asarray(q).reshape(total, H, -1), q_dtype) if total else None
    for s in range(len(ctx_len)):
        lo, hi = int(cu[s]), int(cu[s + 1])
        n = hi - lo
        todo = [r for r in range(lo, hi) if r in rowset]
        if not todo:
            continue
        ctx = int(ctx_len[s])
        L = ctx + n
        kind = seq_kind_of(s, seq_kind, mode)
        pl = None if parent is None else np.asarray(parent)[lo:hi]
        scratch = draft_k is not None and kind == 1
        for kvh in sorted(set(kv_head_of(h, G) for h in headset)):
            K = decode_rows(span_rows(k, draft_k if scratch else None, s, kvh, ctx, n, lo,
                                      page_size=page_size, capacity=capacity,
                                      num_kv_heads=KVH, block_table=block_table), kv_dtype)
            V = decode_rows(span_rows(v, draft_v if scratch else None, s, kvh, ctx, n, lo,
                                      page_size=page_size, capacity=capacity,
                                      num_kv_heads=KVH, block_table=block_table), kv_dtype)
            for r in todo:
                j = r - lo
                pos = visible_positions(ctx, n, kind, pl, j)
                for h in headset:
                    if kv_head_of(h, G) != kvh:
                        continue
                    qv = Q[r, h]
                    if num_splits is None:
                        o, lse, w = attend(qv, K[pos], V[pos], scale)
                        if return_weights:
                            W[(r, h)] = (pos, w)
                    else:
                        parts = [partial(qv, K, V, pos, a, b, scale)
                                 for a, b in split_ranges(L, int(num_splits))]
                        o, lse = merge(parts)
                    O[r, h] = o
                    LSE[r, h] = lse
    if return_weights:
        return O, LSE, W
    return O, LSE


def verify_case(case, **kw):
    """Convenience wrapper taking a case object with the storage fields of
    the synthetic generator (duck-typed; no import of the generator)."""
    return verify_attention(
        case.q, case.k, case.v, kv_dtype=case.kv_dtype, q_dtype=case.q_dtype,
        num_heads=case.num_heads, num_kv_heads=case.num_kv_heads,
        head_dim=case.head_dim, ctx_len=case.ctx_len, cu_rows=case.cu_rows,
        parent=case.parent, seq_kind=case.seq_kind, mode=case.mode,
        page_size=case.page_size, capacity=case.capacity,
        block_table=case.block_table, draft_k=getattr(case, "draft_k", None),
        draft_v=getattr(case, "draft_v", None), scale=case.scale, **kw)


# ---------------------------------------------------------------------------
# Tree commit of the KV (the KV part of lucebox PR #686's tree commit
# transaction, "State and commit invariants": only the accepted prefix is
# promoted, and every domain is checked before any is mutated).

def promote_preflight(*, ctx_len, cu_rows, parent, seq_kind, mode: str, accepted_len,
                      accepted_nodes, page_size: int, capacity: int, num_blocks: int = 0,
                      block_table=None) -> set:
    """The reasons the commit must not happen (empty set: it may).  Per
    sequence: m in [0, n], m > 0 only for a tree; the accepted nodes are a
    root path of the tree (first node's parent -1, each next node's parent
    the previous node); the destinations ctx .. ctx+m-1 fit the capacity
    or the block table, on valid blocks."""
    bad = set()
    cu = np.asarray(cu_rows)
    for s in range(len(cu) - 1):
        lo, hi = int(cu[s]), int(cu[s + 1])
        n, m, ctx = hi - lo, int(accepted_len[s]), int(ctx_len[s])
        if m < 0 or m > n or (m > 0 and seq_kind_of(s, seq_kind, mode) != 1):
            bad.add("rows")
            continue
        path = [int(a) for a in accepted_nodes[lo:lo + m]]
        if any(a < 0 or a >= n for a in path):
            bad.add("rows")
            continue
        expected_parent = [-1] + path[:-1]
        if any(int(parent[lo + a]) != e for a, e in zip(path, expected_parent)):
            bad.add("parent")
            continue
        end = ctx + m
        if page_size == 0:
            if end > capacity:
                bad.add("overflow")
        else:
            pages = -(-end // PAGE)
            bt = np.asarray(block_table)
            if pages > bt.shape[1]:
                bad.add("overflow")
            elif any(not (0 <= int(bt[s, pg]) < num_blocks) for pg in range(ctx // PAGE, pages)):
                bad.add("block")
    return bad


def promote(k, v, draft_k, draft_v, *, ctx_len, cu_rows, parent, seq_kind, mode: str,
            accepted_len, accepted_nodes, page_size: int, capacity: int, num_kv_heads: int,
            block_table=None):
    """Cache arrays after the commit (copies; the inputs are not changed):
    path node i of sequence s (scratch row cu_rows[s] + node) lands at
    position ctx + i, every KV head, K and V.  Returns (k', v', reasons);
    any reason leaves both caches exactly as they were."""
    nb = 0 if page_size == 0 else np.asarray(k).shape[0]
    bad = promote_preflight(ctx_len=ctx_len, cu_rows=cu_rows, parent=parent,
                            seq_kind=seq_kind, mode=mode, accepted_len=accepted_len,
                            accepted_nodes=accepted_nodes, page_size=page_size,
                            capacity=capacity, num_blocks=nb, block_table=block_table)
    k2, v2 = np.array(k, copy=True), np.array(v, copy=True)
    if bad:
        return k2, v2, bad
    kf = k2.reshape(-1, k2.shape[-1])
    vf = v2.reshape(-1, v2.shape[-1])
    cu = np.asarray(cu_rows)
    for s in range(len(cu) - 1):
        lo = int(cu[s])
        ctx = int(ctx_len[s])
        for i in range(int(accepted_len[s])):
            a = int(accepted_nodes[lo + i])
            for kvh in range(num_kv_heads):
                dst = int(gather_index(s, kvh, ctx + i, page_size=page_size, capacity=capacity,
                                       num_kv_heads=num_kv_heads, block_table=block_table))
                kf[dst] = np.asarray(draft_k)[lo + a, kvh]
                vf[dst] = np.asarray(draft_v)[lo + a, kvh]
    return k2, v2, bad
