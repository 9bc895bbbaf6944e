"""Plant plausible mistakes in the oracle (on the CPU) and check that at
least one pin catches each: evidence that the pins constrain every step."""
import math

import numpy as np
import pytest

import oracle.verify_oracle as orc
import oracle_pins as P

ALL_PINS = [
    P.check_fp16_golden, P.check_q8_golden, P.check_tree_masks_golden, P.check_row_map_mixed,
    P.check_split_golden, P.check_gather_golden, P.check_paged_equals_contiguous,
    P.check_golden_attention, P.check_brute_force, P.check_closed_forms,
    P.check_split_invariance, P.check_chain_is_tree_with_chain_parents,
    P.check_tree_commit_golden, P.check_commit_then_chain, P.check_device_split_golden,
]


def _attend_no_scale(q, K, V, scale):
    return _orig["attend"](q, K, V, 1.0)


def _attend_values_are_keys(q, K, V, scale):
    return _orig["attend"](q, K, K, scale)


def _attend_no_max_shift_wrong_lse(q, K, V, scale):
    o, lse, w = _orig["attend"](q, K, V, scale)
    return o, lse - scale * float(np.max(K @ q)), w


def _visible_off_by_one(ctx, n, kind, parent_local, j):
    pos = _orig["visible_positions"](ctx, n, kind, parent_local, j)
    return pos[:-1] if len(pos) > 1 else pos


def _visible_drops_context(ctx, n, kind, parent_local, j):
    pos = _orig["visible_positions"](ctx, n, kind, parent_local, j)
    return pos[1:] if len(pos) > 1 else pos


def _ancestors_parent_only(parent_local, j):
    p = int(parent_local[j])
    return [p] if p >= 0 else []


def _kv_head_modulo(h, G):
    return h % max(1, 4 // G) if G > 1 else h


def _dequant_unsigned(raw):
    raw = np.asarray(raw, dtype=np.uint8)
    nb = raw.shape[-1] // 34
    blk = raw.reshape(raw.shape[:-1] + (nb, 34))
    sbits = blk[..., 0].astype(np.uint16) | (blk[..., 1].astype(np.uint16) << 8)
    d = orc.decode_fp16(sbits)
    q = blk[..., 2:].astype(np.float64)
    return (d[..., None] * q).reshape(raw.shape[:-1] + (nb * 32,))


def _fp16_bias_off(bits):
    return _orig["decode_fp16"](bits) * 2.0


def _split_no_rounding(L, S):
    chunk = -(-L // S)
    return [(min(s * chunk, L), min((s + 1) * chunk, L)) for s in range(S)]


def _device_chunks_tile16(L, T):
    c = max(-(-L // T), 128)
    c = -(-c // 16) * 16
    return [(min(j * c, L), min((j + 1) * c, L)) for j in range(T)]


def _device_chunks_no_minimum(L, T):
    c = -(-(-(-L // T)) // 64) * 64
    return [(min(j * c, L), min((j + 1) * c, L)) for j in range(T)]


def _device_count_unclamped(S, num_kv_heads, sm_count, ctas_per_sm):
    return ctas_per_sm * sm_count // num_kv_heads


def _seq_chunks_ignore_rows(T, S, rows, group, rows_per_block):
    return T


def _seq_chunks_no_floor(T, S, rows, group, rows_per_block):
    return T // max(1, -(-rows * group // rows_per_block))


def _merge_no_rescale(parts):
    live = [p for p in parts if p[1] > 0]
    M = max(p[0] for p in live)
    l = sum(ls for _, ls, _ in live)
    acc = sum(a for _, _, a in live)
    return acc / l, M + math.log(l)


def _gather_slot_swapped(s, kvh, t, *, page_size, capacity, num_kv_heads, block_table=None):
    t = np.asarray(t, dtype=np.int64)
    if page_size == 0:
        return (s * num_kv_heads + kvh) * capacity + t
    blk = np.asarray(block_table)[s, t // 16].astype(np.int64)
    return (blk * num_kv_heads + kvh) * 16 + (15 - t % 16)


def _promote_one_late(k, v, draft_k, draft_v, **kw):
    kw["ctx_len"] = np.asarray(kw["ctx_len"]) + 1
    return _orig["promote"](k, v, draft_k, draft_v, **kw)


def _preflight_ignores_parents(**kw):
    kw["parent"] = _fake_root_paths(kw["parent"], kw["accepted_nodes"], kw["cu_rows"],
                                    kw["accepted_len"])
    return _orig["promote_preflight"](**kw)


def _fake_root_paths(parent, nodes, cu_rows, acc_len):
    """A parent array under which every accepted path is a root path."""
    par = np.array(parent, copy=True)
    for s in range(len(cu_rows) - 1):
        lo = int(cu_rows[s])
        prev = -1
        for i in range(int(acc_len[s])):
            a = int(nodes[lo + i])
            if 0 <= a < int(cu_rows[s + 1]) - lo:
                par[lo + a] = prev
            prev = a
    return par


def _span_rows_scratch_shifted(cache, draft, s, kvh, ctx, n, lo, **kw):
    if draft is None:
        return _orig["span_rows"](cache, None, s, kvh, ctx, n, lo, **kw)
    shifted = np.roll(np.asarray(draft), -1, axis=0)
    return _orig["span_rows"](cache, shifted, s, kvh, ctx, n, lo, **kw)


_orig = {name: getattr(orc, name) for name in
         ["attend", "visible_positions", "ancestors", "kv_head_of", "dequant_q8_0",
          "decode_fp16", "split_ranges", "merge", "gather_index", "promote",
          "promote_preflight", "span_rows", "device_chunk_ranges", "device_chunk_count",
          "device_seq_chunks"]}

MUTATIONS = {
    "scale dropped": ("attend", _attend_no_scale),
    "V replaced by K": ("attend", _attend_values_are_keys),
    "LSE loses its max": ("attend", _attend_no_max_shift_wrong_lse),
    "last visible token dropped": ("visible_positions", _visible_off_by_one),
    "first context token dropped": ("visible_positions", _visible_drops_context),
    "ancestors = parent only": ("ancestors", _ancestors_parent_only),
    "GQA by modulo": ("kv_head_of", _kv_head_modulo),
    "Q8 codes unsigned": ("dequant_q8_0", _dequant_unsigned),
    "fp16 exponent bias": ("decode_fp16", _fp16_bias_off),
    "split chunk not page-rounded": ("split_ranges", _split_no_rounding),
    "merge without rescale": ("merge", _merge_no_rescale),
    "page slot reversed": ("gather_index", _gather_slot_swapped),
    "commit lands one position late": ("promote", _promote_one_late),
    "commit preflight ignores the tree": ("promote_preflight", _preflight_ignores_parents),
    "scratch rows off by one": ("span_rows", _span_rows_scratch_shifted),
    "device chunks in 16-token steps": ("device_chunk_ranges", _device_chunks_tile16),
    "device chunks without the 128-token minimum": ("device_chunk_ranges", _device_chunks_no_minimum),
    "device chunk count not clamped to [S, 16 S]": ("device_chunk_count", _device_count_unclamped),
    "sequence chunk count ignores its row blocks": ("device_seq_chunks", _seq_chunks_ignore_rows),
    "sequence chunk count not floored at S": ("device_seq_chunks", _seq_chunks_no_floor),
}


@pytest.mark.parametrize("label", sorted(MUTATIONS))
def test_planted_mistake_is_caught(label, monkeypatch):
    name, fn = MUTATIONS[label]
    monkeypatch.setattr(orc, name, fn)
    caught = []
    for pin in ALL_PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake: {label}"
