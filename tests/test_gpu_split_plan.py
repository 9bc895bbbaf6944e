"""The chunks the GPU kernels run, read back through va_debug_split_ranges
(the same device functions the partial kernels call) and compared bit for
bit with the oracle's restatement of the library's chunk rule, which the CPU
tests pin to hand-worked cases (tests/golden/device_split_plan.json): T
chunks per sequence, of which a sequence spanning several row blocks uses
fewer, longer ones."""
import numpy as np
import pytest

import oracle.verify_oracle as orc
import oracle_pins as P
import speculative_decoding_verify_kv_gb300 as va
import synthetic as sy

# Spans L = ctx + 16 rows: the hand-worked lengths plus a short one.
SPANS = [1024, 1032, 32784, 100, 8208, 16]
KVH = 4
ROWS = {va.KERNEL_TENSOR: 128, va.KERNEL_CUDA_CORES: 16}  # query rows per CTA


def _case(dtype, S):
    return sy.make_case("split-plan", num_heads=8, num_kv_heads=KVH, head_dim=64, kv_dtype=dtype,
                        q_dtype=sy.BF16, ctx=[L - 16 for L in SPANS], rows=[16] * len(SPANS),
                        seed=41, num_splits=S)


def _sm_count():
    import torch
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.gpu
@pytest.mark.parametrize("S", [1, 8])
@pytest.mark.parametrize("dtype,flags,ctas,kernel", [
    (sy.Q8_0, 0, 1, va.KERNEL_TENSOR),
    (sy.BF16, 0, 1, va.KERNEL_TENSOR),
    (sy.Q8_0, va.FLAG_CUDA_CORES, 2, va.KERNEL_CUDA_CORES),
])
def test_device_chunks_match_the_restated_rule(dtype, flags, ctas, kernel, S):
    case = _case(dtype, S)
    p, kv, mode = va.upload(case, "cuda", num_splits=S, flags=flags)
    pl = va.plan(p, kv, mode)
    assert pl["kernel"] == kernel
    T = orc.device_chunk_count(S, KVH, _sm_count(), ctas)
    assert pl["slots"] == T
    got = va.debug_split_ranges(p, kv, mode).cpu().numpy()
    assert got.shape == (len(SPANS), T, 2)
    Ts = orc.device_seq_chunks(T, S, 16, 2, ROWS[kernel])
    for s, L in enumerate(SPANS):
        want = np.array(orc.device_chunk_ranges(L, Ts) + [(L, L)] * (T - Ts), dtype=np.int32)
        assert np.array_equal(got[s], want), (L, got[s][:4].tolist(), want[:4].tolist())


@pytest.mark.gpu
def test_device_chunks_match_the_hand_worked_cases():
    """The golden cases worked for this GPU's SM count, straight against the
    export (no oracle in between)."""
    sms = _sm_count()
    d = P.load("device_split_plan.json")
    cases = [c for c in d["cases"] if c["sms"] == sms and c["ctas_per_sm"] == 1 and c["KVH"] == KVH
             and c["L"] in SPANS and "rows" not in c]
    if not cases:
        pytest.skip(f"no hand-worked case for {sms} SMs")
    for c in cases:
        case = _case(sy.Q8_0, c["S"])
        p, kv, mode = va.upload(case, "cuda", num_splits=c["S"])
        got = va.debug_split_ranges(p, kv, mode).cpu().numpy()[SPANS.index(c["L"])]
        want = [(j * c["c"], (j + 1) * c["c"]) for j in range(c["full"])]
        if c["tail"] is not None:
            want.append(tuple(c["tail"]))
        want += [(c["L"], c["L"])] * c["empty"]
        assert got.tolist() == [list(r) for r in want], c["work"]


@pytest.mark.gpu
def test_chunks_do_not_depend_on_the_other_sequences():
    """A sequence's chunks are the same alone and in a launch with others."""
    case = _case(sy.Q8_0, 8)
    p, kv, mode = va.upload(case, "cuda", num_splits=8)
    full = va.debug_split_ranges(p, kv, mode).cpu().numpy()
    for s in (0, 2):
        one = sy.subset_sequences(case, [s])
        p1, kv1, mode1 = va.upload(one, "cuda", num_splits=8)
        alone = va.debug_split_ranges(p1, kv1, mode1).cpu().numpy()
        assert np.array_equal(alone[0], full[s])


@pytest.mark.gpu
def test_many_row_sequences_take_fewer_chunks():
    """Sequences of several row blocks (prefill-sized chains) beside a
    one-row sequence in one launch: each sequence's chunks follow its own row
    count (hand-worked cases where the SM count matches, the restated rule
    always), and the one-row sequence keeps all T."""
    sms = _sm_count()
    rows, ctx = [256, 64, 1], [8192, 8384, 8447]   # spans of 8448 tokens
    case = sy.make_case("split-rows", num_heads=24, num_kv_heads=KVH, head_dim=64, kv_dtype=sy.Q8_0,
                        q_dtype=sy.BF16, ctx=ctx, rows=rows, seed=43, num_splits=8)
    p, kv, mode = va.upload(case, "cuda", num_splits=8)
    pl = va.plan(p, kv, mode)
    assert pl["kernel"] == va.KERNEL_TENSOR
    T = orc.device_chunk_count(8, KVH, sms, 1)
    got = va.debug_split_ranges(p, kv, mode).cpu().numpy()
    assert got.shape == (3, T, 2)
    for s in range(3):
        L = ctx[s] + rows[s]
        Ts = orc.device_seq_chunks(T, 8, rows[s], 6, ROWS[va.KERNEL_TENSOR])
        want = orc.device_chunk_ranges(L, Ts) + [(L, L)] * (T - Ts)
        assert got[s].tolist() == [list(r) for r in want], (s, Ts)
    assert orc.device_seq_chunks(T, 8, 1, 6, 128) == T
    d = P.load("device_split_plan.json")
    for c in d["cases"]:
        if c.get("rows") in (256, 64) and c["sms"] == sms and c["L"] == 8448 and c["KVH"] == KVH:
            s = rows.index(c["rows"])
            want = [(j * c["c"], (j + 1) * c["c"]) for j in range(c["full"])]
            if c["tail"] is not None:
                want.append(tuple(c["tail"]))
            want += [(c["L"], c["L"])] * c["empty"]
            assert got[s].tolist() == [list(r) for r in want], c["work"]
