"""Several library calls captured back to back in one CUDA graph, the way
the benchmark launches them, over different KV copies that share one
workspace.  Each replayed output must equal the eager call bit for bit and
the oracle within tolerance.  This covers the programmatic dependency from
one call's merge to the next call's partial kernel inside a graph: the next
partial kernel overwrites the workspace the previous merge reads (hipfire
PR #817, "Default and admission policy": the fixed-grid route kept through
graph capture)."""
import numpy as np
import pytest

import oracle
import speculative_decoding_verify_kv_gb300 as va
import synthetic as sy
from gpu_util import compare

CALLS = 3

RECIPES = {
    # the benchmark's call shape at a shorter context
    "long-q8": ("long_q8", {"ctx": 4096}),
    # direct rows and tree suffixes over a paged Q8_0 cache
    "mixed-q8": ("mixed_tree_direct", {"ctx": [40, 300, 17, 130, 700, 5, 90, 2000]}),
    # bf16 cache (the other tensor-core kernel)
    "dflash-bf16": ("dflash_bf16", {"ctx": 2048}),
}


@pytest.mark.gpu
@pytest.mark.parametrize("name", sorted(RECIPES))
def test_graph_replay_matches_eager_and_oracle(name):
    import torch
    fn, kw = RECIPES[name]
    cases = [getattr(sy, fn)(seed=501 + i, **kw) for i in range(CALLS)]
    ups = [va.upload(c, "cuda", num_splits=8) for c in cases]
    mode = ups[0][2]
    ws = va.alloc_workspace(ups[0][0], ups[0][1])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    # Eager, one after another on the current stream, sharing the workspace.
    eager = []
    for p, kv, _ in ups:
        o, lse = va.verify_attn(p, kv, mode, ws=ws, status=status)
        eager.append((o.clone(), lse.clone()))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    eager = [(o.cpu().numpy(), l.cpu().numpy()) for o, l in eager]

    outs = [(torch.empty_like(torch.from_numpy(o)).cuda(), torch.empty_like(torch.from_numpy(l)).cuda())
            for o, l in eager]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for (p, kv, _), (o, lse) in zip(ups, outs):
            va.verify_attn(p, kv, mode, ws=ws, o=o, lse=lse, status=status)
    for rep in range(2):
        for o, lse in outs:
            o.fill_(float("nan"))
            lse.fill_(float("nan"))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        for i, ((o, lse), (eo, el)) in enumerate(zip(outs, eager)):
            go, gl = o.cpu().numpy(), lse.cpu().numpy()
            assert np.array_equal(go.view(np.uint32), eo.view(np.uint32)), f"replay {rep}, call {i}: O"
            assert np.array_equal(gl.view(np.uint32), el.view(np.uint32)), f"replay {rep}, call {i}: LSE"
    # The calls saw different KV copies, and each matches its own oracle.
    assert not np.array_equal(eager[0][1], eager[1][1])
    for i, c in enumerate(cases):
        O, L = oracle.verify_case(c)
        compare(eager[i][0], eager[i][1], O, L, f"{name} call {i}")
