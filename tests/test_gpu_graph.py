"""The timed path under parity: the benchmark's own stack of layer calls.

bench.py times one CUDA graph per case that holds the layer calls of a whole
stack of independently seeded layers, chained by programmatic dependent
launch and all sharing one workspace. This test builds that graph with the
benchmark's own functions on a small stack, replays it back to back without
a host synchronisation between replays, and compares every layer's output
with the FP64 oracle element by element (|gpu - oracle| <= 4e-3 + 1e-2
|oracle|); the replays must also agree bit for bit.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_common import assert_close, build_all, require_gpu, torch_mod

pytestmark = pytest.mark.gpu

LAYERS = 8
SEED = 424242


@pytest.fixture(scope="module", autouse=True)
def _setup():
    require_gpu()
    build_all()


@pytest.mark.parametrize("inter, mb, group, cases", [
    # the decode kernels (sliced, fused) and the hybrid path's four launches
    (160, 4, 32, [(1, "rotating"), (2, "hot"), (2, "rotating"), (8, "hot"), (8, "rotating"), (16, "rotating"),
                  (32, "zipf")]),
    (640, 3, 32, [(8, "rotating")]),
    # NVFP4 banks: the fused kernel and the hybrid path
    (160, 1, 16, [(1, "rotating"), (8, "hot"), (24, "zipf")]),
])
def test_stack_graph_replays_match_oracle(inter, mb, group, cases):
    import bench
    import awq_int4_moe_gb300 as awq
    torch = torch_mod()
    dev = torch.device("cuda", 0)
    shape = synth.ExpertShape(num_experts=512, top_k=10, hidden=2560, inter=inter, group=group, meta_bytes=mb)
    stack = bench.LayerStack(LAYERS, shape, SEED, dev)
    c_shape = awq.Shape.of(shape)
    ws_bytes = awq.moe_workspace_bytes(c_shape, max(m for m, _ in cases))
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(dev)
    per_case = [bench.make_case(M, r, stack, dev) for M, r in cases]
    for c in per_case:
        c["graph"] = bench.capture_stack_graph(c, stack, ws, ws_bytes, status, stream)
    torch.cuda.synchronize()
    firsts = []
    with torch.cuda.stream(stream):
        # every case's graph, then every case's again, then a third time: no
        # host synchronisation anywhere in between
        for c in per_case:
            c["graph"].replay()
            firsts.append(c["out"].clone())
        for _ in range(2):
            for c in per_case:
                c["graph"].replay()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for c, first in zip(per_case, firsts):
        assert torch.equal(c["out"], first), f"M={c['M']} {c['regime']}: replays differ"
        for layer in range(LAYERS):
            ref, _ = oracle.layer_from_synth(shape, SEED, layer, c["xs"][layer], c["ids"][layer], c["wts"][layer])
            got = c["out"][layer].cpu().numpy().view(np.float16).astype(np.float64)
            assert_close(got, ref, f"M={c['M']} {c['regime']} layer {layer}")
