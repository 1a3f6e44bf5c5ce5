"""The allocation-free layer call (awq_moe_layer_static) against the
workspace-taking awq_moe_layer, on the GPU. Collected last (file name) so it
also runs after every other GPU test has used the device."""
import numpy as np
import pytest

import synth
from gpu_common import (DeviceLayer, assert_close, build_all, host_inputs, require_gpu, run_layer,
                        to_dev, fp16_from_dev, torch_mod)

pytestmark = pytest.mark.gpu

SEED = 77001


@pytest.fixture(scope="module", autouse=True)
def _setup():
    require_gpu()
    build_all()


def static_layer(dl, x, ids, w, M):
    import awq_int4_moe_gb300 as awq
    torch = torch_mod()
    out = torch.full((M, dl.shape.hidden), -1, dtype=torch.int16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    awq.moe_layer_static(to_dev(x), to_dev(ids), to_dev(w), M, dl.c_shape(), dl.weights(), out, st)
    torch.cuda.synchronize()
    return fp16_from_dev(out), int(st.item())


@pytest.mark.parametrize("inter,mb,cases", [
    (160, 4, ((8, "rotating"), (3, "hot"))),
    (640, 3, ((16, "zipf"), (1, "rotating"))),
])
def test_static_scratch_matches_workspace_call_twice_in_a_row(inter, mb, cases):
    shape = synth.ExpertShape(num_experts=512, top_k=10, inter=inter, meta_bytes=mb)
    dl = DeviceLayer(shape, SEED, 2)
    for M, regime in cases:          # two calls in a row on the same static scratch
        x, ids, w = host_inputs(SEED + M, 4, M, shape, regime)
        ref, st_ref = run_layer(dl, x, ids, w, M)
        got, st = static_layer(dl, x, ids, w, M)
        assert st_ref == 0 and st == 0
        assert_close(got, ref, f"static M={M} {regime}")
