"""GPU checks of the latency-floor helper (awq_moe_latency_floor): it writes
zero rows, reports a clean status, advances the workspace's grid-barrier
counter by one arrival per CTA, reports bad expert ids, and leaves the layer
calls that share its workspace bit-identical to calls on a fresh one."""
import numpy as np
import pytest

import awq_int4_moe_gb300 as awq
import synth
from gpu_common import DeviceLayer, build_all, host_inputs, require_gpu, run_layer, to_dev, torch_mod

pytestmark = pytest.mark.gpu

SEED = 20261204
GBAR_OFFSET = 1536     # the grid-barrier counter inside the workspace's counter region


@pytest.fixture(scope="module", autouse=True)
def _setup():
    require_gpu()
    build_all()


@pytest.fixture(scope="module")
def layer():
    return DeviceLayer(synth.ExpertShape(num_experts=512, top_k=10, inter=160), SEED, 0)


def _floor(dl, ids, M, ws, ws_bytes):
    torch = torch_mod()
    shape = dl.c_shape()
    out = torch.full((max(M, 1), shape.hidden), -1, dtype=torch.int16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    awq.moe_latency_floor(to_dev(ids), M, shape, dl.weights(), out, ws, ws_bytes, st)
    torch.cuda.synchronize()
    return out, int(st.item())


def _gbar(ws):
    return int(ws[GBAR_OFFSET:GBAR_OFFSET + 8].cpu().numpy().view(np.uint64)[0])


@pytest.mark.parametrize("M,regime", [(1, "rotating"), (4, "hot"), (8, "zipf"), (16, "rotating")])
def test_floor_writes_zeros_and_counts_arrivals(layer, M, regime):
    torch = torch_mod()
    shape = layer.c_shape()
    ws_bytes = awq.moe_workspace_bytes(shape, 16)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    _, ids, _ = host_inputs(SEED, 0, M, layer.shape, regime)
    for call in range(3):
        out, st = _floor(layer, ids, M, ws, ws_bytes)
        assert st == awq.OK
        assert int((out[:M] != 0).sum().item()) == 0
        assert _gbar(ws) == (call + 1) * sms


def test_floor_reports_bad_ids(layer):
    torch = torch_mod()
    shape = layer.c_shape()
    ws_bytes = awq.moe_workspace_bytes(shape, 16)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    _, ids, _ = host_inputs(SEED, 0, 2, layer.shape, "rotating")
    ids = ids.copy()
    ids[1, 3] = shape.num_experts
    _, st = _floor(layer, ids, 2, ws, ws_bytes)
    assert st == awq.ERR_BAD_EXPERT_ID


@pytest.mark.parametrize("path", [awq.PATH_SLICED, awq.PATH_FUSED])
def test_layer_after_floor_on_shared_workspace(layer, path):
    torch = torch_mod()
    shape = layer.c_shape()
    M = 8
    x, ids, w = host_inputs(SEED, 1, M, layer.shape, "zipf")
    fresh, st0 = run_layer(layer, x, ids, w, M, path=path)
    assert st0 == awq.OK
    ws_bytes = awq.moe_workspace_bytes(shape, 16)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        _, st = _floor(layer, ids, M, ws, ws_bytes)
        assert st == awq.OK
        got, st1 = run_layer(layer, x, ids, w, M, path=path, ws=ws)
        assert st1 == awq.OK
        assert np.array_equal(got.view(np.uint64), fresh.view(np.uint64))
