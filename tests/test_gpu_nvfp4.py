"""GPU parity of the NVFP4 weight format (E2M1 codes, E4M3 scales per 16 K,
fp32 global per expert and matrix) on each layer path that takes NVFP4 banks
(fused decode kernel, hybrid, tensor-core prefill), against the FP64 oracle's
NVFP4 layer; the prepared NVFP4 records against numpy reshapes of the
canonical banks; and the calls that refuse NVFP4 banks."""
import numpy as np
import pytest

import oracle
import synth
from gpu_common import DeviceLayer, assert_close, build_all, host_inputs, require_gpu, run_layer, torch_mod

pytestmark = pytest.mark.gpu

SEED = 20261203


@pytest.fixture(scope="module", autouse=True)
def _setup():
    require_gpu()
    build_all()


_layers = {}


def nv_layer(inter, E=512, k=10):
    key = (inter, E, k)
    if key not in _layers:
        _layers.clear()
        torch_mod().cuda.empty_cache()
        shape = synth.ExpertShape(num_experts=E, top_k=k, inter=inter, group=16, meta_bytes=1)
        _layers[key] = DeviceLayer(shape, SEED, 0)
    return _layers[key]


def nv_layer_at(layer, inter=160):
    """The NVFP4 bank set of `layer` (seeded per layer), cached one at a time."""
    key = ("layer", layer, inter)
    if key not in _layers:
        _layers.clear()
        torch_mod().cuda.empty_cache()
        shape = synth.ExpertShape(num_experts=512, top_k=10, inter=inter, group=16, meta_bytes=1)
        _layers[key] = DeviceLayer(shape, SEED, layer)
    return _layers[key]


def oracle_nvfp4(dl, x, ids, w):
    shape = dl.shape
    b = ({}, {}, {}, {})
    for e in sorted(set(int(v) for v in ids.ravel())):
        q13, s13, q2, s2 = synth.expert_weights(shape, dl.seed, dl.layer, e, 1)
        for d, a in zip(b, (q13, s13[..., 0], q2, s2[..., 0])):
            d[e] = a
    g = synth.nvfp4_global(dl.seed, dl.layer, shape.num_experts)
    return oracle.moe_layer_nvfp4(x, ids, w, shape, *b, g)


@pytest.mark.parametrize("inter", [160, 640])
def test_nvfp4_prepared_records_bit_exact(inter):
    shape = synth.ExpertShape(num_experts=6, top_k=2, inter=inter, group=16, meta_bytes=1)
    dl = DeviceLayer(shape, SEED + 1, 2)
    E, I, PJ, KP = 6, inter, inter // 8, inter // 160
    # words move exactly as in the int4 banks
    q13 = dl.w13_q.cpu().numpy().view(np.uint32).reshape(E, 80, 4, 2, PJ, 8)
    q2 = dl.w2_q.cpu().numpy().view(np.uint32).reshape(E, KP, 20, 80, 32)
    # scales: canonical [e][group 32][block b][half][j][g] -> records [e][j][group][g][half][b]
    m13 = dl.w13_m.cpu().numpy().reshape(E, 80, 2, 2, PJ, 8)
    # canonical [e][kp][group 0..4][b][tile][c] -> rows [e][kp][tile][group][c][b]
    m2 = dl.w2_m.cpu().numpy().reshape(E, KP, 5, 2, 80, 32)
    want = [q13.transpose(0, 4, 1, 2, 5, 3), m13.transpose(0, 4, 1, 5, 3, 2),
            q2.transpose(0, 1, 3, 2, 4), m2.transpose(0, 1, 4, 2, 5, 3)]
    got = [dl.p13_q.cpu().numpy().view(np.uint32), dl.p13_m.cpu().numpy(),
           dl.p2_q.cpu().numpy().view(np.uint32), dl.p2_m.cpu().numpy()]
    for g, w_ in zip(got, want):
        assert np.array_equal(g.ravel(), np.ascontiguousarray(w_).ravel())


@pytest.mark.parametrize("M,regime,inter", [(1, "rotating", 160), (2, "hot", 160), (4, "rotating", 160),
                                            (8, "hot", 160), (8, "rotating", 160), (9, "rotating", 160),
                                            (16, "hot", 160), (128, "zipf", 160), (300, "zipf", 160),
                                            (1, "rotating", 640), (16, "rotating", 640), (160, "zipf", 640)])
def test_nvfp4_layer_parity(M, regime, inter):
    """The layer call on NVFP4 banks against the oracle on every path that
    takes them: the fused decode kernel (up to 16 tokens; HW with its fp16
    residue plane), the hybrid path (stage W13 with the h residue plane,
    tensor-core W2) and the tensor-core prefill path."""
    import awq_int4_moe_gb300 as awq
    dl = nv_layer(inter)
    x, ids, w = host_inputs(SEED + M, 5, M, dl.shape, regime)
    ref, _ = oracle_nvfp4(dl, x, ids, w)
    out, st = run_layer(dl, x, ids, w, M)
    assert st == 0
    assert_close(out, ref, f"nvfp4 layer M={M} {regime} I={inter}")
    paths = (awq.PATH_PREFILL, awq.PATH_HYBRID) + ((awq.PATH_FUSED,) if M <= 16 else ())
    # AUTO takes the fused kernel up to 16 tokens, the hybrid path above
    auto = awq.PATH_FUSED if M <= 16 else awq.PATH_HYBRID
    for path in paths:
        o, s2 = run_layer(dl, x, ids, w, M, path=path)
        assert s2 == 0
        assert_close(o, ref, f"nvfp4 layer M={M} {regime} I={inter} path {path}")
        if path == auto:
            assert np.array_equal(o, out)


@pytest.mark.parametrize("layer", [0, 1, 2, 7])
def test_nvfp4_decode_sweep(layer):
    """NVFP4 decode batches (the path AWQ_PATH_AUTO takes: the fused kernel)
    over a sweep of token counts and both routing regimes, on four layers
    (different banks, inputs and routing), against the oracle."""
    dl = nv_layer_at(layer)
    for M in (1, 2, 3, 5, 8, 11, 16):
        for regime in ("hot", "rotating"):
            x, ids, w = host_inputs(SEED + 7 * M + layer, 9 + layer, M, dl.shape, regime)
            ref, _ = oracle_nvfp4(dl, x, ids, w)
            out, st = run_layer(dl, x, ids, w, M)
            assert st == 0
            assert_close(out, ref, f"nvfp4 M={M} {regime} layer {layer}")


@pytest.mark.parametrize("inter,A", [(160, 1), (160, 3), (160, 10), (160, 12), (160, 13), (160, 15),
                                     (160, 16), (640, 2), (640, 3), (640, 4)])
def test_nvfp4_fused_around_its_tile_mode_switch(inter, A):
    """The fused kernel on NVFP4 banks with exactly A distinct experts over 2
    tokens (repeats within a token where A < 10): its tile mode (units of 3
    segments, at most 4 units: A <= 12 at intermediate 160, A <= 3 with the
    four K parts of intermediate 640) and the flat schedule beyond, against
    the oracle; AUTO takes the same kernel."""
    import awq_int4_moe_gb300 as awq
    dl = nv_layer(inter)
    rng = np.random.default_rng(SEED + 31 * A + inter)
    experts = rng.choice(512, size=A, replace=False)
    M = 2
    ids = rng.permutation(np.resize(experts, M * 10)).reshape(M, 10).astype(np.int32)
    assert len(set(ids.ravel().tolist())) == A
    w = rng.dirichlet(np.ones(10), size=M).astype(np.float32)
    x = synth.hidden_states(SEED, 14, M, dl.shape.hidden)
    ref, _ = oracle_nvfp4(dl, x, ids, w)
    out, st = run_layer(dl, x, ids, w, M, path=awq.PATH_FUSED)
    assert st == 0
    assert_close(out, ref, f"nvfp4 fused A={A} I={inter}")
    auto, st = run_layer(dl, x, ids, w, M)
    assert st == 0
    assert np.array_equal(auto, out)


def test_nvfp4_refused_by_the_other_paths_and_calls():
    import awq_int4_moe_gb300 as awq
    torch = torch_mod()
    dl = nv_layer(160)
    M = 4
    x, ids, w = host_inputs(SEED, 6, M, dl.shape, "rotating")
    for path in (awq.PATH_SLICED, awq.PATH_STAGED):
        with pytest.raises(awq.AwqError) as ei:
            run_layer(dl, x, ids, w, M, path=path)
        assert ei.value.code == awq.ERR_UNSUPPORTED_SHAPE
    # the stage calls and the static entry point take int4 banks only
    S = M * 10
    i32 = dict(dtype=torch.int32, device="cuda")
    act, off, srt, na = (torch.zeros(S, **i32), torch.zeros(S + 1, **i32), torch.zeros(S, **i32),
                         torch.zeros(1, **i32))
    st = torch.zeros(1, **i32)
    h = torch.zeros((S, 160), dtype=torch.int16, device="cuda")
    xd = torch.zeros((M, 2560), dtype=torch.int16, device="cuda")
    with pytest.raises(awq.AwqError) as ei:
        awq.moe_w13_swiglu(xd, M, dl.c_shape(), dl.weights(), act, off, srt, na, h, st)
    assert ei.value.code == awq.ERR_UNSUPPORTED_SHAPE
    # NVFP4 banks without their global scales are refused before any launch
    wts = awq.Weights.of(dl.p13_q, dl.p13_m, dl.p2_q, dl.p2_m, awq.LAYOUT_PREPARED)
    with pytest.raises(awq.AwqError) as ei:
        ws_bytes = awq.moe_workspace_bytes(dl.c_shape(), M)
        ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
        out = torch.zeros((M, 2560), dtype=torch.int16, device="cuda")
        awq.moe_layer(xd, torch.zeros((M, 10), **i32), torch.zeros((M, 10), dtype=torch.float32, device="cuda"),
                      M, dl.c_shape(), wts, out, ws, ws_bytes, st)
    assert ei.value.code == awq.ERR_INVALID_ARG
