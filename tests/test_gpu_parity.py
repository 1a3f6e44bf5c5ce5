"""GPU parity: the CUDA path through the C ABI against the FP64 CPU oracle.

Routing and the compact-metadata conversion are compared bit for bit; the
floating-point stages elementwise within |gpu - oracle| <= 4e-3 + 1e-2*|oracle|.
Each configuration of the workload table is covered (single token, grouped
decode hot/rotating, compact metadata, the prefill-sized Zipf batch, and the
unsharded intermediate 640), plus the edge cases of the method.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_common import (DeviceLayer, assert_close, build_all, fp16_from_dev, host_inputs, oracle_banks,
                        require_gpu, run_layer, run_stages, to_dev, torch_mod)

pytestmark = pytest.mark.gpu

SEED = 20261202


@pytest.fixture(scope="module", autouse=True)
def _setup():
    require_gpu()
    build_all()


_layers = {}


def device_layer(inter, mb, layer=0, E=512, k=10):
    key = (inter, mb, layer, E, k)
    if key not in _layers:
        if len(_layers) > 3:
            _layers.clear()
            torch_mod().cuda.empty_cache()
        shape = synth.ExpertShape(num_experts=E, top_k=k, inter=inter, meta_bytes=mb)
        _layers[key] = DeviceLayer(shape, SEED, layer)
    return _layers[key]


def check_case(dl, x, ids, w, M, stages=True):
    import awq_int4_moe_gb300 as awq
    shape = dl.shape
    banks = oracle_banks(shape, dl.seed, dl.layer, ids, dl.mb)
    ref_out, ref_h = oracle.moe_layer(x, ids, w, shape, *banks, dl.mb)
    out, status = run_layer(dl, x, ids, w, M)
    assert status == 0
    assert_close(out, ref_out, "layer out")
    # every execution path of the layer call that takes this M
    paths = ([awq.PATH_STAGED] if M <= awq.W2_STAGE_MAX_TOKENS else []) + [awq.PATH_PREFILL, awq.PATH_HYBRID] + \
        ([awq.PATH_FUSED] if M <= 16 else []) + \
        ([awq.PATH_SLICED] if M <= 8 and M * shape.top_k <= torch_mod().cuda.get_device_properties(0).multi_processor_count else [])
    for path in paths:
        o, st = run_layer(dl, x, ids, w, M, path=path)
        assert st == 0
        assert_close(o, ref_out, f"layer out (path {path})")
    if stages:
        r = run_stages(dl, x, ids, w, M)
        assert r["status"] == 0
        act, off, srt, A = oracle.route(ids, shape.num_experts)
        assert r["num_active"] == A
        assert np.array_equal(r["active"], act) and np.array_equal(r["offsets"], off)
        assert np.array_equal(r["sorted_slots"], srt)
        # W13 stage: h rows are in sorted-slot order
        assert_close(r["h"], ref_h[srt], "w13 h")
        if r["out"] is None:
            return out
        # W2 stage alone, fed the GPU's own fp16 h
        h_slot = np.zeros_like(ref_h)
        h_slot[srt] = r["h"]
        ref2 = oracle.w2_reduce(h_slot, ids, w, shape, banks[2], banks[3], dl.mb)
        assert_close(r["out"], ref2, "w2 out")
        # the staged layer path is exactly the composition of the stage calls
        o_staged, _ = run_layer(dl, x, ids, w, M, path=awq.PATH_STAGED)
        assert np.array_equal(r["out"], o_staged)
    return out


@pytest.mark.parametrize("mb", [4, 3])
def test_single_token(mb):
    dl = device_layer(160, mb)
    x, ids, w = host_inputs(SEED, 0, 1, dl.shape, "rotating")
    check_case(dl, x, ids, w, 1)


@pytest.mark.parametrize("M", [2, 4, 8])
@pytest.mark.parametrize("regime", ["hot", "rotating"])
def test_grouped_decode_4byte(M, regime):
    dl = device_layer(160, 4)
    x, ids, w = host_inputs(SEED + M, 1, M, dl.shape, regime)
    check_case(dl, x, ids, w, M)


@pytest.mark.parametrize("M,regime", [(1, "rotating"), (8, "hot"), (8, "rotating")])
def test_compact_3byte(M, regime):
    dl = device_layer(160, 3)
    x, ids, w = host_inputs(SEED + 10 + M, 2, M, dl.shape, regime)
    check_case(dl, x, ids, w, M)


def test_prefill_zipf_128():
    dl = device_layer(160, 4)
    x, ids, w = host_inputs(SEED, 3, 128, dl.shape, "zipf")
    counts = np.bincount(ids.ravel(), minlength=512)
    assert counts.max() > 8          # multi-tile segments are exercised
    check_case(dl, x, ids, w, 128)


@pytest.mark.parametrize("M,inter,mb", [(256, 160, 4), (512, 160, 4), (512, 160, 3), (256, 640, 3),
                                         (160, 640, 4)])
def test_prefill_beyond_128_tokens(M, inter, mb):
    """The tensor-core path (tcgen05 W13 + SwiGLU, W2 products, per-token sum)
    on Zipf-routed batches: hundreds of active experts, segments from 1 row to
    several 128-row work items. The W13 stage call above 128 tokens runs the
    same tensor-core kernel (checked against the oracle's h)."""
    dl = device_layer(inter, mb)
    x, ids, w = host_inputs(SEED + M, 4, M, dl.shape, "zipf")
    counts = np.bincount(ids.ravel(), minlength=512)
    assert counts.max() > 32                          # a segment spans several work items
    check_case(dl, x, ids, w, M)


def test_prefill_max_tokens_top16_duplicates():
    """M = AWQ_MAX_TOKENS with top-16 over 64 experts (segments of ~128
    rows, several items each) and a token whose 16 slots all name one expert."""
    import awq_int4_moe_gb300 as awq
    dl = device_layer(160, 4, E=64, k=16)
    M = awq.MAX_TOKENS
    rng = np.random.default_rng(5)
    x = synth.hidden_states(SEED, 14, M)
    ids = np.stack([rng.choice(64, 16, replace=False) for _ in range(M)]).astype(np.int32)
    ids[7, :] = 33
    w = rng.dirichlet(np.ones(16), size=M).astype(np.float32)
    check_case(dl, x, ids, w, M)


@pytest.mark.parametrize("path", ["prefill", "hybrid"])
def test_prefill_workspace_reuse_and_determinism(path):
    """Back-to-back prefill-path (and hybrid-path) calls of different M on
    one workspace match the oracle and repeat bit for bit (no float atomics:
    fixed-order sums)."""
    import awq_int4_moe_gb300 as awq
    torch = torch_mod()
    code = {"prefill": awq.PATH_PREFILL, "hybrid": awq.PATH_HYBRID}[path]
    dl = device_layer(160, 4)
    ws_bytes = awq.moe_workspace_bytes(dl.c_shape(), 300)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    first = {}
    cases = ((300, "zipf"), (1, "rotating"), (37, "zipf"), (129, "rotating"))
    for rep in range(2):
        for M, regime in cases:
            x, ids, w = host_inputs(SEED + 50 + M, 15, M, dl.shape, regime)
            out, st = run_layer(dl, x, ids, w, M, path=code, ws=ws)
            assert st == 0
            if rep == 0:
                banks = oracle_banks(dl.shape, dl.seed, dl.layer, ids, dl.mb)
                ref, _ = oracle.moe_layer(x, ids, w, dl.shape, *banks, dl.mb)
                assert_close(out, ref, f"prefill M={M} {regime}")
                first[(M, regime)] = out
            else:
                assert np.array_equal(out, first[(M, regime)])


def test_prefill_bad_expert_id_sets_device_status():
    import awq_int4_moe_gb300 as awq
    dl = device_layer(160, 4)
    M = 200
    x, ids, w = host_inputs(SEED, 16, M, dl.shape, "zipf")
    ids = ids.copy()
    ids[3, 4] = 512
    ids[150, 0] = -1
    _, status = run_layer(dl, x, ids, w, M)
    assert status == 6
    _, status = run_layer(dl, x, ids, w, M, path=awq.PATH_PREFILL)
    assert status == 6
    _, status = run_layer(dl, x, ids, w, M, path=awq.PATH_HYBRID)
    assert status == 6


def test_staged_path_refuses_beyond_its_token_limit():
    import awq_int4_moe_gb300 as awq
    dl = device_layer(160, 4)
    M = awq.W2_STAGE_MAX_TOKENS + 1
    x, ids, w = host_inputs(SEED, 17, M, dl.shape, "rotating")
    with pytest.raises(awq.AwqError) as ei:
        run_layer(dl, x, ids, w, M, path=awq.PATH_STAGED)
    assert ei.value.code == awq.ERR_UNSUPPORTED_SHAPE


@pytest.mark.parametrize("A", [10, 11, 12, 15, 16])
def test_active_expert_counts_around_the_w2_mode_switch(A):
    # the fused kernel's W2 runs in tile mode for few active experts and in the
    # flat mode above: both sides of the switch, with exactly A distinct experts
    dl = device_layer(160, 4)
    rng = np.random.default_rng(SEED + A)
    experts = rng.choice(512, size=A, replace=False)
    M = 2
    ids = np.empty((M, 10), np.int32)
    ids[0] = experts[:10]
    ids[1] = np.concatenate([experts[10:], experts[:10 - (A - 10)]])
    assert len(set(ids.ravel().tolist())) == A
    w = rng.random((M, 10)).astype(np.float32)
    w /= w.sum(axis=1, keepdims=True)
    x = synth.hidden_states(SEED, 0, M, dl.shape.hidden)
    check_case(dl, x, ids, w, M, stages=False)


@pytest.mark.parametrize("inter,mb,A", [(160, 4, 24), (160, 4, 25), (160, 3, 23), (640, 3, 6), (640, 4, 7)])
def test_sliced_kernel_around_its_tile_mode_switch(inter, mb, A):
    # the sliced kernel computes W2 in tile mode when A * (inter / 160) <= 24
    # and sliced along K above: exactly A distinct experts over 4 tokens, both
    # sides of the switch, at both intermediate sizes
    dl = device_layer(inter, mb)
    rng = np.random.default_rng(SEED + 100 * A + inter)
    experts = rng.choice(512, size=A, replace=False)
    M = 4
    # every expert at least once over the 40 slots (a token may repeat one)
    ids = rng.permutation(np.resize(experts, M * 10)).reshape(M, 10).astype(np.int32)
    assert len(set(ids.ravel().tolist())) == A
    w = rng.dirichlet(np.ones(10), size=M).astype(np.float32)
    x = synth.hidden_states(SEED, 5, M, dl.shape.hidden)
    check_case(dl, x, ids, w, M, stages=False)


@pytest.mark.parametrize("inter,mb,M,k", [(640, 3, 1, 2), (640, 4, 3, 1), (640, 3, 8, 1), (160, 4, 1, 2)])
def test_fused_tile_mode_with_few_experts(inter, mb, M, k):
    # at most 3 active experts: the fused kernel's tile mode, at intermediate 640
    # with its four 160-row K parts per unit (one unit per K part)
    dl = device_layer(inter, mb, k=k)
    rng = np.random.default_rng(SEED + M * 7 + k)
    chosen = rng.choice(512, size=3, replace=False)
    ids = np.stack([rng.choice(chosen, size=k, replace=False) for _ in range(M)]).astype(np.int32)
    w = rng.dirichlet(np.ones(k), size=M).astype(np.float32)
    x = synth.hidden_states(SEED, 12, M, dl.shape.hidden)
    check_case(dl, x, ids, w, M, stages=False)


def test_staged_items_with_four_k_parts():
    # intermediate 640 (four 160-row K parts per W2 tile) with segments longer
    # than one 16-row work item: the staged W2 kernel's items x K parts
    dl = device_layer(640, 3)
    x, ids, w = host_inputs(SEED, 4, 40, dl.shape, "zipf")
    assert np.bincount(ids.ravel(), minlength=512).max() > 16
    check_case(dl, x, ids, w, 40, stages=False)


@pytest.mark.parametrize("M", [1, 2, 4, 8, 16])
def test_unsharded_inter_640(M):
    dl = device_layer(640, 3)
    x, ids, w = host_inputs(SEED + 20 + M, 4, M, dl.shape, "rotating")
    check_case(dl, x, ids, w, M, stages=(M in (1, 16)))


def test_layouts_give_identical_outputs():
    d4, d3 = device_layer(160, 4), device_layer(160, 3)
    x, ids, w = host_inputs(SEED, 5, 8, d4.shape, "rotating")
    o4, s4 = run_layer(d4, x, ids, w, 8)
    o3, s3 = run_layer(d3, x, ids, w, 8)
    assert s4 == 0 and s3 == 0
    assert np.array_equal(o4, o3)


def test_run_to_run_deterministic():
    dl = device_layer(160, 4)
    x, ids, w = host_inputs(SEED, 6, 128, dl.shape, "zipf")
    a, _ = run_layer(dl, x, ids, w, 128)
    b, _ = run_layer(dl, x, ids, w, 128)
    assert np.array_equal(a, b)


# ------------------------------------------------------------------ edge cases

def test_all_tokens_on_one_expert_with_duplicate_slots():
    dl = device_layer(160, 4)
    M = 8
    x = synth.hidden_states(SEED, 7, M)
    ids = np.full((M, 10), 37, np.int32)                 # every slot on expert 37
    w = np.full((M, 10), 0.1, np.float32)
    check_case(dl, x, ids, w, M)


def test_duplicate_ids_within_a_token():
    dl = device_layer(160, 4)
    M = 3
    x = synth.hidden_states(SEED, 8, M)
    ids = np.array([[5, 5, 9, 1, 2, 3, 4, 6, 7, 8],
                    [9, 9, 9, 9, 0, 0, 511, 511, 100, 5],
                    [1, 2, 3, 4, 5, 6, 7, 8, 9, 10]], np.int32)
    w = np.random.default_rng(1).dirichlet(np.ones(10), size=M).astype(np.float32)
    check_case(dl, x, ids, w, M)


def test_extreme_expert_ids_and_zero_weights():
    dl = device_layer(160, 3)
    M = 2
    x = synth.hidden_states(SEED, 9, M)
    ids = np.array([[0, 511, 1, 510, 2, 509, 3, 508, 4, 507],
                    [511, 0, 256, 255, 128, 127, 64, 63, 32, 31]], np.int32)
    w = np.zeros((M, 10), np.float32)
    w[:, 0] = 1.0
    check_case(dl, x, ids, w, M)


def test_small_expert_count_and_top1():
    dl = device_layer(160, 4, E=16, k=1)
    M = 33
    x = synth.hidden_states(SEED, 10, M)
    ids = (np.arange(M) % 5).reshape(M, 1).astype(np.int32)
    w = np.ones((M, 1), np.float32)
    check_case(dl, x, ids, w, M)


def test_max_tokens_and_top16():
    dl = device_layer(160, 4, E=64, k=16)
    M = 128
    rng = np.random.default_rng(3)
    x = synth.hidden_states(SEED, 11, M)
    ids = np.stack([rng.choice(64, 16, replace=False) for _ in range(M)]).astype(np.int32)
    w = rng.dirichlet(np.ones(16), size=M).astype(np.float32)
    check_case(dl, x, ids, w, M, stages=False)


def test_bad_expert_id_sets_device_status():
    dl = device_layer(160, 4)
    x = synth.hidden_states(SEED, 12, 2)
    ids = np.array([[1, 2, 3, 4, 5, 6, 7, 8, 9, 512], [1, 2, 3, 4, 5, 6, 7, 8, 9, -3]], np.int32)
    w = np.full((2, 10), 0.1, np.float32)
    _, status = run_layer(dl, x, ids, w, 2)
    assert status == 6
    r = run_stages(dl, x, ids, w, 2)
    assert r["status"] == 6
    # the valid slots still form correct segments; the bad ones are left out
    assert r["num_active"] == 9
    assert list(r["active"][:9]) == list(range(1, 10))
    assert r["offsets"][9] == 18


# ------------------------------------------------------------ route, compact

@pytest.mark.parametrize("M,k,E,seed", [(0, 10, 512, 0), (1, 10, 512, 1), (8, 10, 512, 2),
                                        (128, 10, 512, 3), (128, 16, 1024, 4), (77, 3, 7, 5),
                                        (5, 1, 1, 6), (512, 10, 512, 7), (512, 16, 1024, 8)])
def test_route_bit_exact(M, k, E, seed):
    import awq_int4_moe_gb300 as awq
    torch = torch_mod()
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, E, size=(M, k)).astype(np.int32)
    S = M * k
    shape = awq.Shape(E, k, 2560, 160, 32, 4)
    act = torch.full((max(S, 1),), -7, dtype=torch.int32, device="cuda")
    off = torch.full((S + 1,), -7, dtype=torch.int32, device="cuda")
    srt = torch.full((max(S, 1),), -7, dtype=torch.int32, device="cuda")
    na = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    idd = to_dev(ids) if S else torch.zeros(1, dtype=torch.int32, device="cuda")
    awq.moe_route(idd, M, shape, act, off, srt, na, st)
    torch.cuda.synchronize()
    if S:
        a, o, s, A = oracle.route(ids, E)
    else:
        a, o, s, A = np.zeros(0, np.int32), np.zeros(1, np.int32), np.zeros(0, np.int32), 0
    assert int(na.item()) == A and int(st.item()) == 0
    assert np.array_equal(act.cpu().numpy()[:S], a)
    assert np.array_equal(off.cpu().numpy(), o)
    assert np.array_equal(srt.cpu().numpy()[:S], s)


@pytest.mark.parametrize("n,offset", [(1, 0), (37, 0), (4096 + 3, 0), (1000, 1), (25600 * 512, 0)])
def test_prepare_compact_bit_exact(n, offset):
    import awq_int4_moe_gb300 as awq
    torch = torch_mod()
    rng = np.random.default_rng(n)
    m4 = rng.integers(0, 256, size=(n, 4), dtype=np.uint8)
    buf4 = torch.zeros(4 * n + 16, dtype=torch.uint8, device="cuda")
    buf3 = torch.zeros(3 * n + 16, dtype=torch.uint8, device="cuda")
    buf4[4 * offset:4 * offset + 4 * n] = torch.from_numpy(m4.ravel()).cuda()
    awq.prepare_compact(buf4.data_ptr() + 4 * offset, buf3.data_ptr() + 3 * offset, n)
    torch.cuda.synchronize()
    got = buf3.cpu().numpy()[3 * offset:3 * offset + 3 * n].reshape(n, 3)
    assert np.array_equal(got, oracle.prepare_compact(m4))
    assert not buf3.cpu().numpy()[3 * offset + 3 * n:].any()


def test_device_generator_matches_host_generator():
    for inter, mb in ((160, 4), (160, 3), (640, 3)):
        dl = device_layer(inter, mb, layer=7)
        for e in (0, 123, 511):
            ref = synth.expert_weights(dl.shape, dl.seed, dl.layer, e, mb)
            got = [dl.w13_q[e].cpu().numpy().view(np.uint32), dl.w13_m[e].cpu().numpy(),
                   dl.w2_q[e].cpu().numpy().view(np.uint32), dl.w2_m[e].cpu().numpy()]
            for g, r in zip(got, ref):
                assert np.array_equal(g, r)


@pytest.mark.parametrize("inter,mb", [(160, 4), (160, 3), (640, 4), (640, 3)])
def test_prepare_weights_permutation_bit_exact(inter, mb):
    """awq_moe_prepare_weights against the prepared order written as numpy
    reshapes of the canonical banks (whole words and records move, nothing
    else changes)."""
    shape = synth.ExpertShape(num_experts=6, top_k=2, inter=inter, meta_bytes=mb)
    dl = DeviceLayer(shape, SEED + 5, 3)
    E, I, PJ, KP = 6, inter, inter // 8, inter // 160
    # W13: [e][group][t][half][j][g] -> pieces [e][j][group][t][g][half]
    q13 = dl.w13_q.cpu().numpy().view(np.uint32).reshape(E, 80, 4, 2, PJ, 8)
    m13 = dl.w13_m.cpu().numpy().reshape(E, 80, 2, PJ, 8, mb)
    # W2: [e][kp][r][tile][32] -> lines [e][kp][tile][r][32]
    q2 = dl.w2_q.cpu().numpy().view(np.uint32).reshape(E, KP, 20, 80, 32)
    m2 = dl.w2_m.cpu().numpy().reshape(E, KP, 5, 80, 32, mb)
    want = [q13.transpose(0, 4, 1, 2, 5, 3), m13.transpose(0, 3, 1, 4, 2, 5),
            q2.transpose(0, 1, 3, 2, 4), m2.transpose(0, 1, 3, 2, 4, 5)]
    got = [dl.p13_q.cpu().numpy().view(np.uint32), dl.p13_m.cpu().numpy(),
           dl.p2_q.cpu().numpy().view(np.uint32), dl.p2_m.cpu().numpy()]
    for g, w_ in zip(got, want):
        assert np.array_equal(g.ravel(), np.ascontiguousarray(w_).ravel())


# ------------------------------------------------------------ fused path only

@pytest.mark.parametrize("path", ["fused", "sliced"])
def test_fused_workspace_reuse_and_determinism(path):
    """Counters in the workspace reset themselves: back-to-back calls on one
    workspace (different M and routings) all match the oracle and repeat."""
    import awq_int4_moe_gb300 as awq
    torch = torch_mod()
    dl = device_layer(160, 4)
    ws_bytes = awq.moe_workspace_bytes(dl.c_shape(), 16)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    first = {}
    cases = ((1, "rotating"), (8, "hot"), (16, "rotating"), (3, "zipf"), (8, "rotating"))
    if path == "sliced":
        cases = ((1, "rotating"), (8, "hot"), (5, "rotating"), (3, "zipf"), (8, "rotating"), (2, "hot"))
    p = awq.PATH_FUSED if path == "fused" else awq.PATH_SLICED
    for rep in range(2):
        for M, regime in cases:
            x, ids, w = host_inputs(SEED + 40 + M, 13, M, dl.shape, regime)
            out, st = run_layer(dl, x, ids, w, M, path=p, ws=ws)
            assert st == 0
            if rep == 0:
                banks = oracle_banks(dl.shape, dl.seed, dl.layer, ids, dl.mb)
                ref, _ = oracle.moe_layer(x, ids, w, dl.shape, *banks, dl.mb)
                assert_close(out, ref, f"fused M={M} {regime}")
                first[(M, regime)] = out
            else:
                assert np.array_equal(out, first[(M, regime)])


def test_fused_single_expert_everywhere():
    """A = 1: far fewer work units than CTAs (empty shares)."""
    dl = device_layer(160, 3)
    M = 4
    x = synth.hidden_states(SEED, 14, M)
    ids = np.full((M, 10), 300, np.int32)
    w = np.full((M, 10), 0.1, np.float32)
    check_case(dl, x, ids, w, M, stages=False)


def test_fused_bounded_wait_reports_timeout():
    """Debug bit 0 withholds one W13 piece's announcement, so the W2 phase's
    bounded wait runs out: the call returns, the status word says
    AWQ_ERR_DEVICE_TIMEOUT, and the context stays usable."""
    import awq_int4_moe_gb300 as awq
    torch = torch_mod()
    dl = device_layer(160, 4)
    x, ids, w = host_inputs(SEED, 15, 2, dl.shape, "rotating")
    ws_bytes = awq.moe_workspace_bytes(dl.c_shape(), 2)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    out, st = run_layer(dl, x, ids, w, 2, path=awq.PATH_FUSED, ws=ws, timeout_ns=20_000_000, debug_flags=1)
    assert st == awq.ERR_DEVICE_TIMEOUT
    # the same workspace, not cleared, serves the following calls correctly
    banks = oracle_banks(dl.shape, dl.seed, dl.layer, ids, dl.mb)
    ref, _ = oracle.moe_layer(x, ids, w, dl.shape, *banks, dl.mb)
    for _ in range(3):
        out, st = run_layer(dl, x, ids, w, 2, path=awq.PATH_FUSED, ws=ws)
        assert st == 0
        assert_close(out, ref, "fused after a timed-out call")
    # the device still works and a clean workspace gives the right answer
    banks = oracle_banks(dl.shape, dl.seed, dl.layer, ids, dl.mb)
    ref, _ = oracle.moe_layer(x, ids, w, dl.shape, *banks, dl.mb)
    out, st = run_layer(dl, x, ids, w, 2, path=awq.PATH_FUSED)
    assert st == 0
    assert_close(out, ref, "after timeout")
    torch.cuda.synchronize()


@pytest.mark.parametrize("inter,mb", [(160, 4), (640, 3)])
def test_sliced_bounded_barrier_wait_reports_timeout(inter, mb):
    """Debug bit 0 makes CTA 0 reach the sliced kernel's grid barrier only
    after twice the wait limit, so every other CTA's bounded wait runs out:
    the call returns, the status word says AWQ_ERR_DEVICE_TIMEOUT, and the
    same workspace, not cleared, serves the following calls correctly."""
    import awq_int4_moe_gb300 as awq
    torch = torch_mod()
    dl = device_layer(inter, mb)
    x, ids, w = host_inputs(SEED, 16, 4, dl.shape, "rotating")
    ws_bytes = awq.moe_workspace_bytes(dl.c_shape(), 4)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    out, st = run_layer(dl, x, ids, w, 4, path=awq.PATH_SLICED, ws=ws, timeout_ns=20_000_000, debug_flags=1)
    assert st == awq.ERR_DEVICE_TIMEOUT
    banks = oracle_banks(dl.shape, dl.seed, dl.layer, ids, dl.mb)
    ref, _ = oracle.moe_layer(x, ids, w, dl.shape, *banks, dl.mb)
    for _ in range(3):
        out, st = run_layer(dl, x, ids, w, 4, path=awq.PATH_SLICED, ws=ws)
        assert st == 0
        assert_close(out, ref, "sliced after a timed-out call")


def test_sliced_rejects_what_it_cannot_run():
    """The sliced path takes M <= 8 with M * top_k <= multiprocessors; an
    explicit request outside that fails closed (nothing launched)."""
    import awq_int4_moe_gb300 as awq
    dl = device_layer(160, 4)
    x, ids, w = host_inputs(SEED, 17, 9, dl.shape, "rotating")
    with pytest.raises(awq.AwqError) as ei:
        run_layer(dl, x, ids, w, 9, path=awq.PATH_SLICED)
    assert ei.value.code == awq.ERR_UNSUPPORTED_SHAPE


# ------------------------------------------------------------------ router from logits
# Ids bit-exact (the choice is taken on the fp32 logits, as the FP64 softmax
# orders them); weights within 4e-6 relative: fp32 exp (a few ulp), a sum of
# ten terms and one division, each at most ~1e-7 relative.
W_RTOL = 4e-6


def run_router(lg, M):
    import awq_int4_moe_gb300 as awq
    torch = torch_mod()
    shape = device_layer(160, 4).c_shape()
    ids = torch.full((max(M, 1), shape.top_k), -7, dtype=torch.int32, device="cuda")
    w = torch.full((max(M, 1), shape.top_k), -7.0, dtype=torch.float32, device="cuda")
    awq.moe_router_topk(to_dev(np.ascontiguousarray(lg, np.float32)), M, shape, ids, w)
    torch.cuda.synchronize()
    return ids.cpu().numpy()[:M], w.cpu().numpy()[:M]


@pytest.mark.parametrize("M,regime", [(1, "rotating"), (3, "hot"), (8, "rotating"), (16, "zipf"),
                                      (100, "rotating"), (128, "zipf")])
def test_router_topk_parity(M, regime):
    lg = synth.router_logits(SEED, 7, M, regime=regime)
    ids_o, w_o = oracle.router_topk(lg, 10)
    ids, w = run_router(lg, M)
    np.testing.assert_array_equal(ids, ids_o)
    np.testing.assert_allclose(w, w_o, rtol=W_RTOL, atol=0)


def test_router_ties_and_equal_rows():
    rng = np.random.default_rng(SEED)
    lg = rng.integers(-3, 4, size=(12, 512)).astype(np.float32)     # many ties
    lg[0] = 0.0                                                     # all equal
    lg[1] = -2.5
    lg[1, 511] = 7.0                                                # one far ahead
    ids_o, w_o = oracle.router_topk(lg, 10)
    ids, w = run_router(lg, 12)
    np.testing.assert_array_equal(ids, ids_o)
    np.testing.assert_allclose(w, w_o, rtol=W_RTOL, atol=0)
    assert ids[0].tolist() == list(range(10))


def test_router_zero_tokens_is_a_no_op():
    ids, w = run_router(np.zeros((1, 512), np.float32), 0)
    assert ids.shape == (0, 10)


@pytest.mark.parametrize("M,regime,path", [(1, "rotating", None), (2, "hot", None), (8, "rotating", None),
                                           (16, "zipf", None), (24, "rotating", None), (8, "hot", "staged")])
def test_layer_from_logits_parity(M, regime, path):
    import awq_int4_moe_gb300 as awq
    torch = torch_mod()
    dl = device_layer(160, 4)
    shape = dl.c_shape()
    x = synth.hidden_states(SEED, 7, M, shape.hidden)
    lg = synth.router_logits(SEED, 7, M, regime=regime)
    ids_o, w_o = oracle.router_topk(lg, 10)
    banks = oracle_banks(dl.shape, dl.seed, dl.layer, ids_o, dl.mb)
    ref_out, _ = oracle.moe_layer(x, ids_o, w_o.astype(np.float32), dl.shape, *banks, dl.mb)
    ws_bytes = awq.moe_workspace_bytes(shape, M)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.full((M, shape.hidden), -1, dtype=torch.int16, device="cuda")
    ids = torch.full((M, 10), -7, dtype=torch.int32, device="cuda")
    w = torch.full((M, 10), -7.0, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    p = awq.PATH_STAGED if path == "staged" else awq.PATH_AUTO
    awq.moe_layer_logits(to_dev(x), to_dev(lg), M, shape, dl.weights(), out, ids, w, ws, ws_bytes, st, path=p)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    np.testing.assert_array_equal(ids.cpu().numpy(), ids_o)
    np.testing.assert_allclose(w.cpu().numpy(), w_o, rtol=W_RTOL, atol=0)
    assert_close(fp16_from_dev(out), ref_out, "layer from logits")


@pytest.mark.parametrize("inter,mb,M,regime", [(160, 4, 1, "hot"), (160, 4, 2, "rotating"), (160, 4, 3, "rotating"),
                                               (160, 4, 8, "hot"), (160, 4, 16, "rotating"),
                                               (160, 4, 17, "zipf"), (160, 3, 200, "zipf"),
                                               (640, 3, 1, "rotating"), (640, 3, 2, "rotating")])
def test_auto_takes_the_documented_path(inter, mb, M, regime):
    """awq_moe_layer (AWQ_PATH_AUTO) gives, bit for bit, the output of the path
    the header documents for that call shape: the sliced kernel at M = 2 and
    at M = 1 with intermediate 160, the fused kernel at other M <= 16, the
    hybrid path above."""
    import awq_int4_moe_gb300 as awq
    dl = device_layer(inter, mb)
    x, ids, w = host_inputs(SEED + 3 * M, 17, M, dl.shape, regime)
    auto, st = run_layer(dl, x, ids, w, M)
    assert st == 0
    if M == 2 or (M == 1 and inter == 160):
        path = awq.PATH_SLICED
    elif M <= 16:
        path = awq.PATH_FUSED
    else:
        path = awq.PATH_HYBRID
    want, st = run_layer(dl, x, ids, w, M, path=path)
    assert st == 0
    assert np.array_equal(auto.view(np.uint64), want.view(np.uint64))
