"""Shared helpers of the GPU tests: device banks from the seeded generator,
host inputs, the C-ABI calls, and the elementwise tolerance of the stage."""
from __future__ import annotations

import numpy as np

import synth

ATOL, RTOL = 4e-3, 1e-2        # |gpu - oracle| <= ATOL + RTOL * |oracle|


def torch_mod():
    import torch
    return torch


def require_gpu():
    import pytest
    torch = torch_mod()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def build_all():
    import awq_int4_moe_gb300.build as b
    import synth.device as sd
    b.build()
    sd.build()


class DeviceLayer:
    """One layer's four weight banks on the device, filled by the CUDA
    generator (byte-identical to synth.expert_weights)."""

    def __init__(self, shape: synth.ExpertShape, seed: int, layer: int = 0, meta_bytes=None):
        import synth.device as sd
        torch = torch_mod()
        mb = shape.meta_bytes if meta_bytes is None else meta_bytes
        E, H, I, G = shape.num_experts, shape.hidden, shape.inter, shape.group
        dev = "cuda"
        self.shape, self.seed, self.layer, self.mb = shape, seed, layer, mb
        self.w13_q = torch.empty((E, H // 8, 2 * I), dtype=torch.int32, device=dev)
        self.w13_m = torch.empty((E, H // G, 2 * I, mb), dtype=torch.uint8, device=dev)
        self.w2_q = torch.empty((E, I // 8, H), dtype=torch.int32, device=dev)
        self.w2_m = torch.empty((E, I // G, H, mb), dtype=torch.uint8, device=dev)
        sd.fill_layer(shape, seed, layer, self.w13_q, self.w13_m, self.w2_q, self.w2_m, mb)
        # prepared copies, the banks the compute calls read
        self.p13_q, self.p13_m = torch.empty_like(self.w13_q), torch.empty_like(self.w13_m)
        self.p2_q, self.p2_m = torch.empty_like(self.w2_q), torch.empty_like(self.w2_m)
        import awq_int4_moe_gb300 as awq
        self._prepared = awq.moe_prepare_weights(
            self.c_shape(), self.canonical_weights(),
            awq.Weights.of(self.p13_q, self.p13_m, self.p2_q, self.p2_m))
        # NVFP4 banks (group 16): the per-expert global scales, not permuted
        self.global_scale = None
        if shape.group == 16:
            self.global_scale = torch.from_numpy(synth.nvfp4_global(seed, layer, E)).to(dev)
            self._prepared.global_scale = self.global_scale.data_ptr()
        torch.cuda.synchronize()

    def canonical_weights(self):
        import awq_int4_moe_gb300 as awq
        return awq.Weights.of(self.w13_q, self.w13_m, self.w2_q, self.w2_m, awq.LAYOUT_CANONICAL)

    def weights(self):
        return self._prepared

    def c_shape(self):
        import awq_int4_moe_gb300 as awq
        s = self.shape
        return awq.Shape(s.num_experts, s.top_k, s.hidden, s.inter, s.group, self.mb)


def host_inputs(seed, layer, M, shape, regime):
    x = synth.hidden_states(seed, layer, M, shape.hidden)
    ids, w = synth.routing(seed, layer, M, shape.num_experts, shape.top_k, regime)
    return x, ids, w


def to_dev(a):
    torch = torch_mod()
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return torch.from_numpy(a.view(np.int16)).cuda()
    return torch.from_numpy(a).cuda()


def fp16_from_dev(t):
    return t.cpu().numpy().view(np.float16).astype(np.float64)


def run_layer(dl: DeviceLayer, x, ids, w, M, path=None, ws=None, timeout_ns=0, debug_flags=0):
    """awq_moe_layer (or awq_moe_layer_ex when a path is given) through the C
    ABI; returns (out f64[M][H], dev_status)."""
    import awq_int4_moe_gb300 as awq
    torch = torch_mod()
    shape = dl.c_shape()
    ws_bytes = awq.moe_workspace_bytes(shape, max(M, 1))
    if ws is None:
        ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.full((max(M, 1), shape.hidden), -1, dtype=torch.int16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    if path is None:
        awq.moe_layer(to_dev(x), to_dev(ids), to_dev(w), M, shape, dl.weights(), out, ws, ws_bytes, st)
    else:
        awq.moe_layer_ex(to_dev(x), to_dev(ids), to_dev(w), M, shape, dl.weights(), out, ws,
                         ws_bytes, st, path=path, timeout_ns=timeout_ns, debug_flags=debug_flags)
    torch.cuda.synchronize()
    return fp16_from_dev(out)[:M], int(st.item())


def run_stages(dl: DeviceLayer, x, ids, w, M):
    """route, W13 + SwiGLU and W2 as three C-ABI calls; returns a dict. The W2
    stage call takes at most W2_STAGE_MAX_TOKENS tokens: above that its
    "out" is None."""
    import awq_int4_moe_gb300 as awq
    torch = torch_mod()
    shape = dl.c_shape()
    S = M * shape.top_k
    dev = "cuda"
    act = torch.full((max(S, 1),), -7, dtype=torch.int32, device=dev)
    off = torch.full((S + 1,), -7, dtype=torch.int32, device=dev)
    srt = torch.full((max(S, 1),), -7, dtype=torch.int32, device=dev)
    na = torch.full((1,), -7, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    h = torch.zeros((max(S, 1), shape.inter), dtype=torch.int16, device=dev)
    out = torch.full((max(M, 1), shape.hidden), -1, dtype=torch.int16, device=dev)
    xd, idd, wd = to_dev(x), to_dev(ids), to_dev(w)
    awq.moe_route(idd, M, shape, act, off, srt, na, st)
    awq.moe_w13_swiglu(xd, M, shape, dl.weights(), act, off, srt, na, h, st)
    w2 = M <= awq.W2_STAGE_MAX_TOKENS
    if w2:
        awq.moe_w2_reduce(h, wd, M, shape, dl.weights(), act, off, srt, na, out, st)
    torch.cuda.synchronize()
    return dict(active=act.cpu().numpy()[:S], offsets=off.cpu().numpy(),
                sorted_slots=srt.cpu().numpy()[:S], num_active=int(na.item()),
                h=fp16_from_dev(h)[:S], out=fp16_from_dev(out)[:M] if w2 else None,
                status=int(st.item()))


def oracle_banks(shape, seed, layer, ids, mb):
    b = ({}, {}, {}, {})
    for e in sorted(set(int(v) for v in np.asarray(ids).ravel() if 0 <= v < shape.num_experts)):
        parts = synth.expert_weights(shape, seed, layer, e, mb)
        for d, p in zip(b, parts):
            d[e] = p
    return b


def assert_close(got, ref, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    rel_l2 = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())}/{bad.size} elements outside {ATOL} + {RTOL}*|ref|; "
            f"worst at {i}: got {got[i]!r} ref {ref[i]!r}; max abs {err.max():.3e}, "
            f"rel L2 {rel_l2:.3e}")
    return float(err.max()), rel_l2
