"""CPU oracle of the AWQ int4 MoE expert stage -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package. It wraps the plain-C FP64 oracle in
``oracle/awq_moe_oracle.c`` (built with ``gcc`` by :func:`build`) and shares
no code with the CUDA library.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "awq_moe_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

OK, BAD_ARG, BAD_EXPERT_ID, NO_MEMORY = 0, 1, 6, 7


def build(force: bool = False) -> str:
    """Compile the oracle to ``oracle/liboracle.so`` (plain C11, FP64, no FMA
    contraction so that x86 and Arm hosts give identical results)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "awq_moe_oracle.h"))):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(_LIB)
        P = C.c_void_p
        i32 = C.c_int
        L.awqo_half_to_double.restype = C.c_double
        L.awqo_half_to_double.argtypes = [C.c_uint16]
        L.awqo_decode_matrix.restype = i32
        L.awqo_decode_matrix.argtypes = [P, P, i32, i32, i32, i32, P]
        L.awqo_prepare_compact.restype = None
        L.awqo_prepare_compact.argtypes = [P, P, C.c_int64]
        L.awqo_route.restype = i32
        L.awqo_route.argtypes = [P, i32, i32, i32, P, P, P, P]
        L.awqo_w13_swiglu.restype = i32
        L.awqo_w13_swiglu.argtypes = [P, P, i32, i32, i32, i32, i32, i32, i32, P, P, P]
        L.awqo_w2_reduce.restype = i32
        L.awqo_w2_reduce.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32, i32, P, P, P]
        L.awqo_moe_layer.restype = i32
        L.awqo_moe_layer.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32, i32,
                                     P, P, P, P, P, P]
        L.awqo_router_topk.restype = i32
        L.awqo_router_topk.argtypes = [P, i32, i32, i32, P, P]
        L.awqo_e2m1_to_double.restype = C.c_double
        L.awqo_e2m1_to_double.argtypes = [C.c_uint8]
        L.awqo_e4m3_to_double.restype = C.c_double
        L.awqo_e4m3_to_double.argtypes = [C.c_uint8]
        L.awqo_decode_nvfp4.restype = i32
        L.awqo_decode_nvfp4.argtypes = [P, P, C.c_float, i32, i32, P]
        L.awqo_moe_layer_nvfp4.restype = i32
        L.awqo_moe_layer_nvfp4.argtypes = [P, P, P, i32, i32, i32, i32, i32, P, P, P, P, P, P, P]
        _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(C.c_void_p)


class OracleError(RuntimeError):
    def __init__(self, code):
        super().__init__(f"oracle returned status {code}")
        self.code = code


def half_to_double(bits: int) -> float:
    return lib().awqo_half_to_double(int(bits) & 0xFFFF)


def decode_matrix(q: np.ndarray, meta: np.ndarray, K: int, N: int, group: int = 32) -> np.ndarray:
    """W[K][N] (FP64) from q u32[K/8][N] and meta u8[K/group][N][mb]."""
    q = np.ascontiguousarray(q, np.uint32)
    meta = np.ascontiguousarray(meta, np.uint8)
    mb = meta.shape[-1]
    W = np.empty((K, N), np.float64)
    rc = lib().awqo_decode_matrix(_p(q), _p(meta), mb, K, N, group, _p(W))
    if rc:
        raise OracleError(rc)
    return W


def e2m1_to_double(code: int) -> float:
    return lib().awqo_e2m1_to_double(int(code) & 0xF)


def e4m3_to_double(code: int) -> float:
    return lib().awqo_e4m3_to_double(int(code) & 0xFF)


def decode_nvfp4(q: np.ndarray, scales: np.ndarray, global_scale: float, K: int, N: int) -> np.ndarray:
    """W[K][N] (FP64) of an NVFP4 matrix: q u32[K/8][N] E2M1 codes, scales
    u8[K/16][N] E4M3 codes, one fp32 global scale."""
    q = np.ascontiguousarray(q, np.uint32)
    scales = np.ascontiguousarray(scales, np.uint8)
    W = np.empty((K, N), np.float64)
    rc = lib().awqo_decode_nvfp4(_p(q), _p(scales), float(np.float32(global_scale)), K, N, _p(W))
    if rc:
        raise OracleError(rc)
    return W


def prepare_compact(meta4: np.ndarray) -> np.ndarray:
    meta4 = np.ascontiguousarray(meta4, np.uint8)
    assert meta4.shape[-1] == 4
    n = meta4.size // 4
    out = np.empty(meta4.shape[:-1] + (3,), np.uint8)
    lib().awqo_prepare_compact(_p(meta4), _p(out), n)
    return out


def route(topk_ids: np.ndarray, num_experts: int):
    """(active_ids i32[S], offsets i32[S+1], sorted_slots i32[S], num_active)."""
    ids = np.ascontiguousarray(topk_ids, np.int32)
    M, k = ids.shape
    S = M * k
    act = np.empty(max(S, 1), np.int32)
    off = np.empty(S + 1, np.int32)
    srt = np.empty(max(S, 1), np.int32)
    na = np.zeros(1, np.int32)
    rc = lib().awqo_route(_p(ids), M, k, num_experts, _p(act), _p(off), _p(srt), _p(na))
    if rc:
        raise OracleError(rc)
    return act[:S], off, srt[:S], int(na[0])


def router_topk(logits: np.ndarray, top_k: int):
    """(ids i32[M][k], weights f64[M][k]): softmax of the fp32 logits, the top_k
    experts by probability (ties to the lower id), renormalised over them."""
    lg = np.ascontiguousarray(logits, np.float32)
    M, E = lg.shape
    ids = np.empty((M, top_k), np.int32)
    w = np.empty((M, top_k), np.float64)
    rc = lib().awqo_router_topk(_p(lg), M, E, top_k, _p(ids), _p(w))
    if rc:
        raise OracleError(rc)
    return ids, w


def _expert_ptrs(bank, num_experts):
    """Per-expert pointer array from either a dense [E][...] array or a dict
    {expert: array}; returns (ctypes array, keep-alive list)."""
    arr = (C.c_void_p * num_experts)()
    keep = []
    if isinstance(bank, dict):
        for e, a in bank.items():
            a = np.ascontiguousarray(a)
            keep.append(a)
            arr[int(e)] = a.ctypes.data
    else:
        bank = np.ascontiguousarray(bank)
        keep.append(bank)
        step = bank[0].nbytes
        base = bank.ctypes.data
        for e in range(num_experts):
            arr[e] = base + e * step
    return arr, keep


def _shape_args(shape):
    return (shape.num_experts, shape.hidden, shape.inter, shape.group)


def w13_swiglu(x, topk_ids, shape, w13_q, w13_meta, meta_bytes):
    x = np.ascontiguousarray(x, np.float16).view(np.uint16)
    ids = np.ascontiguousarray(topk_ids, np.int32)
    M, k = ids.shape
    E, H, I, G = _shape_args(shape)
    qa, k1 = _expert_ptrs(w13_q, E)
    ma, k2 = _expert_ptrs(w13_meta, E)
    h = np.zeros((M * k, I), np.float64)
    rc = lib().awqo_w13_swiglu(_p(x), _p(ids), M, k, E, H, I, G, meta_bytes,
                               C.cast(qa, C.c_void_p), C.cast(ma, C.c_void_p), _p(h))
    if rc:
        raise OracleError(rc)
    return h


def w2_reduce(h_slot, topk_ids, topk_weights, shape, w2_q, w2_meta, meta_bytes):
    h_slot = np.ascontiguousarray(h_slot, np.float64)
    ids = np.ascontiguousarray(topk_ids, np.int32)
    w = np.ascontiguousarray(topk_weights, np.float32)
    M, k = ids.shape
    E, H, I, G = _shape_args(shape)
    qa, k1 = _expert_ptrs(w2_q, E)
    ma, k2 = _expert_ptrs(w2_meta, E)
    out = np.zeros((M, H), np.float64)
    rc = lib().awqo_w2_reduce(_p(h_slot), _p(ids), _p(w), M, k, E, H, I, G, meta_bytes,
                              C.cast(qa, C.c_void_p), C.cast(ma, C.c_void_p), _p(out))
    if rc:
        raise OracleError(rc)
    return out


def moe_layer(x, topk_ids, topk_weights, shape, w13_q, w13_meta, w2_q, w2_meta, meta_bytes):
    """(out f64[M][H], h_slot f64[M*k][I]) of one layer call."""
    x = np.ascontiguousarray(x, np.float16).view(np.uint16)
    ids = np.ascontiguousarray(topk_ids, np.int32)
    w = np.ascontiguousarray(topk_weights, np.float32)
    M, k = ids.shape
    E, H, I, G = _shape_args(shape)
    a1, k1 = _expert_ptrs(w13_q, E)
    a2, k2 = _expert_ptrs(w13_meta, E)
    a3, k3 = _expert_ptrs(w2_q, E)
    a4, k4 = _expert_ptrs(w2_meta, E)
    h = np.zeros((M * k, I), np.float64)
    out = np.zeros((M, H), np.float64)
    rc = lib().awqo_moe_layer(_p(x), _p(ids), _p(w), M, k, E, H, I, G, meta_bytes,
                              C.cast(a1, C.c_void_p), C.cast(a2, C.c_void_p),
                              C.cast(a3, C.c_void_p), C.cast(a4, C.c_void_p), _p(h), _p(out))
    if rc:
        raise OracleError(rc)
    return out, h


def moe_layer_nvfp4(x, topk_ids, topk_weights, shape, w13_q, w13_scales, w2_q, w2_scales, global_scale):
    """(out f64[M][H], h_slot f64[M*k][I]) of one layer call with NVFP4 weights;
    global_scale f32[E][2] (W13, W2)."""
    x = np.ascontiguousarray(x, np.float16).view(np.uint16)
    ids = np.ascontiguousarray(topk_ids, np.int32)
    w = np.ascontiguousarray(topk_weights, np.float32)
    g = np.ascontiguousarray(global_scale, np.float32)
    M, k = ids.shape
    E, H, I = shape.num_experts, shape.hidden, shape.inter
    a1, k1 = _expert_ptrs(w13_q, E)
    a2, k2 = _expert_ptrs(w13_scales, E)
    a3, k3 = _expert_ptrs(w2_q, E)
    a4, k4 = _expert_ptrs(w2_scales, E)
    h = np.zeros((M * k, I), np.float64)
    out = np.zeros((M, H), np.float64)
    rc = lib().awqo_moe_layer_nvfp4(_p(x), _p(ids), _p(w), M, k, E, H, I, C.cast(a1, C.c_void_p),
                                    C.cast(a2, C.c_void_p), C.cast(a3, C.c_void_p), C.cast(a4, C.c_void_p),
                                    _p(g), _p(h), _p(out))
    if rc:
        raise OracleError(rc)
    return out, h


def layer_from_synth(shape, seed, layer, x, topk_ids, topk_weights, meta_bytes=None):
    """Oracle output of one synthetic layer: regenerates only the active
    experts' banks from the seeded generator in ``synth``."""
    import synth
    mb = shape.meta_bytes if meta_bytes is None else meta_bytes
    experts = sorted(set(int(e) for e in np.asarray(topk_ids).ravel()))
    b1, b2, b3, b4 = {}, {}, {}, {}
    for e in experts:
        b1[e], b2[e], b3[e], b4[e] = synth.expert_weights(shape, seed, layer, e, mb)
    if shape.group == 16:       # NVFP4 banks: block-scale codes u8[K/16][N] and the globals
        for d in (b2, b4):
            for e in d:
                d[e] = d[e][..., 0]
        g = synth.nvfp4_global(seed, layer, shape.num_experts)
        return moe_layer_nvfp4(x, topk_ids, topk_weights, shape, b1, b2, b3, b4, g)
    return moe_layer(x, topk_ids, topk_weights, shape, b1, b2, b3, b4, mb)
