"""Python binding of the GB300 AWQ int4 MoE expert-stage library.

Thin marshalling layer over the C ABI in ``include/awq_moe.h``: every
function here has the same name as its C entry point (without the ``awq_``
prefix), passes ``tensor.data_ptr()`` and the current CUDA stream through
ctypes, and raises :class:`AwqError` on a non-zero status. All computation
runs in the CUDA library ``libawqmoe.so``; there is no CPU path and no
fallback. Importing this package does not need a GPU, but the library must
have been built (``awq_int4_moe_gb300.build.build()``).
"""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libawqmoe.so")

MAX_TOKENS = 512
W2_STAGE_MAX_TOKENS = 128
TRACE_POINTS = 16                # AWQ_TRACE_POINTS
STATIC_SCRATCH_BYTES = 2 << 20   # AWQ_STATIC_SCRATCH_BYTES

# awq_status
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED_SHAPE, ERR_MISALIGNED, ERR_CUDA = 0, 1, 2, 3, 4
ERR_DEVICE_TIMEOUT, ERR_BAD_EXPERT_ID, ERR_WORKSPACE_TOO_SMALL, ERR_LAYOUT = 5, 6, 7, 8

# awq_layout
LAYOUT_CANONICAL, LAYOUT_PREPARED = 0, 1


class AwqError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {status_string(code)} (status {code})")
        self.code = code


class Shape(C.Structure):
    _fields_ = [("num_experts", C.c_int32), ("top_k", C.c_int32), ("hidden", C.c_int32),
                ("inter", C.c_int32), ("group", C.c_int32), ("meta_bytes", C.c_int32)]

    @classmethod
    def of(cls, s) -> "Shape":
        """From any object with the six attributes (e.g. synth.ExpertShape)."""
        if isinstance(s, Shape):
            return s
        return cls(s.num_experts, s.top_k, s.hidden, s.inter, s.group, s.meta_bytes)


PATH_AUTO, PATH_FUSED, PATH_STAGED, PATH_SLICED, PATH_PREFILL, PATH_HYBRID = 0, 1, 2, 3, 4, 5


class Options(C.Structure):
    _fields_ = [("timeout_ns", C.c_uint64), ("path", C.c_int32), ("debug_flags", C.c_int32),
                ("trace", C.c_void_p)]


class Weights(C.Structure):
    _fields_ = [("w13_q", C.c_void_p), ("w13_meta", C.c_void_p), ("w2_q", C.c_void_p),
                ("w2_meta", C.c_void_p), ("layout", C.c_int32), ("global_scale", C.c_void_p)]

    @classmethod
    def of(cls, w13_q, w13_meta, w2_q, w2_meta, layout: int = LAYOUT_CANONICAL,
           global_scale=None) -> "Weights":
        """Bank pointers; ``global_scale`` (NVFP4 only) is f32[E][2] on the device."""
        for name, t in (("w13_q", w13_q), ("w13_meta", w13_meta), ("w2_q", w2_q), ("w2_meta", w2_meta),
                        ("global_scale", global_scale)):
            if t is not None and not isinstance(t, int) and not t.is_cuda:
                raise ValueError(f"{name}: must be a CUDA device tensor, got one on {t.device}")
        if global_scale is not None and not isinstance(global_scale, int) and \
                str(global_scale.dtype) != "torch.float32":
            raise TypeError(f"global_scale: expected float32, got {global_scale.dtype}")
        return cls(_ptr(w13_q), _ptr(w13_meta), _ptr(w2_q), _ptr(w2_meta), int(layout), _ptr(global_scale))


_lib = None


def lib() -> C.CDLL:
    """The loaded CUDA library. Raises if it has not been built: there is no
    other implementation to fall back to."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library {LIB_PATH} is missing; build it with "
                               "awq_int4_moe_gb300.build.build()")
        L = C.CDLL(LIB_PATH)
        P, i32, i64 = C.c_void_p, C.c_int32, C.c_int64
        SP, WP = C.POINTER(Shape), C.POINTER(Weights)
        L.awq_status_string.restype = C.c_char_p
        L.awq_status_string.argtypes = [C.c_int]
        L.awq_moe_workspace_bytes.restype = C.c_size_t
        L.awq_moe_workspace_bytes.argtypes = [SP, i32]
        L.awq_moe_prepare_weights.restype = C.c_int
        L.awq_moe_prepare_weights.argtypes = [SP, WP, WP, P]
        L.awq_prepare_compact.restype = C.c_int
        L.awq_prepare_compact.argtypes = [P, P, i64, P]
        L.awq_moe_route.restype = C.c_int
        L.awq_moe_route.argtypes = [P, i32, SP, P, P, P, P, P, P]
        L.awq_moe_w13_swiglu.restype = C.c_int
        L.awq_moe_w13_swiglu.argtypes = [P, i32, SP, WP, P, P, P, P, P, P, P]
        L.awq_moe_w2_reduce.restype = C.c_int
        L.awq_moe_w2_reduce.argtypes = [P, P, i32, SP, WP, P, P, P, P, P, P, P]
        L.awq_moe_layer.restype = C.c_int
        L.awq_moe_layer.argtypes = [P, P, P, i32, SP, WP, P, P, C.c_size_t, P, P]
        L.awq_moe_layer_ex.restype = C.c_int
        L.awq_moe_layer_ex.argtypes = [P, P, P, i32, SP, WP, P, P, C.c_size_t, P,
                                       C.POINTER(Options), P]
        L.awq_moe_router_topk.restype = C.c_int
        L.awq_moe_router_topk.argtypes = [P, i32, SP, P, P, P]
        L.awq_moe_layer_logits.restype = C.c_int
        L.awq_moe_layer_logits.argtypes = [P, P, i32, SP, WP, P, P, P, P, C.c_size_t, P,
                                           C.POINTER(Options), P]
        L.awq_moe_layer_static.restype = C.c_int
        L.awq_moe_layer_static.argtypes = [P, P, P, i32, SP, WP, P, P, P]
        L.awq_moe_latency_floor.restype = C.c_int
        L.awq_moe_latency_floor.argtypes = [P, i32, SP, WP, P, P, C.c_size_t, P, P]
        _lib = L
    return _lib


def _ptr(t):
    """Address of a buffer: a tensor (which must be contiguous: every array of
    the C ABI is dense and row-major), a raw integer address, or None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("the C ABI takes dense row-major arrays; got a non-contiguous tensor "
                         f"of shape {tuple(t.shape)} and strides {tuple(t.stride())}")
    return t.data_ptr()


# Element kinds of the C ABI's arrays and the torch dtypes that carry them
# (fp16 values travel as 16-bit patterns, so int16/uint16 views are accepted).
_KINDS = {"f16": ("float16", "int16", "uint16"), "i32": ("int32",), "f32": ("float32",)}


_DTYPE_NAMES = {}


def _dtype_name(dtype):
    """"float16" for torch.float16 and so on (memoised: this runs on every call)."""
    name = _DTYPE_NAMES.get(dtype)
    if name is None:
        name = _DTYPE_NAMES[dtype] = str(dtype).replace("torch.", "")
    return name


def _checked(**specs):
    """Addresses of a call's buffers after checking what the C call cannot
    see: each spec is (tensor, kind, count) with kind an element type of
    _KINDS or "bytes" for untyped buffers, and count the least number of
    elements (bytes) the call reads or writes. Every buffer's element type and
    size are checked first, then that every one lives on a CUDA device. A raw
    integer address or None passes unchecked (the C call still checks null
    pointers and alignment)."""
    for name, (t, kind, count) in specs.items():
        if t is None or isinstance(t, int):
            continue
        dt = _dtype_name(t.dtype)
        if kind == "bytes":
            n = t.numel() * t.element_size()
        else:
            if dt not in _KINDS[kind]:
                raise TypeError(f"{name}: expected {kind} elements ({' / '.join(_KINDS[kind])}), got {dt}")
            n = t.numel()
        if n < count:
            unit = "bytes" if kind == "bytes" else "elements"
            raise ValueError(f"{name}: holds {n} {unit}; the call needs at least {count}")
    for name, (t, _, _) in specs.items():
        if t is not None and not isinstance(t, int) and not t.is_cuda:
            raise ValueError(f"{name}: must be a CUDA device tensor, got one on {t.device}")
    return {name: _ptr(t) for name, (t, _, _) in specs.items()}


def _dims(shape, M):
    s = Shape.of(shape)
    return s, int(M), int(M) * s.top_k


def _stream(stream):
    if stream is None:
        import torch
        return C.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return C.c_void_p(stream)
    return C.c_void_p(stream.cuda_stream)


def _check(code: int, where: str):
    if code != OK:
        raise AwqError(code, where)


def status_string(code: int) -> str:
    return lib().awq_status_string(int(code)).decode()


def moe_workspace_bytes(shape, M_max: int) -> int:
    return int(lib().awq_moe_workspace_bytes(C.byref(Shape.of(shape)), int(M_max)))


def moe_prepare_weights(shape, src: Weights, dst: Weights, stream=None) -> Weights:
    """Permute canonical banks ``src`` into the caller's buffers ``dst``;
    ``dst.layout`` becomes LAYOUT_PREPARED. Returns ``dst``."""
    _check(lib().awq_moe_prepare_weights(C.byref(Shape.of(shape)), C.byref(src), C.byref(dst),
                                         _stream(stream)), "awq_moe_prepare_weights")
    return dst


def prepare_compact(meta4, meta3, n_records: int, stream=None):
    n = int(n_records)
    a = _checked(meta4=(meta4, "bytes", 4 * n), meta3=(meta3, "bytes", 3 * n))
    _check(lib().awq_prepare_compact(a["meta4"], a["meta3"], n, _stream(stream)), "awq_prepare_compact")


def _route_specs(S, active_expert_ids, active_expert_offsets, sorted_slots, num_active):
    return dict(active_expert_ids=(active_expert_ids, "i32", S),
                active_expert_offsets=(active_expert_offsets, "i32", S + 1),
                sorted_slots=(sorted_slots, "i32", S), num_active=(num_active, "i32", 1))


def moe_route(topk_ids, M: int, shape, active_expert_ids, active_expert_offsets, sorted_slots,
              num_active, dev_status, stream=None):
    s, M, S = _dims(shape, M)
    a = _checked(topk_ids=(topk_ids, "i32", S), dev_status=(dev_status, "i32", 1),
                 **_route_specs(S, active_expert_ids, active_expert_offsets, sorted_slots, num_active))
    _check(lib().awq_moe_route(a["topk_ids"], M, C.byref(s), a["active_expert_ids"], a["active_expert_offsets"],
                               a["sorted_slots"], a["num_active"], a["dev_status"], _stream(stream)),
           "awq_moe_route")


def moe_w13_swiglu(x, M: int, shape, weights: Weights, active_expert_ids, active_expert_offsets,
                   sorted_slots, num_active, h, dev_status, stream=None):
    s, M, S = _dims(shape, M)
    a = _checked(x=(x, "f16", M * s.hidden), h=(h, "f16", S * s.inter), dev_status=(dev_status, "i32", 1),
                 **_route_specs(S, active_expert_ids, active_expert_offsets, sorted_slots, num_active))
    _check(lib().awq_moe_w13_swiglu(a["x"], M, C.byref(s), C.byref(weights), a["active_expert_ids"],
                                    a["active_expert_offsets"], a["sorted_slots"], a["num_active"], a["h"],
                                    a["dev_status"], _stream(stream)), "awq_moe_w13_swiglu")


def moe_w2_reduce(h, topk_weights, M: int, shape, weights: Weights, active_expert_ids,
                  active_expert_offsets, sorted_slots, num_active, out, dev_status, stream=None):
    s, M, S = _dims(shape, M)
    a = _checked(h=(h, "f16", S * s.inter), topk_weights=(topk_weights, "f32", S),
                 out=(out, "f16", M * s.hidden), dev_status=(dev_status, "i32", 1),
                 **_route_specs(S, active_expert_ids, active_expert_offsets, sorted_slots, num_active))
    _check(lib().awq_moe_w2_reduce(a["h"], a["topk_weights"], M, C.byref(s), C.byref(weights),
                                   a["active_expert_ids"], a["active_expert_offsets"], a["sorted_slots"],
                                   a["num_active"], a["out"], a["dev_status"], _stream(stream)),
           "awq_moe_w2_reduce")


def _layer_specs(s, M, S, x, topk_ids, topk_weights, out, dev_status, **more):
    return _checked(x=(x, "f16", M * s.hidden), topk_ids=(topk_ids, "i32", S),
                    topk_weights=(topk_weights, "f32", S), out=(out, "f16", M * s.hidden),
                    dev_status=(dev_status, "i32", 1), **more)


def moe_layer(x, topk_ids, topk_weights, M: int, shape, weights: Weights, out, workspace,
              ws_bytes: int, dev_status, stream=None):
    s, M, S = _dims(shape, M)
    a = _layer_specs(s, M, S, x, topk_ids, topk_weights, out, dev_status,
                     workspace=(workspace, "bytes", int(ws_bytes)))
    _check(lib().awq_moe_layer(a["x"], a["topk_ids"], a["topk_weights"], M, C.byref(s), C.byref(weights),
                               a["out"], a["workspace"], int(ws_bytes), a["dev_status"], _stream(stream)),
           "awq_moe_layer")


def moe_layer_ex(x, topk_ids, topk_weights, M: int, shape, weights: Weights, out, workspace,
                 ws_bytes: int, dev_status, path: int = PATH_AUTO, timeout_ns: int = 0,
                 debug_flags: int = 0, trace=None, stream=None):
    s, M, S = _dims(shape, M)
    a = _layer_specs(s, M, S, x, topk_ids, topk_weights, out, dev_status,
                     workspace=(workspace, "bytes", int(ws_bytes)))
    opts = Options(int(timeout_ns), int(path), int(debug_flags), _ptr(trace))
    _check(lib().awq_moe_layer_ex(a["x"], a["topk_ids"], a["topk_weights"], M, C.byref(s), C.byref(weights),
                                  a["out"], a["workspace"], int(ws_bytes), a["dev_status"], C.byref(opts),
                                  _stream(stream)), "awq_moe_layer_ex")


def moe_router_topk(logits, M: int, shape, topk_ids, topk_weights, stream=None):
    """awq_moe_router_topk: top-k experts and renormalised weights from logits."""
    s, M, S = _dims(shape, M)
    a = _checked(logits=(logits, "f32", M * s.num_experts), topk_ids=(topk_ids, "i32", S),
                 topk_weights=(topk_weights, "f32", S))
    _check(lib().awq_moe_router_topk(a["logits"], M, C.byref(s), a["topk_ids"], a["topk_weights"],
                                     _stream(stream)), "awq_moe_router_topk")


def moe_layer_logits(x, logits, M: int, shape, weights: Weights, out, topk_ids, topk_weights,
                     workspace, ws_bytes: int, dev_status, path: int = PATH_AUTO,
                     timeout_ns: int = 0, stream=None):
    """awq_moe_layer_logits: router from logits, then the expert stage."""
    s, M, S = _dims(shape, M)
    a = _layer_specs(s, M, S, x, topk_ids, topk_weights, out, dev_status,
                     workspace=(workspace, "bytes", int(ws_bytes)),
                     logits=(logits, "f32", M * s.num_experts))
    opts = Options(int(timeout_ns), int(path), 0)
    _check(lib().awq_moe_layer_logits(a["x"], a["logits"], M, C.byref(s), C.byref(weights), a["out"],
                                      a["topk_ids"], a["topk_weights"], a["workspace"], int(ws_bytes),
                                      a["dev_status"], C.byref(opts), _stream(stream)), "awq_moe_layer_logits")


def moe_layer_static(x, topk_ids, topk_weights, M: int, shape, weights: Weights, out, dev_status,
                     stream=None):
    """awq_moe_layer on the library's fixed device scratch (no workspace)."""
    s, M, S = _dims(shape, M)
    a = _layer_specs(s, M, S, x, topk_ids, topk_weights, out, dev_status)
    _check(lib().awq_moe_layer_static(a["x"], a["topk_ids"], a["topk_weights"], M, C.byref(s), C.byref(weights),
                                      a["out"], a["dev_status"], _stream(stream)), "awq_moe_layer_static")


def moe_latency_floor(topk_ids, M: int, shape, weights: Weights, out, workspace, ws_bytes: int,
                      dev_status, stream=None):
    """awq_moe_latency_floor: the persistent layer call's dependency chain
    (ids, one read of the active experts' banks, a grid barrier, the output
    write) with no arithmetic; a measurement helper that writes zeros."""
    s, M, S = _dims(shape, M)
    a = _checked(topk_ids=(topk_ids, "i32", S), out=(out, "f16", M * s.hidden),
                 workspace=(workspace, "bytes", int(ws_bytes)), dev_status=(dev_status, "i32", 1))
    _check(lib().awq_moe_latency_floor(a["topk_ids"], M, C.byref(s), C.byref(weights), a["out"], a["workspace"],
                                       int(ws_bytes), a["dev_status"], _stream(stream)), "awq_moe_latency_floor")
