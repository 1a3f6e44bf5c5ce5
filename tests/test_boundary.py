"""The C ABI without a GPU: the library loads, exports every symbol the
header declares, and rejects host-visible errors synchronously (these paths
return before any CUDA call, so they run on a GPU-less host)."""
import ctypes as C
import os
import re

import pytest

import awq_int4_moe_gb300 as awq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "awq_moe.h")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import awq_int4_moe_gb300.build as b
    b.build()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"AWQ_API\s+[\w\s\*]*?\b(awq_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert {"awq_prepare_compact", "awq_moe_prepare_weights", "awq_moe_route", "awq_moe_w13_swiglu", "awq_moe_w2_reduce",
            "awq_moe_layer"} <= set(names)
    L = awq.lib()
    for n in names:
        assert hasattr(L, n), n


def test_status_strings():
    for code in range(9):
        s = awq.status_string(code)
        assert s and s != "unknown status"
    assert awq.status_string(99) == "unknown status"


SHAPE = awq.Shape(512, 10, 2560, 160, 32, 4)
FAKE = 0x10000000  # a 256-byte aligned non-null address; never dereferenced on these paths


def weights(**over):
    w = dict(w13_q=FAKE, w13_meta=FAKE, w2_q=FAKE, w2_meta=FAKE, layout=awq.LAYOUT_PREPARED)
    w.update(over)
    return awq.Weights(**w)


def call_layer(M=1, shape=SHAPE, w=None, ws_bytes=1 << 20, **ptr):
    p = dict(x=FAKE, ids=FAKE, wts=FAKE, out=FAKE, ws=FAKE, st=FAKE)
    p.update(ptr)
    return awq.lib().awq_moe_layer(p["x"], p["ids"], p["wts"], M, C.byref(shape),
                                   C.byref(w or weights()), p["out"], p["ws"], ws_bytes, p["st"],
                                   None)


def test_workspace_bytes():
    assert awq.moe_workspace_bytes(SHAPE, 0) == 0
    assert awq.moe_workspace_bytes(SHAPE, awq.MAX_TOKENS + 1) == 0
    b1, b8 = awq.moe_workspace_bytes(SHAPE, 1), awq.moe_workspace_bytes(SHAPE, 8)
    assert 0 < b1 <= b8 and b8 % 256 == 0
    assert b8 >= 8 * 10 * 160 * 2 + 4 * (3 * 80 + 2)
    bad = awq.Shape(512, 10, 2560, 161, 32, 4)
    assert awq.moe_workspace_bytes(bad, 8) == 0


@pytest.mark.parametrize("inter,mb", [(160, 4), (640, 3)])
def test_workspace_for_m_max_serves_every_smaller_call(inter, mb):
    # a workspace sized for M_max must hold the need of every call with M <= M_max;
    # calls of up to 16 tokens take the fused path, whose partial blocks are
    # larger than the three launches' arrays of a bigger M
    shape = awq.Shape(512, 10, 2560, inter, 32, mb)
    sizes = [awq.moe_workspace_bytes(shape, m) for m in range(1, awq.MAX_TOKENS + 1)]
    assert all(b > 0 and b % 256 == 0 for b in sizes)
    assert all(a <= b for a, b in zip(sizes, sizes[1:]))          # non-decreasing in M_max
    assert sizes[awq.MAX_TOKENS - 1] >= sizes[15] > 8 * 1024 * 1024


@pytest.mark.parametrize("field,value", [("num_experts", 0), ("num_experts", 1025), ("top_k", 0),
                                         ("top_k", 17), ("hidden", 4096), ("inter", 320),
                                         ("group", 64), ("meta_bytes", 2)])
def test_unsupported_shapes_rejected(field, value):
    s = awq.Shape(512, 10, 2560, 160, 32, 4)
    setattr(s, field, value)
    assert call_layer(shape=s) == awq.ERR_UNSUPPORTED_SHAPE


def test_token_count_limits():
    assert call_layer(M=-1) == awq.ERR_INVALID_ARG
    assert call_layer(M=awq.MAX_TOKENS + 1) == awq.ERR_INVALID_ARG
    assert call_layer(M=0) == awq.OK          # empty batch: nothing to do, nothing launched


@pytest.mark.parametrize("name", ["x", "ids", "wts", "out", "ws", "st"])
def test_null_pointers_rejected(name):
    assert call_layer(**{name: None}) == awq.ERR_INVALID_ARG


@pytest.mark.parametrize("field", ["w13_q", "w13_meta", "w2_q", "w2_meta"])
def test_null_and_misaligned_weights(field):
    assert call_layer(w=weights(**{field: None})) == awq.ERR_INVALID_ARG
    assert call_layer(w=weights(**{field: FAKE + 8})) == awq.ERR_MISALIGNED


def test_misaligned_activations_and_workspace():
    assert call_layer(x=FAKE + 2) == awq.ERR_MISALIGNED
    assert call_layer(out=FAKE + 4) == awq.ERR_MISALIGNED
    assert call_layer(ws=FAKE + 16) == awq.ERR_MISALIGNED


def test_workspace_too_small():
    need = awq.moe_workspace_bytes(SHAPE, 4)
    assert call_layer(M=4, ws_bytes=need - 1) == awq.ERR_WORKSPACE_TOO_SMALL


def test_stage_entry_points_validate():
    L = awq.lib()
    w = weights()
    assert L.awq_moe_route(FAKE, 1, None, FAKE, FAKE, FAKE, FAKE, FAKE, None) == awq.ERR_INVALID_ARG
    assert L.awq_moe_route(FAKE, 1, C.byref(SHAPE), FAKE, None, FAKE, FAKE, FAKE, None) == \
        awq.ERR_INVALID_ARG
    assert L.awq_moe_w13_swiglu(FAKE + 2, 1, C.byref(SHAPE), C.byref(w), FAKE, FAKE, FAKE, FAKE,
                                FAKE, FAKE, None) == awq.ERR_MISALIGNED
    assert L.awq_moe_w13_swiglu(FAKE, 1, C.byref(SHAPE), C.byref(w), FAKE, FAKE, FAKE, FAKE,
                                None, FAKE, None) == awq.ERR_INVALID_ARG
    assert L.awq_moe_w2_reduce(FAKE, FAKE, 1, C.byref(SHAPE), C.byref(w), FAKE, FAKE, FAKE, FAKE,
                               FAKE + 8, FAKE, None) == awq.ERR_MISALIGNED
    assert L.awq_moe_w2_reduce(FAKE, FAKE, awq.MAX_TOKENS + 1, C.byref(SHAPE), C.byref(w), FAKE, FAKE,
                               FAKE, FAKE, FAKE, FAKE, None) == awq.ERR_INVALID_ARG
    # the W2 stage call keeps every token's output tile in shared memory: larger
    # batches are refused before anything is launched (the layer call takes them)
    assert L.awq_moe_w2_reduce(FAKE, FAKE, awq.W2_STAGE_MAX_TOKENS + 1, C.byref(SHAPE), C.byref(w), FAKE,
                               FAKE, FAKE, FAKE, FAKE, FAKE, None) == awq.ERR_UNSUPPORTED_SHAPE


def test_prepare_compact_validation():
    L = awq.lib()
    assert L.awq_prepare_compact(FAKE, FAKE + 4096, -1, None) == awq.ERR_INVALID_ARG
    assert L.awq_prepare_compact(FAKE, FAKE + 4096, 0, None) == awq.OK
    assert L.awq_prepare_compact(None, FAKE, 4, None) == awq.ERR_INVALID_ARG
    assert L.awq_prepare_compact(FAKE, FAKE + 8, 4, None) == awq.ERR_INVALID_ARG   # overlap


def test_compute_calls_need_prepared_banks():
    canon = weights(layout=awq.LAYOUT_CANONICAL)
    assert call_layer(w=canon) == awq.ERR_LAYOUT
    L = awq.lib()
    assert L.awq_moe_w13_swiglu(FAKE, 1, C.byref(SHAPE), C.byref(canon), FAKE, FAKE, FAKE, FAKE,
                                FAKE, FAKE, None) == awq.ERR_LAYOUT
    assert L.awq_moe_w2_reduce(FAKE, FAKE, 1, C.byref(SHAPE), C.byref(canon), FAKE, FAKE, FAKE,
                               FAKE, FAKE, FAKE, None) == awq.ERR_LAYOUT


def test_prepare_weights_validation():
    L = awq.lib()
    E, H, I, mb = SHAPE.num_experts, SHAPE.hidden, SHAPE.inter, SHAPE.meta_bytes
    big = E * H // 8 * 2 * I * 4            # largest bank, bytes
    src = weights(layout=awq.LAYOUT_CANONICAL)
    base = FAKE + 4 * big                    # a disjoint fake region
    dst = weights(w13_q=base, w13_meta=base + big, w2_q=base + 2 * big, w2_meta=base + 3 * big)

    def prep(shape=SHAPE, s=src, d=dst):
        return L.awq_moe_prepare_weights(C.byref(shape) if shape is not None else None,
                                         C.byref(s) if s is not None else None,
                                         C.byref(d) if d is not None else None, None)

    assert prep(shape=None) == awq.ERR_INVALID_ARG
    assert prep(shape=awq.Shape(512, 10, 2560, 161, 32, 4)) == awq.ERR_UNSUPPORTED_SHAPE
    assert prep(s=None) == awq.ERR_INVALID_ARG
    assert prep(d=None) == awq.ERR_INVALID_ARG
    assert prep(s=weights(layout=awq.LAYOUT_PREPARED)) == awq.ERR_LAYOUT
    assert prep(d=weights(w13_q=base + 8, w13_meta=base + big, w2_q=base + 2 * big,
                          w2_meta=base + 3 * big)) == awq.ERR_MISALIGNED
    assert prep(d=weights(w13_q=None, w13_meta=base + big, w2_q=base + 2 * big,
                          w2_meta=base + 3 * big)) == awq.ERR_INVALID_ARG
    # a destination bank overlapping a source bank is refused
    assert prep(d=weights(w13_q=FAKE + 256, w13_meta=base + big, w2_q=base + 2 * big,
                          w2_meta=base + 3 * big)) == awq.ERR_INVALID_ARG
    assert dst.layout == awq.LAYOUT_PREPARED and src.layout == awq.LAYOUT_CANONICAL


def test_static_layer_rejects_calls_beyond_its_scratch():
    L = awq.lib()
    big = awq.Shape(512, 16, 2560, 640, 32, 4)
    # 128 tokens x top-16 x inter 640 needs more than the fixed scratch holds
    assert L.awq_moe_layer_static(FAKE, FAKE, FAKE, 128, C.byref(big), C.byref(weights()), FAKE, FAKE,
                                  None) == awq.ERR_WORKSPACE_TOO_SMALL
    assert L.awq_moe_layer_static(FAKE, FAKE, FAKE, 0, C.byref(big), C.byref(weights()), FAKE, FAKE,
                                  None) == awq.OK
    # beyond the W2 stage kernel's token limit (fits the scratch at inter 160, top-1)
    one = awq.Shape(512, 1, 2560, 160, 32, 4)
    assert L.awq_moe_layer_static(FAKE, FAKE, FAKE, awq.W2_STAGE_MAX_TOKENS + 1, C.byref(one),
                                  C.byref(weights()), FAKE, FAKE, None) == awq.ERR_UNSUPPORTED_SHAPE
    assert L.awq_moe_layer_static(None, FAKE, FAKE, 2, C.byref(SHAPE), C.byref(weights()), FAKE, FAKE,
                                  None) == awq.ERR_INVALID_ARG
    assert L.awq_moe_layer_static(FAKE, FAKE, FAKE, 2, C.byref(SHAPE),
                                  C.byref(weights(layout=awq.LAYOUT_CANONICAL)), FAKE, FAKE,
                                  None) == awq.ERR_LAYOUT


def test_latency_floor_validates():
    L = awq.lib()
    S = C.byref(SHAPE)

    def floor(M=2, shape=S, w=None, ids=FAKE, out=FAKE, ws=FAKE, ws_bytes=1 << 20, st=FAKE):
        return L.awq_moe_latency_floor(ids, M, shape, C.byref(w or weights()), out, ws, ws_bytes, st, None)

    assert floor(M=0) == awq.OK
    assert floor(M=17) == awq.ERR_INVALID_ARG          # a decode-sized helper: 16 tokens at most
    assert floor(M=-1) == awq.ERR_INVALID_ARG
    assert floor(ids=None) == awq.ERR_INVALID_ARG
    assert floor(out=None) == awq.ERR_INVALID_ARG
    assert floor(st=None) == awq.ERR_INVALID_ARG
    assert floor(out=FAKE + 8) == awq.ERR_MISALIGNED
    assert floor(ws=FAKE + 16) == awq.ERR_MISALIGNED
    assert floor(ws_bytes=16) == awq.ERR_WORKSPACE_TOO_SMALL
    assert floor(w=weights(layout=awq.LAYOUT_CANONICAL)) == awq.ERR_LAYOUT
    bad = awq.Shape(512, 10, 2560, 96, 32, 4)
    assert floor(shape=C.byref(bad)) == awq.ERR_UNSUPPORTED_SHAPE


def test_router_entry_points_validate():
    L = awq.lib()
    w = weights()
    S = C.byref(SHAPE)
    assert L.awq_moe_router_topk(None, 1, S, FAKE, FAKE, None) == awq.ERR_INVALID_ARG
    assert L.awq_moe_router_topk(FAKE, 1, S, None, FAKE, None) == awq.ERR_INVALID_ARG
    assert L.awq_moe_router_topk(FAKE + 2, 1, S, FAKE, FAKE, None) == awq.ERR_MISALIGNED
    assert L.awq_moe_router_topk(FAKE, awq.MAX_TOKENS + 1, S, FAKE, FAKE, None) == awq.ERR_INVALID_ARG
    assert L.awq_moe_router_topk(FAKE, 1, None, FAKE, FAKE, None) == awq.ERR_INVALID_ARG
    assert L.awq_moe_router_topk(None, 0, S, None, None, None) == awq.OK
    other = awq.Shape(256, 10, 2560, 160, 32, 4)              # the router is for 512 experts
    assert L.awq_moe_router_topk(FAKE, 1, C.byref(other), FAKE, FAKE, None) == awq.ERR_UNSUPPORTED_SHAPE
    ws = awq.moe_workspace_bytes(SHAPE, 4)
    args = dict(x=FAKE, lg=FAKE, out=FAKE, ids=FAKE, wt=FAKE, ws=FAKE, st=FAKE)

    def call(**kw):
        a = dict(args, **kw)
        return L.awq_moe_layer_logits(a["x"], a["lg"], 4, S, C.byref(w), a["out"], a["ids"], a["wt"],
                                      a["ws"], ws, a["st"], None, None)
    assert call(lg=None) == awq.ERR_INVALID_ARG
    assert call(ids=None) == awq.ERR_INVALID_ARG
    assert call(wt=None) == awq.ERR_INVALID_ARG
    assert call(lg=FAKE + 2) == awq.ERR_MISALIGNED
    other = awq.Shape(256, 10, 2560, 160, 32, 4)
    assert L.awq_moe_layer_logits(FAKE, FAKE, 4, C.byref(other), C.byref(w), FAKE, FAKE, FAKE, FAKE, ws, FAKE,
                                  None, None) == awq.ERR_UNSUPPORTED_SHAPE
    assert call(x=FAKE + 8) == awq.ERR_MISALIGNED


def test_header_is_plain_c_and_links(tmp_path):
    """The header compiles as ISO C99 with every warning an error, and a plain C
    program that takes the address of every declared call links against the
    library (C linkage, no name mangling)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    names = declared_functions()
    src = tmp_path / "abi.c"
    src.write_text('#include "awq_moe.h"\n#include <stdio.h>\n'
                   "typedef void (*any_fn)(void);\n"
                   "static any_fn calls[] = {\n" + "".join(f"    (any_fn){n},\n" for n in names) + "};\n"
                   'int main(void) { printf("%d\\n", (int)(sizeof calls / sizeof calls[0])); return 0; }\n')
    lib_dir = os.path.dirname(awq.LIB_PATH)
    exe = str(tmp_path / "abi")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                        str(src), "-o", exe, "-L", lib_dir, "-lawqmoe", "-Wl,-rpath," + lib_dir,
                        "-Wl,--unresolved-symbols=ignore-in-shared-libs"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_binding_rejects_non_contiguous_tensors():
    import torch
    x = torch.zeros((4, 2560), dtype=torch.int16)
    with pytest.raises(ValueError):
        awq._ptr(x.t())                        # a transposed view: not row-major
    with pytest.raises(ValueError):
        awq._ptr(x[:, ::2])                    # a strided slice
    assert awq._ptr(x[1:3]) == x[1:3].data_ptr()   # row slices stay dense
    assert awq._ptr(12345) == 12345 and awq._ptr(None) is None


def test_binding_rejects_wrong_dtypes_short_buffers_and_host_tensors():
    """The Python wrappers check what the C call cannot see -- element type,
    element count against M / top_k / hidden, and the device -- before any
    address reaches the library (a wrong buffer would otherwise be read or
    written out of bounds on the GPU)."""
    import torch
    M, H, k = 2, SHAPE.hidden, SHAPE.top_k
    w = awq.Weights(FAKE, FAKE, FAKE, FAKE, awq.LAYOUT_PREPARED)
    good = dict(x=torch.zeros((M, H), dtype=torch.float16), ids=torch.zeros((M, k), dtype=torch.int32),
                wts=torch.zeros((M, k), dtype=torch.float32), out=torch.zeros((M, H), dtype=torch.int16),
                st=torch.zeros(1, dtype=torch.int32))
    ws_bytes = awq.moe_workspace_bytes(SHAPE, M)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8)

    def call(**over):
        a = dict(good, **over)
        awq.moe_layer(a["x"], a["ids"], a["wts"], M, SHAPE, w, a["out"], a.get("ws", ws), ws_bytes, a["st"])

    with pytest.raises(TypeError, match="x: expected f16"):
        call(x=torch.zeros((M, H), dtype=torch.float32))
    with pytest.raises(TypeError, match="topk_ids: expected i32"):
        call(ids=torch.zeros((M, k), dtype=torch.int64))
    with pytest.raises(TypeError, match="topk_weights: expected f32"):
        call(wts=torch.zeros((M, k), dtype=torch.float64))
    with pytest.raises(ValueError, match="out: holds"):
        call(out=torch.zeros((M, H - 1), dtype=torch.int16))
    with pytest.raises(ValueError, match="topk_ids: holds"):
        call(ids=torch.zeros((M, k - 1), dtype=torch.int32))
    with pytest.raises(ValueError, match="workspace: holds"):
        call(ws=torch.zeros(ws_bytes - 1, dtype=torch.uint8))
    # right types and sizes, but host memory: refused before the C call
    with pytest.raises(ValueError, match="must be a CUDA device tensor"):
        call()
    with pytest.raises(TypeError, match="h: expected f16"):
        S = M * k
        i32 = torch.zeros(S + 1, dtype=torch.int32)
        awq.moe_w2_reduce(torch.zeros((S, SHAPE.inter), dtype=torch.float32), good["wts"], M, SHAPE, w, i32, i32,
                          i32, i32, good["out"], good["st"])
    with pytest.raises(ValueError, match="logits: holds"):
        awq.moe_router_topk(torch.zeros((M, 100), dtype=torch.float32), M, SHAPE, good["ids"], good["wts"])
    with pytest.raises(ValueError, match="w13_q: must be a CUDA device tensor"):
        awq.Weights.of(torch.zeros(4, dtype=torch.int32), FAKE, FAKE, FAKE)


def test_nvfp4_shapes_and_refusals_on_the_host():
    L = awq.lib()
    nv = awq.Shape(512, 10, 2560, 160, 16, 1)
    assert awq.moe_workspace_bytes(nv, 8) > 0
    # a block of 16 needs one-byte scales; 32-groups need 3- or 4-byte records
    for bad in (awq.Shape(512, 10, 2560, 160, 16, 4), awq.Shape(512, 10, 2560, 160, 32, 1)):
        assert awq.moe_workspace_bytes(bad, 8) == 0
    # NVFP4 banks without global scales, or misaligned ones, are refused
    assert call_layer(shape=nv, ws_bytes=awq.moe_workspace_bytes(nv, 1)) == awq.ERR_INVALID_ARG
    w = weights(global_scale=FAKE + 2)
    assert call_layer(shape=nv, w=w, ws_bytes=awq.moe_workspace_bytes(nv, 1)) == awq.ERR_MISALIGNED
    # the stage calls and the static entry point take int4 banks only
    w = weights(global_scale=FAKE)
    assert L.awq_moe_w13_swiglu(FAKE, 1, C.byref(nv), C.byref(w), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                None) == awq.ERR_UNSUPPORTED_SHAPE
    assert L.awq_moe_w2_reduce(FAKE, FAKE, 1, C.byref(nv), C.byref(w), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                               None) == awq.ERR_UNSUPPORTED_SHAPE
    assert L.awq_moe_layer_static(FAKE, FAKE, FAKE, 2, C.byref(nv), C.byref(w), FAKE, FAKE,
                                  None) == awq.ERR_UNSUPPORTED_SHAPE
    for path in (awq.PATH_STAGED, awq.PATH_SLICED):
        opts = awq.Options(0, path, 0, None)
        assert L.awq_moe_layer_ex(FAKE, FAKE, FAKE, 2, C.byref(nv), C.byref(w), FAKE, FAKE,
                                  awq.moe_workspace_bytes(nv, 2), FAKE, C.byref(opts), None) == \
            awq.ERR_UNSUPPORTED_SHAPE


def test_layer_ex_path_codes():
    L = awq.lib()
    for bad in (-1, awq.PATH_HYBRID + 1):
        opts = awq.Options(0, bad, 0, None)
        assert L.awq_moe_layer_ex(FAKE, FAKE, FAKE, 2, C.byref(SHAPE), C.byref(weights()), FAKE, FAKE, 1 << 30,
                                  FAKE, C.byref(opts), None) == awq.ERR_INVALID_ARG
    # the three stage launches stop at their token limit; the hybrid path does not
    big = awq.W2_STAGE_MAX_TOKENS + 1
    ws = awq.moe_workspace_bytes(SHAPE, big)
    opts = awq.Options(0, awq.PATH_STAGED, 0, None)
    assert L.awq_moe_layer_ex(FAKE, FAKE, FAKE, big, C.byref(SHAPE), C.byref(weights()), FAKE, FAKE, ws,
                              FAKE, C.byref(opts), None) == awq.ERR_UNSUPPORTED_SHAPE
