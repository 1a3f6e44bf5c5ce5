"""Device-side fill of synthetic expert banks (CUDA), byte-identical to the
host generator in ``synth``. Used by the benchmark and the GPU tests to
create multi-GB weight stacks without host round trips."""
from __future__ import annotations

import ctypes as C
import os
import shutil
import subprocess

import synth

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "csrc", "synth_fill.cu")
LIB = os.path.join(HERE, "libawqsynth.so")


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.check_call([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                           "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden", "-shared",
                           "-cudart", "shared", "-o", tmp, SRC])
    os.replace(tmp, LIB)
    return LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"{LIB} is not built; run synth.device.build()")
        L = C.CDLL(LIB)
        L.awq_synth_fill_q.restype = C.c_int
        L.awq_synth_fill_q.argtypes = [C.c_void_p, C.c_int64, C.c_int32, C.c_int32, C.c_uint64,
                                       C.c_int32, C.c_int32, C.c_void_p]
        L.awq_synth_fill_meta.restype = C.c_int
        L.awq_synth_fill_meta.argtypes = [C.c_void_p, C.c_int64, C.c_int32, C.c_int32, C.c_int32,
                                          C.c_uint64, C.c_int32, C.c_int32, C.c_void_p]
        _lib = L
    return _lib


def _stream():
    import torch
    return C.c_void_p(torch.cuda.current_stream().cuda_stream)


def fill_layer(shape: synth.ExpertShape, seed: int, layer: int, w13_q, w13_meta, w2_q, w2_meta,
               meta_bytes: int | None = None):
    """Fill one layer's four device banks (torch tensors, contiguous, [E][...])."""
    mb = shape.meta_bytes if meta_bytes is None else meta_bytes
    E = shape.num_experts
    L = lib()
    st = _stream()
    rc = L.awq_synth_fill_q(w13_q.data_ptr(), shape.w13_words, 0, E, seed, layer, synth.T_W13_Q, st)
    rc |= L.awq_synth_fill_meta(w13_meta.data_ptr(), shape.w13_records, mb, 0, E, seed, layer,
                                synth.T_W13_META, st)
    rc |= L.awq_synth_fill_q(w2_q.data_ptr(), shape.w2_words, 0, E, seed, layer, synth.T_W2_Q, st)
    rc |= L.awq_synth_fill_meta(w2_meta.data_ptr(), shape.w2_records, mb, 0, E, seed, layer,
                                synth.T_W2_META, st)
    if rc:
        raise RuntimeError(f"synthetic bank fill failed ({rc})")
