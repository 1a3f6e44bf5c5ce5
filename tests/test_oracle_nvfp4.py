"""Pins of the oracle's NVFP4 weight format against facts that do not come
from the oracle: the published E2M1 value table and E4M3 landmarks
(``tests/golden/nvfp4_facts.json``), PyTorch's float8_e4m3fn decoder for every
E4M3 code, hand-built packed words, a round trip through a test-side encoder,
and the dense SwiGLU FFN (numpy matmul, scipy's logistic function) on weights
decoded here."""
import json
import math
import os

import numpy as np
import pytest
from scipy.special import expit

import oracle
import synth

FACTS = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "nvfp4_facts.json")))
E2M1 = np.array(FACTS["e2m1_values"]["value"], np.float64)


def e4m3_library(codes):
    """E4M3 codes -> float64 through PyTorch's float8_e4m3fn dtype."""
    torch = pytest.importorskip("torch")
    t = torch.tensor(np.asarray(codes, np.uint8).ravel(), dtype=torch.uint8)
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy().reshape(np.shape(codes))


def test_e2m1_every_code_matches_the_published_table():
    for code in range(16):
        got = oracle.e2m1_to_double(code)
        assert got == E2M1[code] and math.copysign(1.0, got) == math.copysign(1.0, E2M1[code])


def test_e4m3_landmarks_from_the_format_definition():
    f = FACTS["e4m3_facts"]
    for key in ("max_normal", "min_normal", "min_subnormal", "one"):
        assert oracle.e4m3_to_double(f[key]["code"]) == f[key]["value"]
        assert oracle.e4m3_to_double(f[key]["code"] | 0x80) == -f[key]["value"]
    for code in f["nan_codes"]:
        assert math.isnan(oracle.e4m3_to_double(code))


def test_e4m3_every_code_matches_pytorch_float8():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    lib = e4m3_library(codes)
    got = np.array([oracle.e4m3_to_double(int(c)) for c in codes])
    assert np.array_equal(got, lib)
    assert np.array_equal(np.signbit(got), np.signbit(lib))


def pack_codes(C):
    """Encode E2M1 codes C[K][N] (0..15) as u32[K/8][N]: row 8i+j in bits 4j..4j+3."""
    K, N = C.shape
    words = np.zeros((K // 8, N), np.uint64)
    for j in range(8):
        words |= C[j::8, :].astype(np.uint64) << np.uint64(4 * j)
    return words.astype(np.uint32)


def test_decode_hand_built_words_and_block_boundary():
    # column 0: rows 0-7 codes 0..7 (word 0x76543210), rows 8-15 codes 8..15
    # (0xFEDCBA98); rows 16-31 repeat them under the second block scale
    q = np.array([[0x76543210, 0x11111111], [0xFEDCBA98, 0x22222222],
                  [0x76543210, 0x33333333], [0xFEDCBA98, 0x44444444]], np.uint32)
    scales = np.array([[0x38, 0x30], [0x40, 0x01]], np.uint8)     # 1.0, 0.5 / 2.0, 2^-9
    g = 0.75
    W = oracle.decode_nvfp4(q, scales, g, 32, 2)
    col0 = np.concatenate([E2M1 * 1.0, E2M1 * 2.0]) * g
    np.testing.assert_array_equal(W[:, 0], col0)
    col1 = np.concatenate([np.full(8, 0.5), np.full(8, 1.0), np.full(8, 1.5), np.full(8, 2.0)])
    col1 *= np.concatenate([np.full(16, 0.5), np.full(16, 2.0 ** -9)]) * g
    np.testing.assert_array_equal(W[:, 1], col1)


def test_decode_round_trip_against_test_encoder():
    rng = np.random.default_rng(11)
    K, N = 64, 24
    C = rng.integers(0, 16, size=(K, N))
    S = rng.integers(0, 0x7F, size=(K // 16, N)).astype(np.uint8)      # every finite positive code
    g = np.float32(0.8125)
    want = E2M1[C] * np.repeat(e4m3_library(S), 16, axis=0) * float(g)
    got = oracle.decode_nvfp4(pack_codes(C), S, g, K, N)
    np.testing.assert_array_equal(got, want)


def dense_ffn(x, W13, W2, I):
    g = x @ W13[:, :I]
    u = x @ W13[:, I:]
    return (g * expit(g) * u) @ W2


def tiny_nvfp4_bank(rng, E, H, I):
    """Random NVFP4 banks and their dense FP64 weights decoded here."""
    out = {k: [] for k in ("q13", "s13", "q2", "s2", "W13", "W2")}
    glob = (0.5 + rng.integers(0, 256, size=(E, 2)) / 512).astype(np.float32)
    for e in range(E):
        for K, N, qk, sk, wk, which in ((H, 2 * I, "q13", "s13", "W13", 0), (I, H, "q2", "s2", "W2", 1)):
            C = rng.integers(0, 16, size=(K, N))
            S = ((rng.integers(0, 4, size=(K // 16, N)) << 3) | rng.integers(0, 8, size=(K // 16, N))).astype(np.uint8)
            out[qk].append(pack_codes(C))
            out[sk].append(S)
            out[wk].append(E2M1[C] * np.repeat(e4m3_library(S), 16, axis=0) * float(glob[e, which]))
    return {k: np.stack(v) for k, v in out.items()}, glob


def test_nvfp4_single_expert_weight_one_reduces_to_dense_swiglu_ffn():
    rng = np.random.default_rng(5)
    E, H, I, M = 3, 64, 32, 4
    shape = synth.ExpertShape(num_experts=E, top_k=1, hidden=H, inter=I, group=16, meta_bytes=1)
    b, glob = tiny_nvfp4_bank(rng, E, H, I)
    x = (rng.standard_normal((M, H)) * 0.5).astype(np.float16)
    ids = np.array([[1], [0], [2], [1]], np.int32)
    w = np.ones((M, 1), np.float32)
    out, h = oracle.moe_layer_nvfp4(x, ids, w, shape, b["q13"], b["s13"], b["q2"], b["s2"], glob)
    for t in range(M):
        e = ids[t, 0]
        xd = x[t].astype(np.float64)
        np.testing.assert_allclose(out[t], dense_ffn(xd, b["W13"][e], b["W2"][e], I), rtol=1e-12, atol=1e-12)
        g = xd @ b["W13"][e][:, :I]
        u = xd @ b["W13"][e][:, I:]
        np.testing.assert_allclose(h[t], g * expit(g) * u, rtol=1e-12, atol=1e-12)


def test_nvfp4_global_scales_act_linearly_and_exactly():
    rng = np.random.default_rng(9)
    E, H, I, M, k = 4, 64, 32, 3, 2
    shape = synth.ExpertShape(num_experts=E, top_k=k, hidden=H, inter=I, group=16, meta_bytes=1)
    b, glob = tiny_nvfp4_bank(rng, E, H, I)
    x = (rng.standard_normal((M, H)) * 0.5).astype(np.float16)
    ids = np.array([[0, 3], [2, 1], [3, 0]], np.int32)
    w = np.array([[0.25, 0.75], [0.5, 0.5], [1.0, 0.0]], np.float32)
    out, h = oracle.moe_layer_nvfp4(x, ids, w, shape, b["q13"], b["s13"], b["q2"], b["s2"], glob)
    g2 = glob.copy()
    g2[:, 1] *= 2                        # every W2 global doubled: the output doubles exactly
    out2, h2 = oracle.moe_layer_nvfp4(x, ids, w, shape, b["q13"], b["s13"], b["q2"], b["s2"], g2)
    assert np.array_equal(h2, h) and np.array_equal(out2, 2 * out)
    # a slot with router weight 0 (token 2, slot 1 -> expert 0) adds nothing
    b2 = dict(b)
    b2["q2"] = b["q2"].copy()
    b2["q2"][0] ^= np.uint32(0x5A5A5A5A)
    ids_only0 = np.array([[0, 3], [2, 1], [3, 0]], np.int32)
    o3, _ = oracle.moe_layer_nvfp4(x, ids_only0, w, shape, b2["q13"], b2["s13"], b2["q2"], b2["s2"], glob)
    assert np.array_equal(o3[2], out[2])


def test_synthetic_nvfp4_codes_stay_in_the_generators_range():
    shape = synth.ExpertShape(num_experts=4, top_k=2, inter=160, group=16, meta_bytes=1)
    _, s13, _, s2 = synth.expert_weights(shape, 7, 1, 2)
    for s in (s13, s2):
        assert s.dtype == np.uint8 and s.max() <= 0x1F       # exponent field 0..3
    gl = synth.nvfp4_global(7, 1, 4)
    assert gl.dtype == np.float32 and gl.min() >= 0.5 and gl.max() < 1.0
