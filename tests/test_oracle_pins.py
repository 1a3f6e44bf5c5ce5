"""Pins of the CPU oracle against facts that do not come from the oracle.

Every oracle function is checked here by at least one of: a hand-built case
with a known answer, a library routine (numpy's binary16, numpy matmul,
scipy's logistic function), brute force on tiny inputs, an exact invariant of
the mathematics, or a number the pages print (``tests/golden/``).
"""
import json
import os

import numpy as np
import pytest
from scipy.special import expit

import oracle
import synth

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "layout_facts.json")))


# ------------------------------------------------------------- helpers (test-side encoders)

def pack_q(Q):
    """Encode integer Q[K][N] in 0..15 as u32[K/8][N]: row 8i+j in bits 4j..4j+3."""
    K, N = Q.shape
    words = np.zeros((K // 8, N), np.uint64)
    for j in range(8):
        words |= Q[j::8, :].astype(np.uint64) << np.uint64(4 * j)
    return words.astype(np.uint32)


def pack_meta(S16, Z, mb):
    """Encode fp16 scales S16[G][N] and zeros Z[G][N] as records u8[G][N][mb]."""
    bits = S16.astype(np.float16).view(np.uint16)
    rec = np.zeros(S16.shape + (mb,), np.uint8)
    rec[..., 0] = bits & 0xFF
    rec[..., 1] = bits >> 8
    rec[..., 2] = Z
    return rec


def random_quant(rng, K, N, G=32, pow2_scales=False):
    Q = rng.integers(0, 16, size=(K, N))
    Z = rng.integers(0, 16, size=(K // G, N))
    if pow2_scales:
        S = np.float16(2.0) ** rng.integers(-9, -5, size=(K // G, N)).astype(np.float16)
    else:
        S = rng.uniform(0.002, 0.02, size=(K // G, N)).astype(np.float16)
    W = (Q - np.repeat(Z, G, axis=0)) * np.repeat(S.astype(np.float64), G, axis=0)
    return Q, Z, S, W


def tiny_bank(rng, E, H, I, G=32, mb=4, pow2=False):
    """Random expert banks plus their exact dense FP64 weights (test-side)."""
    w13q, w13m, w2q, w2m, W13, W2 = [], [], [], [], [], []
    for _ in range(E):
        Q, Z, S, W = random_quant(rng, H, 2 * I, G, pow2)
        w13q.append(pack_q(Q)); w13m.append(pack_meta(S, Z, mb)); W13.append(W)
        Q, Z, S, W = random_quant(rng, I, H, G, pow2)
        w2q.append(pack_q(Q)); w2m.append(pack_meta(S, Z, mb)); W2.append(W)
    return (np.stack(w13q), np.stack(w13m), np.stack(w2q), np.stack(w2m),
            np.stack(W13), np.stack(W2))


# ------------------------------------------------------------------------ fp16 decode

def test_half_to_double_matches_numpy_binary16_for_every_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


@pytest.mark.parametrize("bits,value", [
    (0x3C00, 1.0), (0x0001, 2.0 ** -24), (0x0400, 2.0 ** -14), (0x7BFF, 65504.0),
    (0xC000, -2.0), (0x3555, 0.333251953125), (0x0000, 0.0)])
def test_half_to_double_closed_forms(bits, value):
    assert oracle.half_to_double(bits) == value


# ------------------------------------------------------------------------ dequant

@pytest.mark.parametrize("mb", [3, 4])
def test_dequant_hand_built_word(mb):
    # one group (K=32), one column; word 0 = 0x76543210 gives q_j = j,
    # word 1 = 0xFEDCBA98 gives q_j = 8 + j; scale 1.0, zero 8 => w = q - 8.
    q = np.array([[0x76543210], [0xFEDCBA98], [0x00000000], [0xFFFFFFFF]], np.uint32)
    rec = np.zeros((1, 1, mb), np.uint8)
    rec[0, 0, 0], rec[0, 0, 1], rec[0, 0, 2] = 0x00, 0x3C, 8
    W = oracle.decode_matrix(q, rec, 32, 1)
    expect = np.array(list(range(8)) + list(range(8, 16)) + [0] * 8 + [15] * 8, np.float64) - 8
    assert np.array_equal(W[:, 0], expect)


def test_dequant_subnormal_and_max_scales():
    q = np.full((4, 2), 0xFFFFFFFF, np.uint32)            # q = 15 everywhere
    rec = np.zeros((1, 2, 4), np.uint8)
    rec[0, 0, :2] = [0x01, 0x00]                            # 2^-24
    rec[0, 1, :2] = [0xFF, 0x7B]                            # 65504
    rec[0, :, 2] = 0
    W = oracle.decode_matrix(q, rec, 32, 2)
    assert np.all(W[:, 0] == 15 * 2.0 ** -24)
    assert np.all(W[:, 1] == 15 * 65504.0)


@pytest.mark.parametrize("mb", [3, 4])
def test_dequant_round_trip_against_test_encoder(mb):
    rng = np.random.default_rng(1)
    K, N = 128, 48
    Q, Z, S, W = random_quant(rng, K, N)
    got = oracle.decode_matrix(pack_q(Q), pack_meta(S, Z, mb), K, N)
    assert np.array_equal(got, W)


def test_three_and_four_byte_layouts_decode_identically():
    assert GOLDEN["layouts_decode_identically"]["value"]
    rng = np.random.default_rng(2)
    shape = synth.ExpertShape(inter=160)
    q13, m13_4, q2, m2_4 = synth.expert_weights(shape, 7, 0, 3, meta_bytes=4)
    _, m13_3, _, m2_3 = synth.expert_weights(shape, 7, 0, 3, meta_bytes=3)
    W4 = oracle.decode_matrix(q13, m13_4, 2560, 320)
    W3 = oracle.decode_matrix(q13, m13_3, 2560, 320)
    assert np.array_equal(W3, W4)
    assert np.array_equal(oracle.decode_matrix(q2, m2_3, 160, 2560),
                          oracle.decode_matrix(q2, m2_4, 160, 2560))
    del rng


# --------------------------------------------------------------- compact layout facts

def test_prepare_compact_drops_byte_three():
    m4 = np.arange(4 * 37, dtype=np.uint32).astype(np.uint8).reshape(37, 4)
    m3 = oracle.prepare_compact(m4)
    assert m3.shape == (37, 3)
    assert np.array_equal(m3, m4[:, :3])
    # record r sits at byte 3r of the compact bank
    flat = m3.ravel()
    for r in (0, 1, 31, 36):
        assert bytes(flat[3 * r:3 * r + 3]) == bytes(m4[r, :3])


def test_compact_tile_geometry_matches_pages():
    g = GOLDEN["compact_tile"]
    assert g["records_per_tile"] * 3 == g["tile_bytes"]
    assert g["tile_bytes"] // 4 == g["aligned_words"]
    # last record of a 32-record tile starts at byte 3 * 31 and ends inside the tile
    assert 3 * (g["records_per_tile"] - 1) == g["last_record_byte_offset"]
    assert g["last_record_byte_offset"] + 3 <= g["tile_bytes"]
    # every metadata row of both matrices is a whole number of tiles
    for n in (320, 2560, 1280):
        assert (3 * n) % g["tile_bytes"] == 0


def test_bytes_saved_by_compact_layout_match_pages():
    s = GOLDEN["shape"]["value"]
    shape = synth.ExpertShape(num_experts=s["num_experts"], hidden=s["hidden"],
                              inter=s["inter_local"], group=s["group"])
    per_expert = shape.expert_bytes(4) - shape.expert_bytes(3)
    assert per_expert == shape.w13_records + shape.w2_records == 38400
    total = per_expert * shape.num_experts * GOLDEN["layers"]["value"]
    assert total == GOLDEN["compact_bytes_saved_per_rank"]["value"]
    assert total == GOLDEN["compact_bytes_saved_per_rank"]["mib"] * 2 ** 20
    # and the oracle's decoder consumes exactly that many records
    q13, m13, q2, m2 = synth.expert_weights(shape, 0, 0, 0, 4)
    assert m13.shape[:2] == (s["w13_K"] // 32, s["w13_N"])
    assert m2.shape[:2] == (s["w2_K"] // 32, s["w2_N"])


# ------------------------------------------------------------------------ route

def brute_route(ids, E):
    M, k = ids.shape
    pairs = sorted((int(ids[t, j]), t * k + j) for t in range(M) for j in range(k))
    experts = sorted(set(p[0] for p in pairs))
    A, S = len(experts), M * k
    act = experts + [-1] * (S - A)
    off = [next(i for i, p in enumerate(pairs) if p[0] == e) for e in experts] + [S] * (S + 1 - A)
    return np.array(act), np.array(off), np.array([p[1] for p in pairs]), A


@pytest.mark.parametrize("M,k,E,seed", [(1, 10, 512, 0), (2, 10, 512, 1), (8, 10, 512, 2),
                                        (8, 10, 16, 3), (37, 3, 7, 4), (128, 10, 512, 5),
                                        (5, 1, 1, 6)])
def test_route_matches_brute_force_sort(M, k, E, seed):
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, E, size=(M, k)).astype(np.int32)   # duplicates allowed
    act, off, srt, A = oracle.route(ids, E)
    ba, bo, bs, bA = brute_route(ids, E)
    assert A == bA
    assert np.array_equal(act, ba) and np.array_equal(off, bo) and np.array_equal(srt, bs)
    # invariants
    S = M * k
    assert np.all(np.diff(off) >= 0) and off[A] == S and off[0] == 0
    assert np.all(np.diff(act[:A]) > 0)
    assert np.array_equal(np.sort(srt), np.arange(S))
    flat = ids.ravel()
    for a in range(A):
        seg = srt[off[a]:off[a + 1]]
        assert np.all(flat[seg] == act[a]) and np.all(np.diff(seg) > 0)


def test_route_rejects_out_of_range_ids():
    with pytest.raises(oracle.OracleError) as e:
        oracle.route(np.array([[0, 512]], np.int32), 512)
    assert e.value.code == oracle.BAD_EXPERT_ID
    with pytest.raises(oracle.OracleError):
        oracle.route(np.array([[-1, 3]], np.int32), 512)


# ------------------------------------------------------------------ expert stage

def dense_ffn(x, W13, W2, I):
    """Textbook SwiGLU FFN: W2^T (silu(W1^T x) * (W3^T x)), silu(g) = g * logistic(g)."""
    g = x @ W13[:, :I]
    u = x @ W13[:, I:]
    return (g * expit(g) * u) @ W2


def test_single_expert_weight_one_reduces_to_dense_swiglu_ffn():
    rng = np.random.default_rng(3)
    E, H, I, M = 4, 64, 32, 3
    shape = synth.ExpertShape(num_experts=E, top_k=1, hidden=H, inter=I)
    w13q, w13m, w2q, w2m, W13, W2 = tiny_bank(rng, E, H, I)
    x = (rng.standard_normal((M, H)) * 0.5).astype(np.float16)
    ids = np.array([[2], [0], [2]], np.int32)
    w = np.ones((M, 1), np.float32)
    out, h = oracle.moe_layer(x, ids, w, shape, w13q, w13m, w2q, w2m, 4)
    for t in range(M):
        e = ids[t, 0]
        ref = dense_ffn(x[t].astype(np.float64), W13[e], W2[e], I)
        np.testing.assert_allclose(out[t], ref, rtol=1e-12, atol=1e-12)
        g = x[t].astype(np.float64) @ W13[e][:, :I]
        u = x[t].astype(np.float64) @ W13[e][:, I:]
        np.testing.assert_allclose(h[t], g * expit(g) * u, rtol=1e-12, atol=1e-12)


def test_weighted_topk_sum_against_dense_per_slot_reference():
    rng = np.random.default_rng(4)
    E, H, I, M, k = 6, 64, 32, 4, 3
    shape = synth.ExpertShape(num_experts=E, top_k=k, hidden=H, inter=I)
    w13q, w13m, w2q, w2m, W13, W2 = tiny_bank(rng, E, H, I, mb=3)
    x = (rng.standard_normal((M, H)) * 0.5).astype(np.float16)
    ids = np.array([[0, 1, 2], [5, 0, 3], [3, 3, 1], [4, 2, 5]], np.int32)
    w = rng.dirichlet(np.ones(k), size=M).astype(np.float32)
    out, _ = oracle.moe_layer(x, ids, w, shape, w13q, w13m, w2q, w2m, 3)
    for t in range(M):
        ref = sum(float(w[t, j]) * dense_ffn(x[t].astype(np.float64), W13[ids[t, j]], W2[ids[t, j]], I)
                  for j in range(k))
        np.testing.assert_allclose(out[t], ref, rtol=1e-11, atol=1e-12)


@pytest.fixture(scope="module")
def small_layer():
    rng = np.random.default_rng(5)
    E, H, I, M, k = 8, 64, 32, 5, 3
    shape = synth.ExpertShape(num_experts=E, top_k=k, hidden=H, inter=I)
    bank = tiny_bank(rng, E, H, I, pow2=False)
    x = (rng.standard_normal((M, H)) * 0.5).astype(np.float16)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(M)]).astype(np.int32)
    w = rng.dirichlet(np.ones(k), size=M).astype(np.float32)
    return shape, bank, x, ids, w


def run(shape, bank, x, ids, w, mb=4):
    return oracle.moe_layer(x, ids, w, shape, bank[0], bank[1], bank[2], bank[3], mb)[0]


def test_token_permutation_equivariance_is_exact(small_layer):
    shape, bank, x, ids, w = small_layer
    out = run(shape, bank, x, ids, w)
    perm = np.array([3, 0, 4, 1, 2])
    outp = run(shape, bank, x[perm], ids[perm], w[perm])
    assert np.array_equal(outp, out[perm])


def test_permuting_slots_with_their_weights_leaves_output_unchanged(small_layer):
    shape, bank, x, ids, w = small_layer
    out = run(shape, bank, x, ids, w)
    p = np.array([2, 0, 1])
    np.testing.assert_allclose(run(shape, bank, x, ids[:, p], w[:, p]), out, rtol=1e-13, atol=1e-14)


def test_zero_router_weight_expert_contributes_nothing(small_layer):
    shape, bank, x, ids, w = small_layer
    w0 = w.copy()
    w0[:, 1] = 0.0
    out = run(shape, bank, x, ids, w0)
    scrambled = [b.copy() for b in bank[:4]]
    rng = np.random.default_rng(9)
    for t in range(ids.shape[0]):
        e = ids[t, 1]
        if e in ids[:, [0, 2]]:
            continue                       # expert also used with a non-zero weight
        for qi in (0, 2):                  # any packed words
            scrambled[qi][e] = rng.integers(0, 2 ** 32, size=scrambled[qi][e].shape,
                                            dtype=np.uint64).astype(np.uint32)
        for mi in (1, 3):                  # any finite scale, any zero byte
            m = scrambled[mi][e]
            sc = rng.uniform(-100, 100, size=m.shape[:-1]).astype(np.float16).view(np.uint16)
            m[..., 0], m[..., 1] = sc & 0xFF, sc >> 8
            m[..., 2] = rng.integers(0, 256, size=m.shape[:-1])
    assert np.array_equal(run(shape, scrambled + list(bank[4:]), x, ids, w0), out)


def test_doubling_every_w2_scale_doubles_output_exactly(small_layer):
    shape, bank, x, ids, w = small_layer
    out = run(shape, bank, x, ids, w)
    m2 = bank[3].copy()
    s = m2[..., 0].astype(np.uint16) | (m2[..., 1].astype(np.uint16) << 8)
    s2 = (s.view(np.float16) * np.float16(2)).view(np.uint16)
    assert np.array_equal(s2.view(np.float16).astype(np.float64), 2 * s.view(np.float16).astype(np.float64))
    m2[..., 0] = s2 & 0xFF
    m2[..., 1] = s2 >> 8
    out2 = run(shape, (bank[0], bank[1], bank[2], m2), x, ids, w)
    assert np.array_equal(out2, 2 * out)


def test_identical_experts_with_weights_summing_to_one_give_single_expert(small_layer):
    shape, bank, x, ids, w = small_layer
    same = [b.copy() for b in bank[:4]]
    for b in same:
        b[:] = b[0]
    out = run(shape, same, x, ids, w)
    single = run(shape, same, x, ids[:, :1] * 0, np.ones((ids.shape[0], 1), np.float32))
    np.testing.assert_allclose(out, single * w.astype(np.float64).sum(1, keepdims=True),
                               rtol=1e-13, atol=1e-14)


def test_silu_zero_gate_gives_zero_h_and_sign_structure():
    # gate weights all zero (q == zero) => g = 0 => h = 0 exactly; up weights
    # arbitrary. Then out = 0 exactly.
    rng = np.random.default_rng(11)
    E, H, I = 2, 64, 32
    shape = synth.ExpertShape(num_experts=E, top_k=1, hidden=H, inter=I)
    w13q, w13m, w2q, w2m, W13, W2 = tiny_bank(rng, E, H, I)
    Q = np.full((H, 2 * I), 5)
    Qu = rng.integers(0, 16, size=(H, I))
    Q[:, I:] = Qu
    w13q[0] = pack_q(Q)
    w13m[0][..., 2] = 5                                      # zero = 5 on every record
    x = (rng.standard_normal((1, H)) * 0.5).astype(np.float16)
    out, h = oracle.moe_layer(x, np.array([[0]], np.int32), np.ones((1, 1), np.float32), shape,
                              w13q, w13m, w2q, w2m, 4)
    assert np.all(h == 0.0) and np.all(out == 0.0)


def test_w2_stage_alone_matches_layer(small_layer):
    shape, bank, x, ids, w = small_layer
    out, h = oracle.moe_layer(x, ids, w, shape, *bank[:4], 4)
    out2 = oracle.w2_reduce(h, ids, w, shape, bank[2], bank[3], 4)
    h2 = oracle.w13_swiglu(x, ids, shape, bank[0], bank[1], 4)
    assert np.array_equal(out2, out) and np.array_equal(h2, h)


# ------------------------------------------------------------------------------ router

def test_router_closed_form_from_log_probabilities():
    # logits = log p for a designed p: the k chosen are the k largest p and the
    # renormalised weights are p_i / (sum of the chosen p), whatever the rest is
    E, k = 32, 4
    p = np.full(E, 1e-9)
    chosen = {5: 0.4, 17: 0.3, 2: 0.2, 30: 0.1}
    for e, v in chosen.items():
        p[e] = v
    lg = np.log(p).astype(np.float32)[None, :]
    ids, w = oracle.router_topk(lg, k)
    assert ids[0].tolist() == [5, 17, 2, 30]
    pl = np.exp(lg[0].astype(np.float64))
    want = pl[[5, 17, 2, 30]] / pl[[5, 17, 2, 30]].sum()
    np.testing.assert_allclose(w[0], want, rtol=1e-13, atol=0)
    np.testing.assert_allclose(w[0], [0.4, 0.3, 0.2, 0.1], rtol=1e-6)


def test_router_equal_logits_choose_lowest_ids_with_equal_weights():
    E, k = 512, 10
    ids, w = oracle.router_topk(np.zeros((2, E), np.float32), k)
    assert ids.tolist() == [list(range(k))] * 2
    np.testing.assert_array_equal(w, np.full((2, k), 1.0 / k))


def test_router_ties_inside_the_top_k_break_to_the_lower_id():
    # integer logits with many ties; the chosen set is fixed by counting
    E, k = 40, 10
    rng = np.random.default_rng(3)
    lg = rng.integers(-3, 4, size=(6, E)).astype(np.float32)
    ids, _ = oracle.router_topk(lg, k)
    for t in range(6):
        # expected: sort by (-value, id) -- a different procedure than the
        # oracle's k selection passes over probabilities
        order = sorted(range(E), key=lambda e: (-float(lg[t, e]), e))[:k]
        assert ids[t].tolist() == order


def test_router_shift_invariance_is_exact():
    # adding a constant to every logit of a token (exactly representable here)
    # changes neither the choice nor the weights
    rng = np.random.default_rng(4)
    lg = (rng.integers(-64, 64, size=(4, 512)) / 8.0).astype(np.float32)
    a_ids, a_w = oracle.router_topk(lg, 10)
    for shift in (16.0, 1000.0):        # 1000: exp of an unshifted logit would overflow
        b_ids, b_w = oracle.router_topk(lg + np.float32(shift), 10)
        np.testing.assert_array_equal(a_ids, b_ids)
        np.testing.assert_allclose(a_w, b_w, rtol=1e-15, atol=0)


def test_router_weights_are_the_softmax_restricted_to_the_chosen_logits():
    # full softmax then renormalisation == softmax over the chosen logits only
    rng = np.random.default_rng(5)
    lg = rng.standard_normal((8, 512)).astype(np.float32)
    ids, w = oracle.router_topk(lg, 10)
    for t in range(8):
        sel = lg[t, ids[t]].astype(np.float64)
        assert np.all(np.diff(sel) <= 0)
        assert sel.min() >= np.delete(lg[t], ids[t]).max()
        e = np.exp(sel - sel.max())
        np.testing.assert_allclose(w[t], e / e.sum(), rtol=1e-13, atol=0)
        assert abs(w[t].sum() - 1.0) < 1e-14


def test_router_with_k_equal_to_e_is_the_full_softmax_in_descending_order():
    rng = np.random.default_rng(6)
    lg = rng.standard_normal((2, 16)).astype(np.float32)
    ids, w = oracle.router_topk(lg, 16)
    for t in range(2):
        assert sorted(ids[t].tolist()) == list(range(16))
        from scipy.special import softmax
        np.testing.assert_allclose(w[t], softmax(lg[t].astype(np.float64))[ids[t]], rtol=1e-13)


def test_router_matches_the_input_generator_on_its_workloads():
    # the seeded harness (softmax in FP64, lexsort) and the oracle are written
    # independently; on the generator's own logits they agree on the ids
    # bit-exactly and on the weights to fp32 rounding
    for regime, M in (("rotating", 8), ("hot", 4), ("zipf", 32)):
        lg = synth.router_logits(9, 2, M, regime=regime)
        ids_h, w_h = synth.router_topk(lg, 10)
        ids_o, w_o = oracle.router_topk(lg, 10)
        np.testing.assert_array_equal(ids_h, ids_o)
        np.testing.assert_allclose(w_h, w_o, rtol=2e-7, atol=0)
