"""The seeded input generator: determinism, value ranges and routing regimes."""
import numpy as np
import pytest

import synth


def test_splitmix64_reference_values():
    # SplitMix64 with state 0 (Vigna's splitmix64.c: x += gamma; mix(x)):
    # the first outputs of the published generator.
    key = 0
    d = synth.draws(key, 0, 3)
    assert [int(v) for v in d] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_expert_weights_are_deterministic_and_independent_per_stream():
    shape = synth.ExpertShape()
    a = synth.expert_weights(shape, 1, 2, 3)
    b = synth.expert_weights(shape, 1, 2, 3)
    c = synth.expert_weights(shape, 1, 2, 4)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    assert not np.array_equal(a[0], c[0])


def test_weight_value_ranges():
    shape = synth.ExpertShape()
    q13, m13, q2, m2 = synth.expert_weights(shape, 0, 0, 0, 4)
    nib = np.stack([(q13 >> (4 * j)) & 0xF for j in range(8)])
    counts = np.bincount(nib.ravel(), minlength=16)
    assert counts.min() > 0.9 * nib.size / 16 and counts.max() < 1.1 * nib.size / 16
    s = (m13[..., 0].astype(np.uint16) | (m13[..., 1].astype(np.uint16) << 8)).view(np.float16)
    assert s.min() >= np.float16(0.002) and s.max() <= np.float16(0.02)
    assert set(np.unique(m13[..., 2]).tolist()) == set(range(16))
    assert np.all(m13[..., 3] == 0) and np.all(m2[..., 3] == 0)


def test_three_byte_records_are_the_four_byte_records_without_pad():
    shape = synth.ExpertShape()
    a = synth.expert_weights(shape, 5, 1, 9, 4)
    b = synth.expert_weights(shape, 5, 1, 9, 3)
    assert np.array_equal(a[1][..., :3], b[1]) and np.array_equal(a[3][..., :3], b[3])


@pytest.mark.parametrize("regime", ["rotating", "hot", "zipf"])
def test_routing_properties(regime):
    ids, w = synth.routing(3, 0, 8, regime=regime)
    assert ids.shape == (8, 10) and w.dtype == np.float32
    for t in range(8):
        assert len(set(ids[t].tolist())) == 10
    np.testing.assert_allclose(w.astype(np.float64).sum(1), 1.0, atol=1e-6)
    assert np.all(np.diff(w, axis=1) <= 0)                 # descending probability
    if regime == "hot":
        assert len(set(ids.ravel().tolist())) == 10


def test_rotating_union_grows_with_tokens():
    u = [len(set(synth.routing(0, layer, 8)[0].ravel().tolist())) for layer in range(20)]
    assert 70 <= np.mean(u) <= 80 and max(u) <= 80


def test_topk_ties_go_to_lower_expert_id():
    lg = np.zeros((1, 16), np.float32)
    lg[0, [3, 7, 11]] = 1.0
    ids, w = synth.router_topk(lg, 4)
    assert ids[0].tolist() == [3, 7, 11, 0]
    lg = np.ones((2, 8), np.float32)
    ids, w = synth.router_topk(lg, 3)
    assert ids.tolist() == [[0, 1, 2], [0, 1, 2]]
    np.testing.assert_allclose(w, 1.0 / 3, rtol=1e-6)


def test_hidden_states_distribution():
    x = synth.hidden_states(0, 0, 64)
    assert x.dtype == np.float16 and x.shape == (64, 2560)
    assert abs(float(x.astype(np.float64).std()) - 0.5) < 0.01


def test_integer_scale_encoding_matches_correctly_rounded_cast():
    r20 = np.arange(1 << 20, dtype=np.uint64)
    n = np.uint64(synth.SCALE_BASE) + r20 * np.uint64(synth.SCALE_STEP)
    ref = (n.astype(np.float64) * 2.0 ** -40).astype(np.float16).view(np.uint16)
    assert np.array_equal(synth.scale_bits(n), ref)
    # ties go to even: 1 + 2**-11 is halfway between 1 and 1 + 2**-10
    assert synth.scale_bits(np.array([(1 << 40) + (1 << 29)], np.uint64))[0] == 0x3C00
    assert synth.scale_bits(np.array([(1 << 40) + (3 << 29)], np.uint64))[0] == 0x3C02
