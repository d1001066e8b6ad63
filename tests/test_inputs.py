"""The seeded input generators: determinism, chunking, bf16 rounding, distributions."""
import math

import numpy as np
import torch

from tile_level_copy_gb300 import inputs


def rne_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bits by round-to-nearest-even on the bit pattern."""
    u = a.astype(np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    return ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)


def test_bf16_conversion_is_round_to_nearest_even():
    rng = np.random.default_rng(0)
    a = np.concatenate([
        rng.standard_normal(100000).astype(np.float32) * 7,
        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 1 + 2 ** -8 + 2 ** -20, 0.0, -0.0],
                 np.float32),
    ])
    got = inputs.to_bf16(a).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(got, rne_bits(a))
    # ties go to even: 1 + 2^-8 -> 1.0; 1 + 3*2^-8 -> 1 + 2^-6
    vals = inputs.to_bf16(np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8], np.float32)).float().tolist()
    assert vals == [1.0, 1.0 + 2 ** -6]


def test_stream_is_deterministic_and_sliceable():
    n = inputs.CHUNK * 2 + 12345
    a = inputs.normal_f32(n, seed=7, tag=3)
    b = inputs.normal_f32(n, seed=7, tag=3)
    np.testing.assert_array_equal(a, b)
    c = inputs.normal_f32(1000, seed=7, tag=3, start=inputs.CHUNK - 500)
    np.testing.assert_array_equal(c, a[inputs.CHUNK - 500:inputs.CHUNK + 500])
    assert not np.array_equal(a[:100], inputs.normal_f32(100, seed=8, tag=3))
    assert not np.array_equal(a[:100], inputs.normal_f32(100, seed=7, tag=4))


def test_weights_per_expert_match_whole_tensor():
    w = inputs.WORKLOADS["tiny"]
    full = inputs.make_weight(w, 3, "W2")
    part = inputs.make_weight(w, 3, "W2", range(2, 3))
    assert full.shape == (w.E, w.d, w.ffn) and full.dtype == torch.bfloat16
    assert torch.equal(full[2], part[0])
    dst = torch.empty_like(full)
    inputs.make_weight_into(w, 3, "W2", dst)
    assert torch.equal(dst, full)


def test_distributions_and_shapes():
    w = inputs.WORKLOADS["tiny"].replace(T=2048)
    a = inputs.make_all(w, seed=1)
    assert a["logits"].dtype == np.float32 and a["logits"].shape == (w.T, w.E)
    assert a["x"].shape == (w.T, w.d) and a["W1"].shape == (w.E, w.ffn, w.d)
    assert abs(float(a["x"].float().std()) - 1.0) < 0.02
    assert abs(float(a["W1"].float().std()) - 1 / math.sqrt(w.d)) < 0.002
    assert abs(float(a["logits"].std()) - 1.0) < 0.02


def test_skew_bias_is_zipf_like():
    b = inputs.expert_bias(16)
    assert b[0] == 0.0
    assert abs(b[1] - (-2.4 * math.log(2))) < 1e-6
    assert np.all(np.diff(b) < 0)
    w = inputs.WORKLOADS["skew"]
    l0 = inputs.make_logits(w.replace(skew=False), 0)
    l1 = inputs.make_logits(w, 0)
    np.testing.assert_array_equal(l1, l0 + b[None, :])
