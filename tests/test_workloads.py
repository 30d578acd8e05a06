"""The seeded input generator: determinism, shapes and recipe (CPU only)."""
import numpy as np

from workloads import WORKLOADS, Generator, bf16_bits_to_f32, f32_to_bf16_bits, scaled


def test_bf16_round_to_nearest_even():
    a = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, -2.5, 3.0e38], dtype=np.float32)
    b = bf16_bits_to_f32(f32_to_bf16_bits(a))
    assert b[0] == 1.0 and b[1] == 1.0 and b[2] == 1.0 + 2**-6 and b[3] == -2.5


def test_thread_count_does_not_change_values():
    s = scaled(WORKLOADS["mixtral_bf16"], T=64, h=256, d_ff=384, E=4)
    a = Generator(s, threads=1)
    b = Generator(s, threads=7)
    for fa, fb in zip(a.experts(), b.experts()):
        assert (fa == fb).all()
    assert (a.x() == b.x()).all()
    w1, w3, w2 = a.expert(2)
    W1, W3, W2 = b.experts()
    assert (w1 == W1[2]).all() and (w3 == W3[2]).all() and (w2 == W2[2]).all()


def test_row_slice_matches_full():
    s = scaled(WORKLOADS["tiny_f32"], T=5000, h=1024)  # several 4M-element pieces
    g = Generator(s)
    full = g.x()
    assert (g.x(slice(4000, 4200)) == full[4000:4200]).all()
    assert (g.x(slice(0, 3)) == full[:3]).all()


def test_recipe_statistics():
    s = scaled(WORKLOADS["mixtral_bf16"], T=512, h=1024, d_ff=2048, E=2)
    g = Generator(s)
    x = bf16_bits_to_f32(g.x())
    assert abs(x.std() - 1.0) < 0.01
    w1, _, w2 = g.expert(0)
    assert abs(bf16_bits_to_f32(w1).std() * np.sqrt(1024) - 1.0) < 0.01
    assert abs(bf16_bits_to_f32(w2).std() * np.sqrt(2048) - 1.0) < 0.01
    zb = Generator(WORKLOADS["skewed_bf16"]).logit_bias()
    assert zb.shape == (64,) and abs(zb.sum() - 1.0) < 1e-6 and (np.diff(zb) < 0).all()
    sb = Generator(WORKLOADS["finegrained_bf16"]).select_bias()
    assert sb.shape == (256,) and sb.min() >= -0.1 and sb.max() <= 0.1


def test_topk_idx_distinct():
    s = scaled(WORKLOADS["finegrained_bf16"], T=100)
    idx = Generator(s).topk_idx()
    assert idx.shape == (100, 8)
    assert all(len(set(r)) == 8 for r in idx.tolist())
    assert idx.min() >= 0 and idx.max() < 256
