"""The shared seeded generators: NumPy and torch backends agree bit for bit."""
import numpy as np
import torch

from synth import C2_MID, C4_CONVKV, gen


def test_numpy_torch_bit_identical():
    key = gen.qkv_key(C2_MID, 3, 17, 1, "k")
    for dt in ("f32", "bf16"):
        a = gen.tensor_np(key, (97, 12, 128), dt)
        b = gen.tensor_torch(key, (97, 12, 128), dt).float().numpy()
        np.testing.assert_array_equal(a, b)


def test_index_map_subset():
    key = gen.qkv_key(C2_MID, 0, 1, 0, "q")
    full = gen.tensor_np(key, (10, 12, 128), "bf16")
    idx = np.array([5, 1000, 15359])
    np.testing.assert_array_equal(gen.tensor_np(key, None, "bf16", index_map=idx),
                                  full.reshape(-1)[idx])


def test_moments_and_keys_differ():
    k1 = gen.qkv_key(C2_MID, 0, 1, 0, "q")
    k2 = gen.qkv_key(C2_MID, 0, 2, 0, "q")
    assert k1 != k2
    x = gen.tensor_np(k1, (200000,), "f32")
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01
    assert np.abs(x).max() <= 2 * np.sqrt(3) + 1e-6


def test_conv_weights_backends_agree():
    a = gen.conv_weights_np(C4_CONVKV.with_(num_heads=3), 5)
    b = gen.conv_weights_torch(C4_CONVKV.with_(num_heads=3), 5).float().numpy()
    np.testing.assert_array_equal(a, b)
    assert a.shape == (2, 3, 128, 5)
    assert 0.17 < a.std() < 0.23
