"""The seeded input generators: determinism, shapes and the stated recipes."""
import numpy as np
import pytest

from lora_serving_device_gb300 import workloads as W


def test_bf16_round_is_rne():
    a = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -9, -2.5, 0.0, 1e-3], np.float32)
    r = W.bf16_round(a)
    assert r[0] == 1.0
    assert r[1] == 1.0                      # exact tie -> even mantissa
    assert r[2] == np.float32(1.0 + 2 ** -7)  # above tie -> up
    assert r[3] == -2.5 and r[4] == 0.0
    assert np.all(W.bf16_round(r) == r)      # idempotent
    b = W.bf16_bits(r)
    assert b.dtype == np.uint16 and b[0] == 0x3F80


def test_toy_shapes():
    w = W.toy_mixed_batch()
    assert (w.T, w.d_in, w.d_out, w.r, w.n_slots) == (53, 256, 256, 16, 8)
    assert w.dtype == "f32"
    assert w.slot_ids.tolist()[:3] == [3, 5, 3]
    w2 = W.toy_mixed_batch()
    np.testing.assert_array_equal(w.x, w2.x)
    np.testing.assert_array_equal(w.A_pool, w2.A_pool)


def test_decode_ids_recipe():
    ids = W.decode_ids(2)
    assert ids.size == 64 and (ids == -1).sum() == 8
    assert ids.max() < 256
    np.testing.assert_array_equal(ids, W.decode_ids(2))


def test_prefill_recipe():
    lengths, slots = W.prefill_ids()
    assert len(lengths) == 64
    assert all(64 <= n <= 1024 for n in lengths[:16]) and lengths[16:] == [1] * 48
    assert len(set(slots[:16])) == 16
    assert all(0 <= s < 64 for s in slots)


@pytest.mark.parametrize("T,k", W.SWEEP_POINTS)
def test_sweep_ids(T, k):
    ids = W.sweep_ids(T, k)
    vals, counts = np.unique(ids, return_counts=True)
    assert vals.size == k and np.all(counts == T // k)


def test_stack_requests():
    lengths, slots = W.stack_requests()
    assert sum(lengths) == 256 and len(lengths) == 68
    assert sum(1 for s in slots if s == -1) == 7
    ranks = W.stack_ranks()
    assert set(ranks.tolist()) <= {8, 16, 64} and ranks.size == 250


def test_pools_zero_padding_and_subset():
    ranks = np.array([8, 16, 64, 8])
    A, B = W.make_pools(77, 4, 32, 24, 64, ranks=ranks)
    for j, rk in enumerate(ranks):
        assert np.all(A[j, :, rk:] == 0) and np.all(B[j, rk:, :] == 0)
        assert np.any(A[j, :, :rk] != 0)
    A2, B2 = W.make_pools(77, 4, 32, 24, 64, slots=[2], ranks=ranks)
    np.testing.assert_array_equal(A2[2], A[2])
    assert np.all(A2[0] == 0)


def test_decode_init_statistics():
    w = W.decode_bgmv()
    assert w.x.shape == (64, 4096) and w.A_pool.shape == (256, 4096, 16)
    assert abs(w.W0.std() - 0.02) < 0.001
    assert abs(w.A_pool[:4].std() - 1 / 64) < 0.001
    assert abs(w.B_pool[:4].std() - 0.02) < 0.001
    assert np.all(W.bf16_round(w.W0[:8]) == w.W0[:8])
