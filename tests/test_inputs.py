"""The seeded input generator: determinism, chunk independence, bf16
rounding and the stated distributions (host side; the device fill is checked
bit for bit against it in the GPU tests)."""

import numpy as np

from kvq_inputs import gen


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -9, 1.0 + 2 ** -9, -2.5, 0.0], dtype=np.float32)
    r = gen.round_to_bf16(x)
    assert r[0] == 1.0
    assert r[1] == 1.0                             # exactly halfway -> even mantissa
    assert r[2] == 1.0 + 2 ** -7                   # above halfway rounds up
    assert r[3] == 1.0                             # below halfway rounds down
    assert r[4] == -2.5 and r[5] == 0.0
    y = np.random.default_rng(0).standard_normal(10000).astype(np.float32)
    ry = gen.round_to_bf16(y)
    assert np.all((ry.view(np.uint32) & 0xFFFF) == 0)
    assert np.all(np.abs(ry - y) <= np.abs(y) * 2 ** -8)


def test_blocks_are_independent_of_chunking():
    spec = gen.InputSpec(seed=3, n_kv_heads=2, n_q_heads=4, head_dim=32, bf16=True, spikes=True)
    K, V = spec.kv_block(layer=1, seqs=[0, 5], t0=0, n=100)
    K2, V2 = spec.kv_block(layer=1, seqs=[5], t0=37, n=40)
    np.testing.assert_array_equal(K2[0], K[1, :, 37:77])
    np.testing.assert_array_equal(V2[0], V[1, :, 37:77])
    K3, _ = spec.kv_block(layer=1, seqs=[0, 5], t0=0, n=100)
    np.testing.assert_array_equal(K, K3)
    q1 = spec.q_block(layer=0, seqs=[0, 1], step=4)
    q2 = spec.q_block(layer=0, seqs=[1], step=4)
    np.testing.assert_array_equal(q1[1], q2[0])
    assert not np.array_equal(spec.q_block(layer=0, seqs=[0], step=5), q1[:1])


def test_distributions():
    spec = gen.InputSpec(seed=0, n_kv_heads=2, n_q_heads=2, head_dim=128, bf16=False)
    sig = spec.sigma(layer=0)
    assert sig.shape == (2, 128)
    assert sig.min() >= 0.05 * (1 - 1e-6) and sig.max() <= 50.0 * (1 + 1e-6)
    # one outlier (x10) per block of 16 channels: the block max is >= 10 * 0.05
    for h in range(2):
        for blk in range(0, 128, 16):
            assert sig[h, blk:blk + 16].max() >= 0.5 - 1e-6
    K, V = spec.kv_block(layer=0, seqs=[0], t0=0, n=4096)
    z = K[0] / sig[:, None, :]
    assert abs(z.mean()) < 0.02 and abs(z.std() - 1.0) < 0.02
    tau_ratio = np.abs(V[0]).max(axis=-1)
    assert tau_ratio.max() < 2.0 * 4.5
    assert np.abs(gen.NORMAL_TABLE).max() < 4.5 and abs(gen.NORMAL_TABLE.mean()) < 1e-6
    assert gen.TAU_TABLE.min() > 0.5 and gen.TAU_TABLE.max() < 2.0


def test_spikes_rate():
    spec = gen.InputSpec(seed=3, n_kv_heads=1, n_q_heads=1, head_dim=128, bf16=False, spikes=True)
    plain = gen.InputSpec(seed=3, n_kv_heads=1, n_q_heads=1, head_dim=128, bf16=False, spikes=False)
    K, _ = spec.kv_block(layer=0, seqs=[0], t0=0, n=8192)
    K0, _ = plain.kv_block(layer=0, seqs=[0], t0=0, n=8192)
    rate = np.mean(K != K0)
    assert 0.0007 < rate < 0.0013


def test_lengths_in_range():
    spec = gen.InputSpec(seed=3, n_kv_heads=8, n_q_heads=32, head_dim=128)
    lens = spec.lengths(4, 1024, 131072)
    assert len(set(lens)) == 4 and all(1024 <= n <= 131072 for n in lens)
