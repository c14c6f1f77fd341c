"""GPU parity of the paged cache (a pool of blocks and a block table per
sequence) against the contiguous cache and the oracle.

The same appends go to a paged cache, a contiguous cache and the oracle, with
sequences interleaved so that each sequence's blocks lie scattered in the
pool.  The paged cache must give the same raw page bytes, codes, scales,
counters, restored tensors and attention outputs as the contiguous one, bit
for bit (the kernels' arithmetic does not depend on where a page lives), and
the attention within |d| <= 1e-3 + 1e-2 |ref| of the oracle.  Release returns
blocks to the pool, later appends reuse them, and an append the pool cannot
hold fails before any launch with the state unchanged.
"""

import numpy as np
import pytest

from kvq_inputs import gen
from oracle import kvq_oracle as O
from oracle import layout as L

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-3, 1e-2


@pytest.fixture(scope="module")
def torch():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


@pytest.fixture(scope="module")
def kvq(torch):
    import quantized_kv_cache_02_gb300 as kvq
    kvq.load_library()
    return kvq


class Trio:
    """A paged cache, a contiguous cache and the oracle fed the same appends."""

    def __init__(self, kvq, torch, batch, Hkv, Hq, D, R, G, qmax, capacity, pool_blocks, seed, spikes=False):
        self.torch, self.kvq = torch, kvq
        self.spec = gen.InputSpec(seed=seed, n_kv_heads=Hkv, n_q_heads=Hq, head_dim=D, spikes=spikes)
        self.paged = kvq.KVQCache(batch, Hkv, Hq, D, R, G, qmax, capacity, pool_blocks=pool_blocks)
        self.flat = kvq.KVQCache(batch, Hkv, Hq, D, R, G, qmax, capacity)
        self.args = (Hkv, D, R, G, qmax)
        self.seqs = [O.GroupedSequence(*self.args) for _ in range(batch)]
        self.t = [0] * batch  # tokens drawn per sequence (inputs keep advancing after a release)
        self.G, self.qmax = G, qmax

    def dev(self, a):
        return self.torch.from_numpy(np.ascontiguousarray(a)).to("cuda").to(self.torch.bfloat16).contiguous()

    def append(self, b, n):
        k, v = self.spec.kv_block(0, [b], self.t[b], n)
        self.t[b] += n
        for c in (self.paged, self.flat):
            c.append(self.dev(k), self.dev(v), b)
        self.seqs[b].append(k[0], v[0])

    def release(self, b):
        self.paged.release(b, 1)
        self.flat.release(b, 1)
        self.seqs[b] = O.GroupedSequence(*self.args)

    def check(self, b, heads=(0, 3, 7)):
        seq = self.seqs[b]
        for c in (self.paged, self.flat):
            st = c.seq_state(b)
            assert (st["total"], st["quantized"]) == (seq.total, seq.quantized)
        bits = O.code_bits(self.qmax)
        G = self.G
        for h in heads:
            raw = self.paged.export_pages(b, h)
            assert raw == self.flat.export_pages(b, h)
            assert raw == b"".join(
                L.pack_group_page(seq.key_codes()[h][j * G:(j + 1) * G], seq.value_codes()[h][j * G:(j + 1) * G],
                                  seq.key_scales()[h][j], seq.value_scales()[h][j * G:(j + 1) * G], bits)
                for j in range(seq.quantized // G))
            got = self.paged.export_unit(b, h)
            np.testing.assert_array_equal(got["window_k"], seq.window_kv()[0][h])

    def attend(self, step):
        B = len(self.seqs)
        q = self.spec.q_block(0, range(B), step)
        qd = self.dev(q)
        for kernel in (1, 2, 4):
            got = self.paged.decode_attention(qd, kernel=kernel).cpu().numpy()
            flat = self.flat.decode_attention(qd, kernel=kernel).cpu().numpy()
            np.testing.assert_array_equal(got, flat)
            for b, seq in enumerate(self.seqs):
                if seq.total == 0:
                    assert not got[b].any()
                    continue
                ref = seq.attend(q[b])
                excess = np.abs(got[b] - ref) - (ATOL + RTOL * np.abs(ref))
                assert excess.max() <= 0, f"kernel {kernel} seq {b}: |d| {np.abs(got[b] - ref).max():.3e}"


def test_paged_scattered_blocks_match_contiguous_and_oracle(kvq, torch):
    trio = Trio(kvq, torch, 4, 8, 32, 128, 128, 32, 7, 3000, pool_blocks=300, seed=31)
    # interleaved prefill chunks: each sequence's blocks are scattered in the pool
    for rnd in range(5):
        for b, n in enumerate((200, 64, 333, 40)):
            trio.append(b, n + rnd)
    for step in range(3):
        for b in range(4):
            trio.append(b, 1)
        trio.attend(step)
    for b in range(4):
        trio.check(b)
    kp, vp = trio.paged.restore(out_dtype="fp32")
    kf, vf = trio.flat.restore(out_dtype="fp32")
    np.testing.assert_array_equal(kp.cpu().numpy(), kf.cpu().numpy())
    np.testing.assert_array_equal(vp.cpu().numpy(), vf.cpu().numpy())
    used = sum(trio.seqs[b].quantized // 32 for b in range(4))
    assert trio.paged.pool_state() == (300 - used, 300)
    assert trio.paged.device_status() == 0


def test_paged_release_and_reuse(kvq, torch):
    trio = Trio(kvq, torch, 3, 8, 32, 128, 128, 32, 7, 2000, pool_blocks=60, seed=32)
    trio.append(0, 900)     # 24 groups
    trio.append(1, 1000)    # 27 groups
    free0, _ = trio.paged.pool_state()
    assert free0 == 60 - 24 - 27
    trio.release(0)
    assert trio.paged.pool_state()[0] == free0 + 24
    # sequence 2 now needs more blocks than were free before the release
    trio.append(2, 128 + 32 * 20 + 7)
    trio.append(0, 300)
    for step in range(2):
        for b in range(3):
            trio.append(b, 1)
        trio.attend(step)
    for b in range(3):
        trio.check(b)
    assert trio.paged.device_status() == 0


def test_paged_pool_exhaustion_leaves_state_unchanged(kvq, torch):
    trio = Trio(kvq, torch, 2, 8, 32, 128, 128, 32, 7, 4000, pool_blocks=10, seed=33)
    trio.append(0, 128 + 32 * 8)   # 8 groups, 2 left
    before = trio.paged.seq_state(1), trio.paged.pool_state()
    k, v = trio.spec.kv_block(0, [1], 0, 128 + 32 * 3)
    with pytest.raises(kvq.KVQError) as e:
        trio.paged.append(trio.dev(k), trio.dev(v), 1)
    assert e.value.status == kvq.binding.KVQ_ECAPACITY
    assert (trio.paged.seq_state(1), trio.paged.pool_state()) == before
    trio.append(1, 128 + 32 * 2)   # exactly the two free blocks
    assert trio.paged.pool_state() == (0, 10)
    trio.attend(0)
    for b in range(2):
        trio.check(b)


def test_paged_two_bit(kvq, torch):
    trio = Trio(kvq, torch, 2, 8, 32, 128, 128, 32, 1, 1500, pool_blocks=80, seed=34, spikes=True)
    for rnd in range(3):
        trio.append(0, 300)
        trio.append(1, 170)
    trio.append(0, 1)
    trio.append(1, 1)
    trio.attend(0)
    trio.check(0)
    trio.check(1)
