"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.  Codes, scales, counters and raw page bytes must match bit
for bit; attention outputs within |d| <= 1e-3 + 1e-2 |ref| (bf16 or fp32
inputs, fp32 accumulation, fp64 oracle)."""

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


def assert_attention_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    excess = np.abs(got - ref) - (ATOL + RTOL * np.abs(ref))
    worst = np.unravel_index(np.argmax(excess), excess.shape)
    assert excess.max() <= 0, (f"{what}: |d| = {abs(got - ref)[worst]:.3e} at {worst} "
                               f"(ref {ref[worst]:.4e}, got {got[worst]:.4e})")


class Pair:
    """A GPU cache and the oracle sequences fed the same inputs."""

    def __init__(self, kvq, torch, batch, Hkv, Hq, D, R, G, qmax, capacity, dtype="bf16"):
        self.torch = torch
        self.cache = kvq.KVQCache(batch, Hkv, Hq, D, R, G, qmax, capacity, dtype=dtype)
        self.seqs = [O.GroupedSequence(Hkv, D, R, G, qmax) for _ in range(batch)]
        self.tdtype = torch.bfloat16 if dtype == "bf16" else torch.float32
        self.D, self.G, self.Hkv, self.Hq, self.qmax = D, G, Hkv, Hq, qmax

    def to_dev(self, a):
        return self.torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to("cuda").to(self.tdtype).contiguous()

    def append(self, k, v, seq_begin=0):
        """k, v: host fp32 [n_seqs, Hkv, n, D] (values representable in the dtype)."""
        self.cache.append(self.to_dev(k), self.to_dev(v), seq_begin)
        for i in range(k.shape[0]):
            self.seqs[seq_begin + i].append(k[i], v[i])

    def attend(self, q, kernel=0, seqs=None):
        out = self.cache.decode_attention(self.to_dev(q), kernel=kernel).cpu().numpy()
        seqs = range(len(self.seqs)) if seqs is None else seqs
        ref = np.stack([self.seqs[b].attend(q[b]) for b in seqs])
        return out[list(seqs)], ref

    def check_unit(self, b, h):
        seq = self.seqs[b]
        st = self.cache.seq_state(b)
        assert (st["total"], st["quantized"], st["window"]) == (seq.total, seq.quantized, seq.window)
        got = self.cache.export_unit(b, h)
        np.testing.assert_array_equal(got["k_codes"], seq.key_codes()[h])
        np.testing.assert_array_equal(got["v_codes"], seq.value_codes()[h])
        np.testing.assert_array_equal(got["k_scales"].view(np.uint32), seq.key_scales()[h].view(np.uint32))
        np.testing.assert_array_equal(got["v_scales"].view(np.uint32), seq.value_scales()[h].view(np.uint32))
        wk, wv = seq.window_kv()
        np.testing.assert_array_equal(got["window_k"], wk[h])
        np.testing.assert_array_equal(got["window_v"], wv[h])
        # raw bytes of every group page against the layout encoder
        bits = O.code_bits(self.qmax)
        raw = self.cache.export_pages(b, h)
        G = self.G
        expect = b"".join(
            L.pack_group_page(seq.key_codes()[h][j * G:(j + 1) * G], seq.value_codes()[h][j * G:(j + 1) * G],
                              seq.key_scales()[h][j], seq.value_scales()[h][j * G:(j + 1) * G], bits)
            for j in range(seq.quantized // G))
        assert raw == expect

    def status_ok(self):
        assert self.cache.device_status() == 0


# --------------------------------------------------------------------------
# input generator: the device fill equals the host generator bit for bit
# --------------------------------------------------------------------------

@pytest.mark.parametrize("bf16,spikes", [(True, False), (True, True), (False, False)])
def test_device_inputs_match_host(torch, bf16, spikes):
    from kvq_inputs.device import DeviceInputs
    spec = gen.InputSpec(seed=11, n_kv_heads=8, n_q_heads=32, head_dim=128, bf16=bf16, spikes=spikes)
    dev = DeviceInputs(spec)
    K, V = dev.kv_block(layer=3, seq_begin=2, nseq=2, t0=1000, n=333)
    Kh, Vh = spec.kv_block(layer=3, seqs=[2, 3], t0=1000, n=333)
    np.testing.assert_array_equal(K.float().cpu().numpy(), Kh)
    np.testing.assert_array_equal(V.float().cpu().numpy(), Vh)
    q = dev.q_block(layer=3, seq_begin=0, nseq=4, step=7)
    np.testing.assert_array_equal(q.float().cpu().numpy(), spec.q_block(layer=3, seqs=range(4), step=7))


# --------------------------------------------------------------------------
# tiny fp32 case: every code, scale, counter and every step's attention
# --------------------------------------------------------------------------

def test_tiny_fp32_schedule(kvq, torch):
    spec = gen.InputSpec(seed=0, n_kv_heads=2, n_q_heads=2, head_dim=16, bf16=False)
    pair = Pair(kvq, torch, 1, 2, 2, 16, 8, 8, 7, 64, dtype="fp32")
    k, v = spec.kv_block(0, [0], 0, 40)
    pair.append(k, v)
    assert pair.cache.seq_state(0)["quantized"] == 32 and pair.cache.seq_state(0)["window"] == 8
    for step in range(24):
        k, v = spec.kv_block(0, [0], 40 + step, 1)
        pair.append(k, v)
        for h in range(2):
            pair.check_unit(0, h)
        q = spec.q_block(0, [0], step)
        for kernel in (0, 1):
            got, ref = pair.attend(q, kernel=kernel)
            assert_attention_close(got, ref, f"step {step} kernel {kernel}")
    st = pair.cache.seq_state(0)
    assert (st["total"], st["quantized"], st["window"], st["n_groups"]) == (64, 56, 8, 7)
    pair.status_ok()


# --------------------------------------------------------------------------
# Llama-3-8B single layer, batch 1, 4096 context, 4-bit, R=128, G=32
# --------------------------------------------------------------------------

def test_llama_single_layer(kvq, torch):
    spec = gen.InputSpec(seed=1, n_kv_heads=8, n_q_heads=32, head_dim=128)
    pair = Pair(kvq, torch, 1, 8, 32, 128, 128, 32, 7, 4096 + 64)
    k, v = spec.kv_block(0, [0], 0, 4096)
    pair.append(k, v)
    for h in range(8):
        pair.check_unit(0, h)
    for step in range(40):
        k, v = spec.kv_block(0, [0], 4096 + step, 1)
        pair.append(k, v)
        if step % 8 == 0 or step in (31, 32, 39):
            q = spec.q_block(0, [0], step)
            for kernel in (1, 2, 4):
                got, ref = pair.attend(q, kernel=kernel)
                assert_attention_close(got, ref, f"step {step} kernel {kernel}")
    for h in range(8):
        pair.check_unit(0, h)
    assert pair.cache.seq_state(0)["n_groups"] == 125
    pair.status_ok()


# --------------------------------------------------------------------------
# 8-bit ragged batch, G=64 (lengths reduced so that every unit is compared)
# --------------------------------------------------------------------------

def test_ragged_8bit(kvq, torch):
    spec = gen.InputSpec(seed=3, n_kv_heads=8, n_q_heads=32, head_dim=128, spikes=True)
    lens = spec.lengths(4, 300, 3000)
    pair = Pair(kvq, torch, 4, 8, 32, 128, 128, 64, 127, [n + 16 for n in lens])
    for b, n in enumerate(lens):
        k, v = spec.kv_block(0, [b], 0, n)
        pair.append(k, v, seq_begin=b)
    for step in range(3):
        k, v = spec.kv_block(0, range(4), 0, 1)
        k = np.stack([spec.kv_block(0, [b], lens[b] + step, 1)[0][0] for b in range(4)])
        v = np.stack([spec.kv_block(0, [b], lens[b] + step, 1)[1][0] for b in range(4)])
        pair.append(k, v)
        q = spec.q_block(0, range(4), step)
        for kernel in (1, 2, 4):
            got, ref = pair.attend(q, kernel=kernel)
            assert_attention_close(got, ref, f"step {step} kernel {kernel}")
    for b in range(4):
        for h in (0, 7):
            pair.check_unit(b, h)
    pair.status_ok()


# --------------------------------------------------------------------------
# 2-bit codes (KIVI's 2-bit, qmax = 1): tiny fp32 schedule on the CUDA-core
# kernel, Llama head shape ragged on both kernels, head_dim 64
# --------------------------------------------------------------------------

def test_two_bit_tiny_fp32(kvq, torch):
    spec = gen.InputSpec(seed=21, n_kv_heads=2, n_q_heads=4, head_dim=16, bf16=False)
    pair = Pair(kvq, torch, 1, 2, 4, 16, 8, 8, 1, 64, dtype="fp32")
    k, v = spec.kv_block(0, [0], 0, 37)
    pair.append(k, v)
    for step in range(12):
        k, v = spec.kv_block(0, [0], 37 + step, 1)
        pair.append(k, v)
        for h in range(2):
            pair.check_unit(0, h)
        got, ref = pair.attend(spec.q_block(0, [0], step), kernel=1)
        assert_attention_close(got, ref, f"2-bit step {step}")
    pair.status_ok()


@pytest.mark.parametrize("D,G,qmax", [(128, 32, 1), (64, 64, 1), (128, 96, 1), (128, 32, 7)])
def test_two_bit_ragged_both_kernels(kvq, torch, D, G, qmax):
    """Ragged lengths with Key spikes (x50 entries); qmax 7 runs the same case
    with 4-bit codes."""
    spec = gen.InputSpec(seed=22, n_kv_heads=8, n_q_heads=32, head_dim=D, spikes=True)
    lens = [G * 9 + 5, 3 * G + 128 + 1, 40, 2000]
    pair = Pair(kvq, torch, 4, 8, 32, D, 128, G, qmax, [n + 8 for n in lens])
    for b, n in enumerate(lens):
        k, v = spec.kv_block(0, [b], 0, n)
        pair.append(k, v, seq_begin=b)
    for step in range(3):
        k = np.stack([spec.kv_block(0, [b], lens[b] + step, 1)[0][0] for b in range(4)])
        v = np.stack([spec.kv_block(0, [b], lens[b] + step, 1)[1][0] for b in range(4)])
        pair.append(k, v)
        q = spec.q_block(0, range(4), step)
        for kernel in (1, 2, 4):
            got, ref = pair.attend(q, kernel=kernel)
            assert_attention_close(got, ref, f"qmax {qmax} D {D} G {G} step {step} kernel {kernel}")
    for b in range(4):
        for h in (0, 5):
            pair.check_unit(b, h)
    pair.status_ok()


# --------------------------------------------------------------------------
# chunked prefill (long-video shape, reduced length) and chunking invariance
# --------------------------------------------------------------------------

def test_chunked_prefill_and_invariance(kvq, torch):
    spec = gen.InputSpec(seed=4, n_kv_heads=8, n_q_heads=32, head_dim=128)
    T = 3 * 1440 + 77
    k, v = spec.kv_block(0, [0], 0, T)
    caches = []
    for chunks in ([1440, 1440, 1440, 77], [T], [7] * (T // 7) + [T % 7]):
        pair = Pair(kvq, torch, 1, 8, 32, 128, 256, 128, 7, T)
        pos = 0
        for n in chunks:
            if n == 0:
                continue
            pair.append(k[:, :, pos:pos + n], v[:, :, pos:pos + n])
            pos += n
        caches.append(pair)
    first = caches[0]
    for h in range(8):
        first.check_unit(0, h)
    for other in caches[1:]:
        for h in (0, 3, 7):
            assert other.cache.export_pages(0, h) == first.cache.export_pages(0, h)
            a, b = other.cache.export_unit(0, h), first.cache.export_unit(0, h)
            np.testing.assert_array_equal(a["window_k"], b["window_k"])
    q = spec.q_block(0, [0], 0)
    for kernel in (1, 2, 4):
        got, ref = first.attend(q, kernel=kernel)
        assert_attention_close(got, ref, f"kernel {kernel}")
    first.status_ok()


# --------------------------------------------------------------------------
# edge cases
# --------------------------------------------------------------------------

def test_edge_cases(kvq, torch):
    spec = gen.InputSpec(seed=5, n_kv_heads=8, n_q_heads=32, head_dim=128)
    pair = Pair(kvq, torch, 3, 8, 32, 128, 128, 32, 7, [1000, 1000, 1000])
    # sequence 0 stays empty -> zeros; sequence 1 holds only a window (no flush yet)
    k, v = spec.kv_block(0, [1], 0, 150)
    pair.append(k, v, seq_begin=1)
    assert pair.cache.seq_state(1)["quantized"] == 0
    # sequence 2: one append larger than the ring that also flushes (two launches)
    k2, v2 = spec.kv_block(0, [2], 0, 100)
    pair.append(k2, v2, seq_begin=2)
    k3, v3 = spec.kv_block(0, [2], 100, 500)
    pair.append(k3, v3, seq_begin=2)
    assert pair.cache.seq_state(2)["last_flushed"] == 448
    for h in range(8):
        pair.check_unit(1, h)
        pair.check_unit(2, h)
    q = spec.q_block(0, range(3), 0)
    for kernel in (1, 2, 4):
        got, ref = pair.attend(q, kernel=kernel, seqs=[0, 1, 2])
        assert not got[0].any()
        assert_attention_close(got[1:], ref[1:], f"kernel {kernel}")
    # the window-only sequence attends its raw values exactly as the plain formula
    kk = k[0].transpose(1, 0, 2)
    np.testing.assert_allclose(ref[1], O.attn_step(q[1], kk, v[0].transpose(1, 0, 2)), rtol=1e-12, atol=1e-12)
    # errors leave the state unchanged
    with pytest.raises(kvq.KVQError) as e:
        pair.append(*[np.zeros((1, 8, 600, 128), np.float32)] * 2, seq_begin=2)
    assert e.value.status == kvq.binding.KVQ_ECAPACITY
    assert pair.cache.seq_state(2)["total"] == 600
    with pytest.raises(kvq.KVQError):
        kvq.kvq_append(pair.cache.handle, 16, 16, 0, 0, 1, 0)
    with pytest.raises(kvq.KVQError):
        kvq.kvq_append(pair.cache.handle, 16, 16, 1, 2, 2, 0)
    pair.status_ok()
