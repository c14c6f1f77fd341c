"""The segmented cache on the GPU: the datawhale page's flush rule
(append_and_partition, the whole overflow of an append as one segment)
against the oracle's page rule (``group=None``), and the page's mechanism
checks run on the GPU path.  The cache needs head_dim >= 16, so the page's
tiny shapes use head_dim 16 with the page's token schedules.

Codes, scales and counters bit-exact; restore bit-exact (fp32); attention
within |d| <= 1e-3 + 1e-2 |ref|.
"""

import numpy as np
import pytest

from kvq_inputs import gen
from oracle import kvq_oracle as O

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


def _r(*shape, seed=0):
    return np.random.default_rng(seed).standard_normal(shape).astype(np.float32)


class SegPair:
    """A segmented GPU cache (batch 1) and the oracle's page-rule state."""

    def __init__(self, kvq, torch, Hkv, Hq, D, R, qmax=7, capacity=512, dtype="fp32"):
        self.torch = torch
        self.tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
        self.cache = kvq.KVQCache(1, Hkv, Hq, D, R, 8, qmax, capacity, dtype=dtype, segmented=True)
        self.state = None
        self.R, self.qmax = R, qmax

    def append(self, k, v):
        """k, v: [Hkv, n, D] fp32 (values representable in the cache dtype)."""
        dev = lambda a: self.torch.from_numpy(np.ascontiguousarray(a[None])).to("cuda").to(self.tdt).contiguous()
        self.cache.append(dev(k), dev(v), 0)
        self.state = O.append_and_partition(self.state, k[None], v[None], self.R, self.qmax, group=None)

    def check_unit(self, h):
        st = self.cache.seq_state(0)
        assert (st["total"], st["quantized"]) == (self.state["total_tokens"], self.state["quantized_tokens"])
        assert st["n_groups"] == len(self.state["key_q_segments"])
        got = self.cache.export_unit(0, h)
        if st["quantized"]:
            kq = np.concatenate([s[0, h] for s in self.state["key_q_segments"]], axis=0)
            vq = np.concatenate([s[0, h] for s in self.state["value_q_segments"]], axis=0)
            ks = np.stack([s[0, h, 0] for s in self.state["key_scale_segments"]])
            vs = np.concatenate([s[0, h, :, 0] for s in self.state["value_scale_segments"]])
            np.testing.assert_array_equal(got["k_codes"], kq)
            np.testing.assert_array_equal(got["v_codes"], vq)
            np.testing.assert_array_equal(got["k_scales"].view(np.uint32), ks.view(np.uint32))
            np.testing.assert_array_equal(got["v_scales"].view(np.uint32), vs.view(np.uint32))
        np.testing.assert_array_equal(got["window_k"], self.state["key_residual"][0, h])
        np.testing.assert_array_equal(got["window_v"], self.state["value_residual"][0, h])
        return got

    def attend(self, q, kernels=(0,)):
        qd = self.torch.from_numpy(np.ascontiguousarray(q[None])).to("cuda").to(self.tdt).contiguous()
        ref = O.decode_attention(self.state, q[None])[0]
        for kernel in kernels:
            got = self.cache.decode_attention(qd, kernel=kernel).cpu().numpy()[0].astype(np.float64)
            excess = np.abs(got - ref) - (ATOL + RTOL * np.abs(ref))
            assert excess.max() <= 0, f"kernel {kernel}: |d| {np.abs(got - ref).max():.3e}"


# ---- the page's mechanism checks, on the GPU path --------------------------

def test_segment_scale_axes(kvq, torch):
    """Key: one scale per channel over the segment; Value: one per token."""
    pair = SegPair(kvq, torch, 2, 2, 16, 2)
    pair.append(_r(2, 5, 16), _r(2, 5, 16, seed=1))   # 3 tokens flush as one segment
    for h in range(2):
        got = pair.check_unit(h)
        assert got["k_scales"].shape == (1, 16) and got["v_scales"].shape == (3,)


def test_segment_token_conservation(kvq, torch):
    pair = SegPair(kvq, torch, 2, 2, 16, 4)
    pair.append(_r(2, 3, 16), _r(2, 3, 16, seed=1))
    pair.append(_r(2, 2, 16, seed=2), _r(2, 2, 16, seed=3))
    st = pair.cache.seq_state(0)
    assert st["total"] == 5 and st["quantized"] + st["window"] == 5
    for h in range(2):
        pair.check_unit(h)


def test_segment_partition_residual_two(kvq, torch):
    pair = SegPair(kvq, torch, 2, 2, 16, 2)
    pair.append(_r(2, 3, 16), _r(2, 3, 16, seed=1))
    pair.append(_r(2, 2, 16, seed=2), _r(2, 2, 16, seed=3))
    st = pair.cache.seq_state(0)
    assert (st["quantized"], st["window"], st["n_groups"]) == (3, 2, 2)
    for h in range(2):
        pair.check_unit(h)


def test_segment_prefix_not_rewritten(kvq, torch):
    pair = SegPair(kvq, torch, 1, 1, 16, 2)
    pair.append(_r(1, 3, 16), _r(1, 3, 16, seed=1))
    first = pair.check_unit(0)
    pair.append(_r(1, 2, 16, seed=2) * 100, _r(1, 2, 16, seed=3))
    after = pair.check_unit(0)
    np.testing.assert_array_equal(after["k_codes"][:1], first["k_codes"])
    np.testing.assert_array_equal(after["k_scales"][:1], first["k_scales"])
    assert pair.cache.seq_state(0)["last_flushed"] == 2


def test_segment_no_overflow(kvq, torch):
    pair = SegPair(kvq, torch, 1, 1, 16, 4)
    pair.append(_r(1, 1, 16), _r(1, 1, 16, seed=1))
    pair.append(_r(1, 1, 16, seed=2), _r(1, 1, 16, seed=3))
    st = pair.cache.seq_state(0)
    assert (st["quantized"], st["last_flushed"], st["window"]) == (0, 0, 2)
    pair.check_unit(0)
    pair.attend(_r(1, 16, seed=4))


def test_segment_zero_range(kvq, torch):
    pair = SegPair(kvq, torch, 2, 2, 16, 2)
    z = np.zeros((2, 6, 16), np.float32)
    pair.append(z, z)
    got = pair.check_unit(0)
    assert np.isfinite(got["k_scales"]).all() and not got["k_codes"].any()
    pair.attend(_r(2, 16, seed=5))


def test_segment_ledger(kvq, torch):
    pair = SegPair(kvq, torch, 2, 2, 16, 4, qmax=7)
    pair.append(_r(2, 10, 16), _r(2, 10, 16, seed=1))       # segment of 6
    pair.append(_r(2, 3, 16, seed=2), _r(2, 3, 16, seed=3))  # segment of 3
    led = pair.cache.bytes()
    Q, W = 9, 4
    assert led["code_bytes"] == 2 * 2 * Q * 16 // 2
    assert led["n_scales"] == 2 * (2 * 16 + Q)
    assert led["window_elems"] == 2 * 2 * W * 16


def test_segment_validation(kvq, torch):
    with pytest.raises(kvq.KVQError) as e:
        kvq.KVQCache(1, 1, 1, 16, 0, 8, 7, 64, dtype="fp32", segmented=True)   # R <= 0
    assert e.value.status == kvq.binding.KVQ_EINVAL
    pair = SegPair(kvq, torch, 1, 1, 16, 2)
    with pytest.raises(kvq.KVQError) as e:
        kvq.kvq_append(pair.cache.handle, 0, 0, 1, 0, 1, 0)                       # NULL inputs
    assert e.value.status == kvq.binding.KVQ_EINVAL
    with pytest.raises(kvq.KVQError) as e:
        kvq.kvq_export_pages(pair.cache.handle, 0, 0, 0, 0, 0)
    assert e.value.status == kvq.binding.KVQ_EUNSUPPORTED


# ---- longer schedules: codes, restore and attention -----------------------

@pytest.mark.parametrize("dtype,qmax,D", [("fp32", 7, 64), ("bf16", 7, 128), ("bf16", 127, 64), ("fp32", 1, 32)])
def test_segment_schedule_matches_oracle(kvq, torch, dtype, qmax, D):
    Hkv, Hq, R = 4, 8, 32
    spec = gen.InputSpec(seed=41, n_kv_heads=Hkv, n_q_heads=Hq, head_dim=D, bf16=dtype == "bf16", spikes=True)
    pair = SegPair(kvq, torch, Hkv, Hq, D, R, qmax=qmax, capacity=400, dtype=dtype)
    t = 0
    for n in [100] + [1] * 12 + [50, 7, 1, 1, 70]:
        k, v = spec.kv_block(0, [0], t, n)
        t += n
        pair.append(k[0], v[0])
        if n != 1 or t % 5 == 0:
            pair.attend(spec.q_block(0, [0], t)[0])
    for h in range(Hkv):
        pair.check_unit(h)
    k_out, v_out = pair.cache.restore(out_dtype="fp32")
    K, V = O.restored_kv(pair.state)
    np.testing.assert_array_equal(k_out.cpu().numpy()[0].view(np.uint32), K[0].view(np.uint32))
    np.testing.assert_array_equal(v_out.cpu().numpy()[0].view(np.uint32), V[0].view(np.uint32))
    assert pair.cache.device_status() == 0


@pytest.mark.parametrize("dtype,D,Hkv,Hq", [("bf16", 128, 2, 16), ("bf16", 128, 2, 12), ("bf16", 256, 2, 8),
                                            ("fp32", 16, 2, 2), ("bf16", 256, 1, 6)])
def test_segment_head_groups(kvq, torch, dtype, D, Hkv, Hq):
    """The segmented decode sums each pass's (token, head) dot products over
    the warp in sets of four heads: eight and six query heads per KV head take
    two sets (the second partly padding), one head pads a single set, and
    head_dim 256 runs one token per pass (sets of four values)."""
    R = 32
    spec = gen.InputSpec(seed=43, n_kv_heads=Hkv, n_q_heads=Hq, head_dim=D, bf16=dtype == "bf16", spikes=True)
    pair = SegPair(kvq, torch, Hkv, Hq, D, R, qmax=7, capacity=400, dtype=dtype)
    t = 0
    for n in [90, 1, 1, 40, 1, 3, 1, 60]:
        k, v = spec.kv_block(0, [0], t, n)
        t += n
        pair.append(k[0], v[0])
        pair.attend(spec.q_block(0, [0], t)[0])
    for h in range(Hkv):
        pair.check_unit(h)
    assert pair.cache.device_status() == 0


@pytest.mark.parametrize("D,Hkv,Hq", [(128, 2, 8), (128, 2, 16), (64, 2, 4), (128, 1, 8)])
def test_segment_tensor_cores(kvq, torch, D, Hkv, Hq):
    """4-bit bf16 segmented caches on the tensor-core kernel (kernel 2; the
    automatic choice, 0, takes it too) and on the CUDA-core kernel (1): a long
    first segment (whole 32-token tiles on the tensor cores), its partial last
    tile, one-token segments (tiles of many Key scale rows, on the CUDA cores
    inside the same kernel), segments that begin and end inside a tile, and a
    decode after each kind of append."""
    R = 64
    spec = gen.InputSpec(seed=47, n_kv_heads=Hkv, n_q_heads=Hq, head_dim=D, spikes=True)
    pair = SegPair(kvq, torch, Hkv, Hq, D, R, qmax=7, capacity=2400, dtype="bf16")
    t = 0
    for n in [700] + [1] * 37 + [45, 1, 1, 1, 1, 333, 96, 1, 1, 640]:
        k, v = spec.kv_block(0, [0], t, n)
        t += n
        pair.append(k[0], v[0])
        if n != 1 or t % 9 == 0:
            pair.attend(spec.q_block(0, [0], t)[0], kernels=(0, 1, 2))
    for h in range(Hkv):
        pair.check_unit(h)
    assert pair.cache.device_status() == 0


def test_segment_tensor_cores_batch(kvq, torch):
    """A batch of segmented sequences of different lengths (one empty, one
    with only a window) on the tensor-core kernel against the oracle."""
    H, Hq, D, R = 4, 16, 128, 64
    lens = [[1000, 1, 1, 70], [], [30], [64, 1, 1, 1, 2000]]
    spec = gen.InputSpec(seed=48, n_kv_heads=H, n_q_heads=Hq, head_dim=D, spikes=True)
    cache = kvq.KVQCache(len(lens), H, Hq, D, R, 8, 7, [sum(x) + 8 for x in lens], segmented=True)
    states = [None] * len(lens)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda().bfloat16()
    for b, chunks in enumerate(lens):
        t = 0
        for n in chunks:
            k, v = spec.kv_block(0, [b], t, n)
            t += n
            cache.append(dev(k), dev(v), b)
            states[b] = O.append_and_partition(states[b], k, v, R, 7, group=None)
    q = spec.q_block(0, range(len(lens)), 0)
    for kernel in (0, 2):
        got = cache.decode_attention(dev(q), kernel=kernel).cpu().numpy().astype(np.float64)
        for b in range(len(lens)):
            if states[b] is None:
                assert not got[b].any()
                continue
            ref = O.decode_attention(states[b], q[b][None])[0]
            excess = np.abs(got[b] - ref) - (ATOL + RTOL * np.abs(ref))
            assert excess.max() <= 0, f"kernel {kernel} seq {b}: |d| {np.abs(got[b] - ref).max():.3e}"
    assert cache.device_status() == 0


@pytest.mark.parametrize("vmag,kmag", [(6e4, 1.0), (1.0, 1e6), (300.0, 1e4)])
def test_segment_tensor_cores_input_range(kvq, torch, vmag, kmag):
    """Inputs beyond the tensor-core operands' range on a segmented cache
    (Value rows of absmax up to 6e4; Key spikes up to 1e6 against q x 24):
    the segment flush records the unit's maxima and the decode takes the
    CUDA-core path for such units inside the same launch; every kernel
    against the oracle."""
    Hkv, Hq, D, R = 2, 8, 128, 64
    spec = gen.InputSpec(seed=49, n_kv_heads=Hkv, n_q_heads=Hq, head_dim=D)
    pair = SegPair(kvq, torch, Hkv, Hq, D, R, qmax=7, capacity=1200, dtype="bf16")
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).bfloat16().float().numpy()
    t = 0
    for n in [600, 1, 1, 200]:
        k, v = spec.kv_block(0, [0], t, n)
        k, v = k[0].copy(), v[0].copy()
        v[:, ::8] *= vmag                  # every 8th token
        k[:, ::5, 3] *= kmag               # one channel of every 5th token
        t += n
        pair.append(bf(k), bf(v))
        q = spec.q_block(0, [0], t)[0] * (24.0 if kmag > 1 else 1.0)
        pair.attend(bf(q), kernels=(0, 1, 2))
    assert pair.cache.device_status() == 0
