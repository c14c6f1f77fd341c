"""GPU parity at the edges of the value range, on every decode kernel.

The tensor-core kernels carry q / sK and p / sV as f16 MMA operands and, for
4- and 8-bit codes, take the offset bias of the stored codes out in fp32.
These cases drive both past the plain path: Value rows whose absmax reaches
1e3, 1e4 and 6e4 (whole rows, and single channels of a row), 2-bit Values
beyond 256, Key spikes of 1e4 against queries up to 100 and of 1e6 against
plain queries, and Key and Value groups whose absmax exceeds qmax / eps, where
the scale falls below eps and the page's restore divides by eps instead
("54. KV Cache Quantization Strategies", Step 4 ``restore``:
``scale.clamp_min(eps)``).  The oracle restores and attends in fp32 / fp64;
attention must stay within |d| <= 1e-3 + 1e-2 |ref| and finite, and the
device status word 0.

Inputs are the seeded generator's K, V and q, multiplied by fixed per-token /
per-channel factors and rounded to bf16 once (the values both sides see).
"""

import numpy as np
import pytest

from kvq_inputs import gen
from oracle import kvq_oracle as O

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-3, 1e-2
H, HQ, D, R, G = 2, 8, 128, 64, 32
LENS = [300, 517, 64 + 3 * 32 + 5]


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


def bf16(torch, a):
    """Round an fp32 array to the nearest bf16 (ties to even), as fp32."""
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).bfloat16().float().numpy()


def close(got, ref, what):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    excess = np.abs(got - ref) - (ATOL + RTOL * np.abs(ref))
    w = np.unravel_index(np.argmax(excess), excess.shape)
    assert excess.max() <= 0, f"{what}: |d| {abs(got - ref)[w]:.3e} at {w} (ref {ref[w]:.4e}, got {got[w]:.4e})"


def run_case(kvq, torch, qmax, kmul, vmul, qmul, seed, kernels, what):
    """kmul / vmul(b, t) -> factors broadcastable to [H, len(t), D]; qmul -> [HQ, D]."""
    spec = gen.InputSpec(seed=seed, n_kv_heads=H, n_q_heads=HQ, head_dim=D)
    cache = kvq.KVQCache(len(LENS), H, HQ, D, R, G, qmax, [n + 8 for n in LENS])
    seqs = [O.GroupedSequence(H, D, R, G, qmax) for _ in LENS]
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda().bfloat16()
    for b, n in enumerate(LENS):
        k, v = spec.kv_block(0, [b], 0, n)
        t = np.arange(n)
        k = bf16(torch, k[0] * kmul(b, t))
        v = bf16(torch, v[0] * vmul(b, t))
        # two appends: a prefill and the last token alone (a decode step)
        cache.append(dev(k[None, :, :-1]), dev(v[None, :, :-1]), b)
        cache.append(dev(k[None, :, -1:]), dev(v[None, :, -1:]), b)
        seqs[b].append(k[:, :-1], v[:, :-1])
        seqs[b].append(k[:, -1:], v[:, -1:])
    q = bf16(torch, spec.q_block(0, range(len(LENS)), 0) * qmul)
    ref = np.stack([seqs[b].attend(q[b]) for b in range(len(LENS))])
    for kernel in kernels:
        out = cache.decode_attention(dev(q), kernel=kernel).cpu().numpy()
        close(out, ref, f"{what}, kernel {kernel}")
    assert cache.device_status() == 0


def kernels_for(qmax):
    # 0 automatic, 1 CUDA cores, 2 mma.sync tensor cores, 3 tcgen05 (4-bit
    # only), 4 persistent-warp mma.sync
    return (0, 1, 2, 3, 4) if qmax == 7 else (0, 1, 2, 4)


def ones(b, t):
    return np.ones((1, len(t), 1), np.float32)


# the generator's Value rows have absmax up to about 8.6 (|z| <= 4.3, tau <= 2):
# a factor mag / 8 gives rows with absmax up to about mag
ROW = 1.0 / 8.0


def value_rows(mags):
    """Whole Value rows scaled to absmax about mags[k]: every 5th token by
    mags[0], every 7th by mags[1], every 11th by mags[2] (later factors win),
    so that sub-tiles mix plain and large rows."""
    def f(b, t):
        m = np.ones(len(t), np.float32)
        for period, mag in zip((5, 7, 11), mags):
            m[(t + b) % period == 0] = mag * ROW
        return m[None, :, None]
    return f


@pytest.mark.parametrize("qmax", [7, 127])
@pytest.mark.parametrize("mags", [(1e3, 1e3, 1e3), (1e3, 1e4, 6e4), (6e4, 6e4, 6e4)])
def test_large_value_rows(kvq, torch, qmax, mags):
    run_case(kvq, torch, qmax, ones, value_rows(mags), 1.0, 61, kernels_for(qmax), f"V rows {mags} qmax {qmax}")


@pytest.mark.parametrize("qmax", [7, 127])
def test_large_value_single_channel(kvq, torch, qmax):
    """One channel of some rows at 6e4, the others plain: the row's other
    codes round to 0, so the Value bias term of a large p / sV meets channels
    whose true output is small."""
    def vmul(b, t):
        m = np.ones((1, len(t), D), np.float32)
        m[0, (t + b) % 6 == 1, 17] = 6e4 * ROW
        m[0, (t + b) % 9 == 4, 90] = 2e4 * ROW
        return m
    run_case(kvq, torch, qmax, ones, vmul, 1.0, 62, kernels_for(qmax), f"V channel spikes qmax {qmax}")


@pytest.mark.parametrize("mag", [300.0, 1e3])
def test_two_bit_large_values(kvq, torch, mag):
    run_case(kvq, torch, 1, ones, value_rows((mag, mag, mag)), 1.0, 63, kernels_for(1), f"2-bit V {mag}")


def key_spikes(mag):
    """Channel 5 of one token in every group of G and channel 77 of another.
    One spike a group keeps the spiked channel's other codes at 0, so the
    spike token's huge score term is not shared by tied codes (2-bit codes
    would otherwise tie, and the softmax among them would hang on fp32
    rounding of that term, on any kernel)."""
    def f(b, t):
        m = np.ones((1, len(t), D), np.float32)
        m[0, (t + b) % G == 2, 5] = mag
        m[0, (t + b) % G == 19, 77] = mag
        return m
    return f


@pytest.mark.parametrize("qmax", [7, 127, 1])
def test_key_spikes_1e4_against_large_queries(kvq, torch, qmax):
    # |q| up to ~100 on the generator's discretized normal (|z| <= 4.3)
    run_case(kvq, torch, qmax, key_spikes(1e4), ones, 24.0, 64, kernels_for(qmax), f"K 1e4, q x24, qmax {qmax}")


@pytest.mark.parametrize("qmax", [7, 127, 1])
def test_key_spikes_1e6(kvq, torch, qmax):
    run_case(kvq, torch, qmax, key_spikes(1e6), ones, 1.0, 65, kernels_for(qmax), f"K 1e6, qmax {qmax}")


@pytest.mark.parametrize("qmax", [7, 127])
def test_scales_below_eps(kvq, torch, qmax):
    """Key and Value groups with absmax ~1e9 > qmax / eps: their scales fall
    below eps and restore divides by eps.  Queries are scaled by 2^-27 so
    that the logits stay moderate."""
    def kmul(b, t):
        m = np.ones((1, len(t), D), np.float32)
        m[0, (t // G + b) % 3 == 1, :] = 2.0 ** 30     # whole groups of Keys
        return m

    def vmul(b, t):
        m = np.ones(len(t), np.float32)
        m[(t + b) % 4 == 0] = 2.0 ** 30
        return m[None, :, None]
    run_case(kvq, torch, qmax, kmul, vmul, 2.0 ** -27, 66, kernels_for(qmax), f"scales below eps, qmax {qmax}")



def test_mixed_batch_one_wide_unit(kvq, torch):
    """One sequence with Value rows of absmax 1e4, the others plain: in one
    launch the plain units run on the tensor cores and the wide one on the
    CUDA-core path, and the partials of both merge alike."""
    def vmul(b, t):
        m = np.ones(len(t), np.float32)
        if b == 1:
            m[t % 5 == 0] = 1e4 * ROW
        return m[None, :, None]
    run_case(kvq, torch, 7, ones, vmul, 1.0, 67, kernels_for(7), "one wide sequence")
