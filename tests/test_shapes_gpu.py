"""GPU parity across the shapes the main workloads do not reach: head_dim
16..256 (the combine then holds one or two 16-byte pieces of o per lane, or
lanes without any), batches above the 256 sequences one launch holds, eight
query heads per KV head and a padded GQA group on the tensor cores, and larger
groups staged in 32-token units.  Codes and scales bit-exact; attention within
|d| <= 1e-3 + 1e-2 |ref| of the fp64 oracle.
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


def close(got, ref, what):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite"
    excess = np.abs(got - ref) - (ATOL + RTOL * np.abs(ref))
    assert excess.max() <= 0, f"{what}: |d| {np.abs(got - ref).max():.3e}"


def run_case(kvq, torch, lens, Hkv, Hq, D, R, G, qmax, dtype, kernels, seed, check_heads=(0,), steps=2, chunks=(0,)):
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    spec = gen.InputSpec(seed=seed, n_kv_heads=Hkv, n_q_heads=Hq, head_dim=D, bf16=dtype == "bf16")
    cache = kvq.KVQCache(len(lens), Hkv, Hq, D, R, G, qmax, [n + steps + 1 for n in lens], dtype=dtype)
    seqs = [O.GroupedSequence(Hkv, D, R, G, qmax) for _ in lens]
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to("cuda").to(tdt).contiguous()
    for b, n in enumerate(lens):
        if n:
            k, v = spec.kv_block(0, [b], 0, n)
            cache.append(dev(k), dev(v), b)
            seqs[b].append(k[0], v[0])
    B = len(lens)
    for s in range(steps):
        k = np.stack([spec.kv_block(0, [b], lens[b] + s, 1)[0][0] for b in range(B)])
        v = np.stack([spec.kv_block(0, [b], lens[b] + s, 1)[1][0] for b in range(B)])
        cache.append(dev(k), dev(v), 0)
        for b in range(B):
            seqs[b].append(k[b], v[b])
    q = spec.q_block(0, range(B), steps)
    refs = [seq.attend(q[b]) for b, seq in enumerate(seqs)]
    for kernel in kernels:
        for chunk in chunks:
            out = cache.decode_attention(dev(q), kernel=kernel, chunk_pages=chunk).cpu().numpy()
            for b, seq in enumerate(seqs):
                close(out[b], refs[b], f"kernel {kernel} chunk {chunk} seq {b} (T={seq.total})")
    for b in {0, B - 1}:
        for h in check_heads:
            got = cache.export_unit(b, h)
            np.testing.assert_array_equal(got["k_codes"], seqs[b].key_codes()[h])
            np.testing.assert_array_equal(got["v_codes"], seqs[b].value_codes()[h])
            np.testing.assert_array_equal(got["k_scales"].view(np.uint32), seqs[b].key_scales()[h].view(np.uint32))
    assert cache.device_status() == 0


@pytest.mark.parametrize("D", [16, 48, 80, 192, 256])
@pytest.mark.parametrize("qmax", [7, 127])
def test_head_dims_cuda_cores(kvq, torch, D, qmax):
    run_case(kvq, torch, [200, 77, 131], 2, 4, D, 32, 16, qmax, "fp32", kernels=(0, 1), seed=61)


def test_head_dim_256_bf16_two_bit(kvq, torch):
    run_case(kvq, torch, [300, 95], 2, 6, 256, 64, 32, 1, "bf16", kernels=(0,), seed=62)


def test_batch_above_one_launch(kvq, torch):
    """300 sequences: the decode runs as two launches of 256 and 44."""
    lens = [(37 * b) % 150 + (b % 3) * 64 for b in range(300)]
    run_case(kvq, torch, lens, 2, 4, 64, 32, 32, 7, "bf16", kernels=(0, 1, 2, 4), seed=63, steps=1)


@pytest.mark.parametrize("Hq", [16, 24, 64])
def test_gqa_on_tensor_cores(kvq, torch, Hq):
    """g = 2, 3 (padded to 4) and 8 query heads per KV head on the mma.sync kernel."""
    run_case(kvq, torch, [700, 1234], 8, Hq, 128, 128, 32, 7, "bf16", kernels=(2, 4), seed=64, check_heads=(0, 7))


@pytest.mark.parametrize("G", [64, 256])
def test_large_groups_staged(kvq, torch, G):
    run_case(kvq, torch, [G * 5 + 129, G + 128, 100], 4, 16, 64, 128, G, 7, "bf16", kernels=(1, 2, 4), seed=65)


@pytest.mark.parametrize("G", [32, 128])
def test_odd_chunks_tensor_cores(kvq, torch, G):
    """Split items of odd page counts on the mma.sync kernel (as the whole-wave
    plan picks for long staged units): each warp's run ends on a one-page group."""
    run_case(kvq, torch, [G * 9 + 50, G * 4 + 3, 130], 4, 16, 128, 128, G, 7, "bf16", kernels=(2, 4), seed=66,
             chunks=(0, 1, 3, 5, 7))


@pytest.mark.parametrize("chunk", [0, 2, 8, 40])
def test_in_launch_merge_and_combine_kernel(kvq, torch, chunk):
    """A short decode (one wave, items of at most 16 pages: automatic, 2 and
    8 pages an item) merges each unit's partials in its last finishing CTA; a
    decode of 40-page items merges in the combine kernel.  Batch 3 with an
    empty sequence, a window-only sequence and a 4096-token one, decoded
    three times in a row (the arrival counts must come back to zero), each
    against the oracle."""
    H, Hq, D, R, G = 8, 32, 128, 128, 32
    lens = [4096, 0, 77]
    spec = gen.InputSpec(seed=67, n_kv_heads=H, n_q_heads=Hq, head_dim=D)
    cache = kvq.KVQCache(len(lens), H, Hq, D, R, G, 7, [n + 8 for n in lens])
    seqs = [O.GroupedSequence(H, D, R, G, 7) for _ in lens]
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda().bfloat16()
    for b, n in enumerate(lens):
        if n:
            k, v = spec.kv_block(0, [b], 0, n)
            cache.append(dev(k), dev(v), b)
            seqs[b].append(k[0], v[0])
    for rep in range(3):
        q = spec.q_block(0, range(len(lens)), rep)
        out = cache.decode_attention(dev(q), kernel=2, chunk_pages=chunk).cpu().numpy()
        assert not out[1].any(), "a sequence without tokens attends to zeros"
        for b in (0, 2):
            close(out[b], seqs[b].attend(q[b]), f"chunk {chunk} decode {rep} seq {b}")
    assert cache.device_status() == 0
