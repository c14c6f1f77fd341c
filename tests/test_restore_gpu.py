"""GPU parity of the dequantize-to-HBM path against the oracle:

* ``kvq_restore`` writes the cache as dense tensors: restore(code, scale) rows
  bit-exact against the oracle's ``restored_kv`` (fp32 output), and its
  round-to-nearest-even bf16 rounding for bf16 output;
* ``kvq_dense_decode_attention`` (the foil's standard attention over the
  restored bf16 tensors) within |d| <= 1e-3 + 1e-2 |ref| of the oracle's
  attention over the same bf16 values;
* ``kvq_compare`` against the oracle's ``compare_bytes`` (the page's compare):
  byte counts exact, mean squared errors to 1e-5 relative (both sums add the
  same fp32 squares, in different orders and precisions: fp64 here, numpy's
  pairwise fp32 mean in the oracle).
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


def build(kvq, torch, lens, Hkv, Hq, D, R, G, qmax, dtype, seed, singles=3):
    """A cache and oracle sequences fed the same inputs: per sequence a prefill
    of len - singles tokens, then ``singles`` one-token appends."""
    spec = gen.InputSpec(seed=seed, n_kv_heads=Hkv, n_q_heads=Hq, head_dim=D, bf16=dtype == "bf16")
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    cache = kvq.KVQCache(len(lens), Hkv, Hq, D, R, G, qmax, max(max(lens), 1) + 8, dtype=dtype)
    seqs = [O.GroupedSequence(Hkv, D, R, G, qmax) for _ in lens]
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to("cuda").to(tdt).contiguous()
    for b, n in enumerate(lens):
        cuts = [0] + ([n - singles] if n > singles else []) + list(range(max(n - singles, 0) + 1, n + 1))
        for t0, t1 in zip(cuts[:-1], cuts[1:]):
            if t1 <= t0:
                continue
            k, v = spec.kv_block(0, [b], t0, t1 - t0)
            cache.append(dev(k), dev(v), b)
            seqs[b].append(k[0], v[0])
    return spec, cache, seqs


def oracle_restored(seq):
    """fp32 [heads, total, head_dim] Keys and Values as attention sees them."""
    K, V = O.restored_kv(seq.state)
    return K[0], V[0]


def to_bf16_f32(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).float().numpy()


@pytest.mark.parametrize("dtype,qmax,G,lens", [
    ("fp32", 7, 8, [0, 5, 45, 17]),            # empty, window only, pages + window
    ("bf16", 7, 32, [300, 700]),               # Llama head shape
    ("bf16", 127, 64, [130, 64 * 5 + 128]),    # 8-bit codes, ragged
    ("bf16", 1, 32, [500, 129]),               # 2-bit codes
    ("fp32", 1, 8, [45, 3]),                   # 2-bit codes, fp32 cache
])
def test_restore_fp32_bit_exact(kvq, torch, dtype, qmax, G, lens):
    D, Hkv, Hq, R = (16, 2, 4, 8) if dtype == "fp32" else (128, 8, 32, 128)
    _, cache, seqs = build(kvq, torch, lens, Hkv, Hq, D, R, G, qmax, dtype, seed=5)
    stride = max(lens) + 3
    k, v = cache.restore(t_stride=stride, out_dtype="fp32")
    k, v = k.cpu().numpy(), v.cpu().numpy()
    for b, seq in enumerate(seqs):
        T = seq.total
        assert T == lens[b]
        if T:
            Ko, Vo = oracle_restored(seq)
            np.testing.assert_array_equal(k[b, :, :T].view(np.uint32), Ko.view(np.uint32))
            np.testing.assert_array_equal(v[b, :, :T].view(np.uint32), Vo.view(np.uint32))
        assert not k[b, :, T:].any() and not v[b, :, T:].any(), "rows past the length were written"
    assert cache.device_status() == 0


def test_restore_bf16_is_rounded_fp32(kvq, torch):
    lens = [300, 700, 33]
    _, cache, seqs = build(kvq, torch, lens, 8, 32, 128, 128, 32, 7, "bf16", seed=6)
    k, v = cache.restore(out_dtype="bf16")
    k, v = k.float().cpu().numpy(), v.float().cpu().numpy()
    for b, seq in enumerate(seqs):
        Ko, Vo = oracle_restored(seq)
        np.testing.assert_array_equal(k[b, :, :seq.total], to_bf16_f32(torch, Ko))
        np.testing.assert_array_equal(v[b, :, :seq.total], to_bf16_f32(torch, Vo))


def test_restore_sub_range(kvq, torch):
    lens = [40, 100, 70]
    _, cache, seqs = build(kvq, torch, lens, 2, 4, 16, 8, 8, 7, "fp32", seed=7)
    k, v = cache.restore(seq_begin=1, n_seqs=2, t_stride=128, out_dtype="fp32")
    for j, b in enumerate((1, 2)):
        Ko, Vo = oracle_restored(seqs[b])
        np.testing.assert_array_equal(k[j, :, :lens[b]].cpu().numpy(), Ko)
        np.testing.assert_array_equal(v[j, :, :lens[b]].cpu().numpy(), Vo)


def test_restore_rejects_bad_arguments(kvq, torch):
    _, cache, _ = build(kvq, torch, [40], 2, 4, 16, 8, 8, 7, "fp32", seed=8)
    out = torch.zeros(1, 2, 64, 16, device="cuda")
    with pytest.raises(kvq.KVQError, match="EINVAL"):
        kvq.kvq_restore(cache.handle, 0, 1, out.data_ptr(), out.data_ptr(), 39, kvq.KVQ_FP32, 0)  # stride < 40
    with pytest.raises(kvq.KVQError, match="EINVAL"):
        kvq.kvq_restore(cache.handle, 0, 2, out.data_ptr(), out.data_ptr(), 64, kvq.KVQ_FP32, 0)  # range
    with pytest.raises(kvq.KVQError, match="EINVAL"):
        kvq.kvq_restore(cache.handle, 0, 1, out.data_ptr() + 4, out.data_ptr(), 64, kvq.KVQ_FP32, 0)


@pytest.mark.parametrize("lens,Hq", [([0, 300, 700, 1], 32), ([8192 + 77, 4100], 32), ([513, 40], 8)])
def test_dense_decode_matches_oracle(kvq, torch, lens, Hq):
    spec, cache, seqs = build(kvq, torch, lens, 8, Hq, 128, 128, 32, 7, "bf16", seed=9)
    k, v = cache.restore(t_stride=max(lens) + 5, out_dtype="bf16")
    q = spec.q_block(0, range(len(lens)), 0)
    qd = torch.from_numpy(q).to("cuda").to(torch.bfloat16).contiguous()
    got = cache.dense_decode_attention(k, v, qd).cpu().numpy().astype(np.float64)
    for b, seq in enumerate(seqs):
        if seq.total == 0:
            assert not got[b].any()
            continue
        Ko, Vo = oracle_restored(seq)
        Kb = np.transpose(to_bf16_f32(torch, Ko), (1, 0, 2))
        Vb = np.transpose(to_bf16_f32(torch, Vo), (1, 0, 2))
        ref = O.attn_step(q[b], Kb, Vb)
        excess = np.abs(got[b] - ref) - (ATOL + RTOL * np.abs(ref))
        assert excess.max() <= 0, f"seq {b}: worst |d| {np.abs(got[b] - ref).max():.3e}"
    assert cache.device_status() == 0


def test_dense_decode_agrees_with_fused(kvq, torch):
    """The foil and the fused kernel attend over the same cache: they differ
    only by the bf16 rounding of the restored values."""
    lens = [2000, 1500]
    spec, cache, _ = build(kvq, torch, lens, 8, 32, 128, 128, 32, 7, "bf16", seed=10)
    k, v = cache.restore(out_dtype="bf16")
    qd = torch.from_numpy(spec.q_block(0, range(2), 0)).to("cuda").to(torch.bfloat16).contiguous()
    fused = cache.decode_attention(qd).cpu().numpy()
    dense = cache.dense_decode_attention(k, v, qd).cpu().numpy()
    assert np.abs(fused - dense).max() <= 2e-2 * max(1.0, np.abs(fused).max())


@pytest.mark.parametrize("dtype,group,shape", [
    ("fp32", 0, (2, 4, 64, 32)),
    ("bf16", 0, (2, 4, 64, 32)),
    ("fp32", 16, (2, 4, 64, 32)),
    ("bf16", 32, (1, 8, 256, 128)),
])
def test_compare_matches_oracle(kvq, torch, dtype, group, shape):
    b, h, t, d = shape
    spec = gen.InputSpec(seed=12, n_kv_heads=h, n_q_heads=h, head_dim=d, bf16=dtype == "bf16")
    key, value = spec.kv_block(0, range(b), 0, t)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    got = kvq.compare(torch.from_numpy(key).to("cuda").to(tdt).contiguous(),
                      torch.from_numpy(value).to("cuda").to(tdt).contiguous(), qmax=7, eps=1e-8, group=group)
    esize = 2 if dtype == "bf16" else 4
    if group == 0:
        ref = O.compare_bytes(key, value, esize, qmax=7, eps=1e-8)
        n_kscales = b * h * d
    else:
        # the grouped reading: one Key scale per channel per run of ``group`` tokens
        errs, n_kscales = [], 0
        for g0 in range(0, t, group):
            kq, ks = O.quantize_key_per_channel(key[:, :, g0:g0 + group], 7, 1e-8)
            errs.append((key[:, :, g0:g0 + group] - O.restore(kq, ks, 1e-8)) ** 2)
            n_kscales += ks.size
        ref = O.compare_bytes(key, value, esize, qmax=7, eps=1e-8)
        ref["key_mse"] = float(np.mean(np.concatenate(errs, axis=2), dtype=np.float64))
        ref["container_quantized_bytes"] += 4 * (n_kscales - b * h * d)
        ref["packed_quantized_bytes"] += 4 * (n_kscales - b * h * d)
    assert got["n_key_scales"] == n_kscales and got["n_value_scales"] == b * h * t
    for k in ("raw_bytes", "container_quantized_bytes", "packed_quantized_bytes"):
        assert got[k] == ref[k], k
    np.testing.assert_allclose(got["key_mse"], ref["key_mse"], rtol=1e-5)
    np.testing.assert_allclose(got["value_mse"], ref["value_mse"], rtol=1e-5)


def test_compare_all_zero(kvq, torch):
    z = torch.zeros(1, 2, 16, 16, device="cuda")
    got = kvq.compare(z, z.clone())
    assert got["key_mse"] == 0.0 and got["value_mse"] == 0.0
