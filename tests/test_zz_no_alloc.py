"""kvq_decode_attention_noalloc: the decode attention for callers that cannot
allocate device memory when they decode (a plugin whose host framework owns
every device allocation, a deployment that reserves all memory at start-up).
It keeps the split scratch in a fixed array inside the library.  Checked
through the C ABI against kvq_decode_attention on two calls in a row, with
the attention tolerance the other parity tests use, on contiguous, paged and
segmented caches; and, where the array forces a smaller split count than the
usual plan, against the oracle as well.  Kept in its own file, collected
last, so a stop-at-first-failure run has already run every other test before
this one."""

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


def _close(got, ref):
    excess = np.abs(got - ref) - (ATOL + RTOL * np.abs(ref))
    assert excess.max() <= 0, f"max excess {excess.max():.3e}"


def _noalloc_twice(kvq, torch, cache, q, B, Hq, D):
    stream = torch.cuda.current_stream().cuda_stream
    outs = []
    for _ in range(2):
        out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
        kvq.kvq_decode_attention_noalloc(cache.handle, q.data_ptr(), out.data_ptr(), stream)
        got = out.cpu().numpy()
        assert np.isfinite(got).all()
        outs.append(got)
    return outs


@pytest.mark.parametrize("form", ["contiguous", "paged", "segmented"])
@pytest.mark.parametrize("dtype,D,G,qmax", [("bf16", 128, 32, 7), ("fp32", 16, 8, 7), ("bf16", 128, 64, 127)])
def test_noalloc_matches_decode_attention(torch, dtype, D, G, qmax, form):
    import quantized_kv_cache_02_gb300 as kvq
    H, Hq, B = (8, 32, 4) if D == 128 else (2, 4, 3)
    spec = gen.InputSpec(seed=21, n_kv_heads=H, n_q_heads=Hq, head_dim=D, bf16=(dtype == "bf16"))
    lens = [1500, 40, 777, 2100][:B]
    caps = [n + 4 for n in lens]
    pool = sum(c // G for c in caps) if form == "paged" else 0
    cache = kvq.KVQCache(B, H, Hq, D, 128 if D == 128 else 8, G, qmax, caps, dtype=dtype, pool_blocks=pool,
                         segmented=form == "segmented")
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    for b, n in enumerate(lens):
        k, v = spec.kv_block(0, [b], 0, n)
        cache.append(torch.from_numpy(k).cuda().to(tdt), torch.from_numpy(v).cuda().to(tdt), seq_begin=b)
    q = torch.from_numpy(spec.q_block(0, range(B), 0)).cuda().to(tdt)
    ref = cache.decode_attention(q).cpu().numpy()
    for got in _noalloc_twice(kvq, torch, cache, q, B, Hq, D):
        _close(got, ref)
    assert cache.device_status() == 0


def test_noalloc_lowers_the_split_count(torch):
    """A cache whose usual split plan does not fit the array: batch 16 x 8 KV
    heads x 8 query heads a KV head at head_dim 256 needs 16 * 8 * 8 * 260 =
    266,240 floats a split column, so the 2^21-float array holds 7 columns.
    Each sequence holds 56 group pages (1932 tokens, R 128, G 32): the usual
    plan (about 6 items an SM over 128 units, at least 8 pages an item) takes
    chunks of 8 pages, 7 quantized columns plus the window's = 8 > 7, so the
    entry point lowers it to chunks of 10 pages (6 + 1 columns).  Compared
    with kvq_decode_attention and with the oracle."""
    import quantized_kv_cache_02_gb300 as kvq
    B, H, Hq, D, R, G, T = 16, 8, 64, 256, 128, 32, 1932
    per_column = B * H * (Hq // H) * (D + 4)
    assert (2 << 20) // per_column == 7
    assert (T - R) // G == 56
    spec = gen.InputSpec(seed=23, n_kv_heads=H, n_q_heads=Hq, head_dim=D)
    cache = kvq.KVQCache(B, H, Hq, D, R, G, 7, T + 4)
    k, v = spec.kv_block(0, range(B), 0, T)
    cache.append(torch.from_numpy(k).cuda().bfloat16(), torch.from_numpy(v).cuda().bfloat16(), 0)
    q = spec.q_block(0, range(B), 0)
    qd = torch.from_numpy(q).cuda().bfloat16()
    ref = cache.decode_attention(qd).cpu().numpy()
    outs = _noalloc_twice(kvq, torch, cache, qd, B, Hq, D)
    for got in outs:
        _close(got, ref)
    for b in (0, 7, 15):
        seq = O.GroupedSequence(H, D, R, G, 7)
        seq.append(k[b], v[b])
        _close(outs[1][b], seq.attend(q[b]))
    assert cache.device_status() == 0


def test_noalloc_rejects_oversized_batch(torch):
    import quantized_kv_cache_02_gb300 as kvq
    # one split column alone needs 1024 sequences x 8 KV heads x 8 query heads
    # x 132 floats (head_dim + 4) = 8.65M floats, beyond the 2^21-float array
    cache = kvq.KVQCache(1024, 8, 64, 128, 128, 32, 7, 64)
    q = torch.zeros(1024, 64, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(1024, 64, 128, dtype=torch.float32, device="cuda")
    launches = kvq.kvq_kernel_launches()
    with pytest.raises(kvq.KVQError) as e:
        kvq.kvq_decode_attention_noalloc(cache.handle, q.data_ptr(), out.data_ptr(),
                                         torch.cuda.current_stream().cuda_stream)
    assert e.value.status == kvq.binding.KVQ_ECAPACITY
    assert "8 MiB" in str(e.value)
    assert kvq.kvq_kernel_launches() == launches
