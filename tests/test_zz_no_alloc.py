"""kvq_decode_attention_noalloc: the decode attention for callers that cannot
allocate device memory when they decode (a plugin whose host framework owns
every device allocation, a deployment that reserves all memory at start-up).
It keeps the split scratch in a fixed array inside the library.  Checked
through the C ABI against kvq_decode_attention on two calls in a row, with
the attention tolerance the other parity tests use.  Kept in its own file,
collected last, so a stop-at-first-failure run has already run every other
test before this one."""

import numpy as np
import pytest

from kvq_inputs import gen

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


@pytest.mark.parametrize("dtype,D,G,qmax", [("bf16", 128, 32, 7), ("fp32", 16, 8, 7), ("bf16", 128, 64, 127)])
def test_noalloc_matches_decode_attention(torch, dtype, D, G, qmax):
    import quantized_kv_cache_02_gb300 as kvq
    H, Hq, B = (8, 32, 4) if D == 128 else (2, 4, 3)
    spec = gen.InputSpec(seed=21, n_kv_heads=H, n_q_heads=Hq, head_dim=D, bf16=(dtype == "bf16"))
    lens = [1500, 40, 777, 2100][:B]
    cache = kvq.KVQCache(B, H, Hq, D, 128 if D == 128 else 8, G, qmax, [n + 4 for n in lens], dtype=dtype)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    for b, n in enumerate(lens):
        k, v = spec.kv_block(0, [b], 0, n)
        cache.append(torch.from_numpy(k).cuda().to(tdt), torch.from_numpy(v).cuda().to(tdt), seq_begin=b)
    stream = torch.cuda.current_stream().cuda_stream
    q = torch.from_numpy(spec.q_block(0, range(B), 0)).cuda().to(tdt)
    ref = cache.decode_attention(q).cpu().numpy()
    for _ in range(2):
        out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
        kvq.kvq_decode_attention_noalloc(cache.handle, q.data_ptr(), out.data_ptr(), stream)
        got = out.cpu().numpy()
        assert np.isfinite(got).all()
        _close(got, ref)
    assert cache.device_status() == 0


def test_noalloc_rejects_oversized_batch(torch):
    import quantized_kv_cache_02_gb300 as kvq
    # one split column alone needs 1024 sequences x 8 KV heads x 8 query heads
    # x 130 floats = 8.5M floats, beyond the 2^21-float array
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
