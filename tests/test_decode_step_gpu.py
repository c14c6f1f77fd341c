"""kvq_decode_step against kvq_append + kvq_decode_attention: identical
outputs, counters and raw pages, on steps with and without a flush, for the
fused tensor-core path (contiguous, paged, large groups, 2-bit) and the
paths that fall back to the two calls (fp32, the CUDA-core kernel)."""

import numpy as np
import pytest

from kvq_inputs import gen

pytestmark = pytest.mark.gpu


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


@pytest.mark.parametrize("D,G,qmax,dtype,pool,kernel", [
    (128, 32, 7, "bf16", 0, 0),     # fused, contiguous
    (128, 32, 7, "bf16", 400, 0),   # fused, paged
    (64, 64, 1, "bf16", 0, 0),      # fused, staged large group, 2-bit
    (128, 32, 127, "bf16", 0, 2),   # fused, 8-bit, kernel forced
    (128, 32, 7, "bf16", 0, 3),     # fused, the tcgen05 kernel's window items
    (128, 64, 7, "bf16", 300, 3),   # fused, tcgen05 kernel, paged, staged units
    (64, 32, 7, "fp32", 0, 0),      # falls back (fp32 runs the CUDA-core kernel)
    (128, 32, 7, "bf16", 0, 1),     # falls back (CUDA-core kernel asked for)
])
def test_decode_step_equals_append_then_decode(kvq, torch, D, G, qmax, dtype, pool, kernel):
    B, H, Hq, R = 3, 4, 16, 64
    bf16 = dtype == "bf16"
    spec = gen.InputSpec(seed=51, n_kv_heads=H, n_q_heads=Hq, head_dim=D, bf16=bf16)
    tdt = torch.bfloat16 if bf16 else torch.float32
    lens = [R + G - 3, 200, 37]            # sequence 0 flushes on the third step
    cap = max(lens) + 2 * G + 8
    a = kvq.KVQCache(B, H, Hq, D, R, G, qmax, cap, dtype=dtype, pool_blocks=pool)
    b = kvq.KVQCache(B, H, Hq, D, R, G, qmax, cap, dtype=dtype, pool_blocks=pool)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to("cuda").to(tdt).contiguous()
    for s, n in enumerate(lens):
        k, v = spec.kv_block(0, [s], 0, n)
        a.append(dev(k), dev(v), s)
        b.append(dev(k), dev(v), s)
    for step in range(2 * G + 3):
        k = np.concatenate([spec.kv_block(0, [s], lens[s] + step, 1)[0] for s in range(B)])
        v = np.concatenate([spec.kv_block(0, [s], lens[s] + step, 1)[1] for s in range(B)])
        q = dev(spec.q_block(0, range(B), step))
        got = a.decode_step(dev(k), dev(v), q, kernel=kernel).cpu().numpy()
        b.append(dev(k), dev(v), 0)
        ref = b.decode_attention(q, kernel=kernel).cpu().numpy()
        np.testing.assert_array_equal(got, ref)
    for s in range(B):
        assert a.seq_state(s) == b.seq_state(s)
        assert a.export_pages(s, 1) == b.export_pages(s, 1)
        ua, ub = a.export_unit(s, 2), b.export_unit(s, 2)
        np.testing.assert_array_equal(ua["window_k"], ub["window_k"])
        np.testing.assert_array_equal(ua["window_v"], ub["window_v"])
    assert a.device_status() == 0


@pytest.mark.parametrize("kernel", [0, 3])
def test_decode_step_against_the_oracle(kvq, torch, kernel):
    """kvq_decode_step compared with the oracle directly: the oracle appends
    the step's token ("KV Cache Quantization Strategies", append_and_partition,
    grouped) and attends over the held tokens, the new one included ("KV
    Cache 与自回归视频生成" 3.1); attention within |d| <= 1e-3 + 1e-2 |ref|,
    codes, scales and window bit for bit, over steps with and without a
    flush."""
    from oracle import kvq_oracle as O
    B, H, Hq, D, R, G, qmax = 3, 4, 16, 128, 64, 32, 7
    spec = gen.InputSpec(seed=52, n_kv_heads=H, n_q_heads=Hq, head_dim=D)
    lens = [R + G - 2, 300, 70]
    cache = kvq.KVQCache(B, H, Hq, D, R, G, qmax, max(lens) + G + 8)
    seqs = [O.GroupedSequence(H, D, R, G, qmax) for _ in range(B)]
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to("cuda").bfloat16().contiguous()
    for s, n in enumerate(lens):
        k, v = spec.kv_block(0, [s], 0, n)
        cache.append(dev(k), dev(v), s)
        seqs[s].append(k[0], v[0])
    for step in range(G + 3):
        k = np.concatenate([spec.kv_block(0, [s], lens[s] + step, 1)[0] for s in range(B)])
        v = np.concatenate([spec.kv_block(0, [s], lens[s] + step, 1)[1] for s in range(B)])
        q = spec.q_block(0, range(B), step)
        got = cache.decode_step(dev(k), dev(v), dev(q), kernel=kernel).cpu().numpy()
        for s in range(B):
            seqs[s].append(k[s], v[s])
        if step % 4 == 0 or step in (1, 2, G + 2):
            ref = np.stack([seqs[s].attend(q[s]) for s in range(B)])
            excess = np.abs(got - ref) - (1e-3 + 1e-2 * np.abs(ref))
            assert excess.max() <= 0, f"step {step}: max excess {excess.max():.3e}"
    for s in range(B):
        st = cache.seq_state(s)
        assert (st["total"], st["quantized"], st["window"]) == (seqs[s].total, seqs[s].quantized, seqs[s].window)
        for h in (0, 3):
            u = cache.export_unit(s, h)
            np.testing.assert_array_equal(u["k_codes"], seqs[s].key_codes()[h])
            np.testing.assert_array_equal(u["v_codes"], seqs[s].value_codes()[h])
            np.testing.assert_array_equal(u["k_scales"].view(np.uint32), seqs[s].key_scales()[h].view(np.uint32))
            np.testing.assert_array_equal(u["v_scales"].view(np.uint32), seqs[s].value_scales()[h].view(np.uint32))
            np.testing.assert_array_equal(u["window_k"], seqs[s].window_kv()[0][h])
    assert cache.device_status() == 0
