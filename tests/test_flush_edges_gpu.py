"""Grouped flush (append_kernel) on the method's degenerate inputs, bit for
bit against the oracle, at 4-, 8- and 2-bit codes and bf16 / fp32 caches.

"54. KV Cache Quantization Strategies": the zero-range test (an all-zero
range still gets a finite scale, qmax / eps, and codes 0) and ``_quantize``
(``torch.round``: ties to even).  Cases, all inside groups that the append
flushes:
  - an all-zero Key channel and an all-zero Value token;
  - a Key channel and a Value token whose absmax lies below eps, so the scale
    is qmax / eps and the codes are rint(x * qmax / eps);
  - exact ties: a Key channel with absmax qmax (scale 1) and a Value token
    with absmax qmax, whose other entries are k + 1/2, so x * s lands on the
    half-way points and rounds to the even neighbour.
Codes, scales, counters, the window and the raw page bytes must equal the
oracle's.
"""

import numpy as np
import pytest

from kvq_inputs import gen
from oracle import kvq_oracle as O
from oracle import layout as L

pytestmark = pytest.mark.gpu

H, HQ, D, R, G = 2, 8, 128, 32, 32


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


def edge_tensors(qmax, n, seed):
    """K, V [H, n, D] from the seeded generator with the edge cases planted.

    Group 0 (tokens 0..31): Key channel 3 and Value token 5 all zero.
    Group 1 (tokens 32..63): Key channel 9 and Value token 40 below eps.
    Group 2 (tokens 64..95): Key channel 20 and Value token 70 hold the
    half-way points k + 1/2 with absmax qmax (scale exactly 1)."""
    spec = gen.InputSpec(seed=seed, n_kv_heads=H, n_q_heads=HQ, head_dim=D)
    k, v = spec.kv_block(0, [0], 0, n)
    k, v = k[0].copy(), v[0].copy()
    k[:, 0:32, 3] = 0.0
    v[:, 5, :] = 0.0
    tiny = np.float32(2.0 ** -30)          # ~9.3e-10 < eps (1e-8); x * qmax / eps is not a tie
    k[:, 32:64, 9] = tiny * np.where(np.arange(32) % 2 == 0, 1.0, -0.5)
    v[:, 40, :] = tiny * np.where(np.arange(D) % 3 == 0, -1.0, 0.25)
    # ties: values +-(k + 1/2) for k < qmax, plus one entry at qmax
    halves = np.arange(qmax, dtype=np.float32) + np.float32(0.5)          # 0.5 .. qmax - 0.5
    signs = np.where(np.arange(len(halves)) % 2 == 0, 1.0, -1.0).astype(np.float32)
    ties = np.resize(halves * signs, 32 - 1)
    k[:, 64:95, 20] = ties
    k[:, 95, 20] = qmax
    row = np.resize(halves * signs, D - 1)
    v[:, 70, :D - 1] = row
    v[:, 70, D - 1] = -qmax
    return k, v


def check(cache, seq, qmax):
    st = cache.seq_state(0)
    assert (st["total"], st["quantized"], st["window"]) == (seq.total, seq.quantized, seq.window)
    bits = O.code_bits(qmax)
    for h in range(H):
        got = cache.export_unit(0, h)
        np.testing.assert_array_equal(got["k_codes"], seq.key_codes()[h])
        np.testing.assert_array_equal(got["v_codes"], seq.value_codes()[h])
        np.testing.assert_array_equal(got["k_scales"].view(np.uint32), seq.key_scales()[h].view(np.uint32))
        np.testing.assert_array_equal(got["v_scales"].view(np.uint32), seq.value_scales()[h].view(np.uint32))
        wk, wv = seq.window_kv()
        np.testing.assert_array_equal(got["window_k"], wk[h])
        np.testing.assert_array_equal(got["window_v"], wv[h])
        raw = cache.export_pages(0, h)
        expect = b"".join(
            L.pack_group_page(seq.key_codes()[h][j * G:(j + 1) * G], seq.value_codes()[h][j * G:(j + 1) * G],
                              seq.key_scales()[h][j], seq.value_scales()[h][j * G:(j + 1) * G], bits)
            for j in range(seq.quantized // G))
        assert raw == expect


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("qmax", [7, 127, 1])
@pytest.mark.parametrize("chunks", [[140], [100, 1, 1, 1, 37]])
def test_flush_edge_cases(kvq, torch, qmax, dtype, chunks):
    n = sum(chunks)
    k, v = edge_tensors(qmax, n, seed=71)
    # the values the cache holds: rounded to bf16 first for a bf16 cache (the
    # planted values are all bf16-exact)
    if dtype == "bf16":
        k = torch.from_numpy(k).bfloat16().float().numpy()
        v = torch.from_numpy(v).bfloat16().float().numpy()
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    cache = kvq.KVQCache(1, H, HQ, D, R, G, qmax, n + 8, dtype=dtype)
    seq = O.GroupedSequence(H, D, R, G, qmax)
    pos = 0
    for c in chunks:
        kk, vv = k[:, pos:pos + c], v[:, pos:pos + c]
        cache.append(torch.from_numpy(np.ascontiguousarray(kk[None])).cuda().to(tdt),
                     torch.from_numpy(np.ascontiguousarray(vv[None])).cuda().to(tdt), 0)
        seq.append(kk, vv)
        pos += c
    assert seq.quantized >= 3 * G
    check(cache, seq, qmax)
    # the oracle's own view of the planted groups (independent of the GPU)
    kc, vc = seq.key_codes(), seq.value_codes()
    ks, vs = seq.key_scales(), seq.value_scales()
    eps = np.float32(1e-8)
    assert ks[0, 0, 3] == np.float32(qmax) / eps and not kc[0, 0:32, 3].any()
    assert vs[0, 5] == np.float32(qmax) / eps and not vc[0, 5].any()
    assert ks[0, 1, 9] == np.float32(qmax) / eps and vs[0, 40] == np.float32(qmax) / eps
    assert ks[0, 2, 20] == 1.0 and vs[0, 70] == 1.0
    tie = k[0, 64:95, 20]
    np.testing.assert_array_equal(kc[0, 64:95, 20], np.rint(tie).astype(np.int8))
    assert cache.device_status() == 0
