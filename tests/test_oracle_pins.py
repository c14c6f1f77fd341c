"""Pins of the CPU oracle to what the pages and the mathematics fix.

Each test names the page and section it follows.  None of these values comes
from the CUDA library.
"""

import json
import math
import os

import numpy as np
import pytest
import scipy.special

from oracle import kvq_oracle as O
from oracle import layout as L

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
MiB = 1 << 20
GiB = 1 << 30


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# Worked examples ("KV Cache 量化与压缩", section 03)
# --------------------------------------------------------------------------

def test_key_only_worked_example():
    ex = _golden("worked_examples.json")["key_only"]
    q = np.array([[ex["q"]]])
    K = np.array(ex["keys"]).reshape(2, 1, 1)
    V = np.array(ex["values"]).reshape(2, 1, 1)
    out = O.attn_step(q, K, V)[0, 0]
    assert round(out, ex["printed_decimals"]) == ex["output"]
    # closed form: 1*p0 + 3*p1 with p1 = 1 / (1 + exp(-(0.26 - 0.14)))
    assert out == pytest.approx(1.0 + 2.0 / (1.0 + math.exp(-0.12)), abs=1e-15)
    p = scipy.special.softmax(np.array(ex["keys"]) * ex["q"])
    np.testing.assert_allclose(np.round(p, 5), ex["softmax"])
    # keys on the 0.2 grid tie, so the weights become equal and the output 2.0
    Kq = O.quantize_on_grid(np.array(ex["keys"], dtype=np.float32), ex["grid_step"])
    np.testing.assert_allclose(Kq, ex["keys_on_grid"], rtol=1e-6)
    assert Kq[0] == Kq[1]
    out_q = O.attn_step(q, Kq.reshape(2, 1, 1), V)[0, 0]
    assert out_q == pytest.approx(ex["output_on_grid"], abs=1e-12)


def test_value_only_worked_example():
    ex = _golden("worked_examples.json")["value_only"]
    vals = np.array(ex["values"], dtype=np.float32)
    Vq = O.quantize_on_grid(vals, ex["grid_step"])
    np.testing.assert_allclose(Vq, ex["values_on_grid"], rtol=1e-7)
    # equal keys give the fixed weights [0.5, 0.5]
    q = np.array([[1.0]])
    K = np.zeros((2, 1, 1))
    before = O.attn_step(q, K, vals.reshape(2, 1, 1))[0, 0]
    after = O.attn_step(q, K, Vq.reshape(2, 1, 1))[0, 0]
    assert before == pytest.approx(ex["output"], abs=1e-6)
    assert after == pytest.approx(ex["output_on_grid"], abs=1e-12)


# --------------------------------------------------------------------------
# Byte accounting ("KV Cache 量化与压缩" 01/05; "KV Cache 与自回归视频生成" 3.3)
# --------------------------------------------------------------------------

def test_capacity_ledger_matches_explainer():
    g = _golden("accounting.json")
    c = g["explainer_cache"]
    args = (c["n_layer"], c["n_kv_head"], c["d_head"], c["positions"])
    assert O.cache_bytes(*args, bits=16)["total"] == g["bf16_MiB"] * MiB
    assert O.cache_bytes(*args, bits=8)["total"] == g["int8_MiB"] * MiB
    assert O.cache_bytes(*args, bits=4)["total"] == g["int4_MiB"] * MiB
    assert O.cache_bytes(*args, bits=4)["scalars"] == g["scalars"]
    meta = dict(scale_bytes=g["scale_bytes"], scalars_per_scale=g["scalars_per_scale"])
    assert O.cache_bytes(*args, bits=8, **meta)["total"] == g["int8_with_scales_MiB"] * MiB
    assert O.cache_bytes(*args, bits=4, **meta)["total"] == g["int4_with_scales_MiB"] * MiB
    win = O.cache_bytes(*args, bits=4, window_positions=g["window_positions"])
    assert win["window_bytes"] == g["window_MiB"] * MiB
    assert win["code_bytes"] == g["old_region_int4_MiB"] * MiB
    assert win["total"] == g["codes_with_window_MiB"] * MiB


def test_bytes_per_token_llama3_and_video():
    g = _golden("accounting.json")
    m = g["llama3_8b"]
    bpt = O.kv_bytes_per_token(m["n_layer"], m["n_kv_head"], m["d_head"], m["dtype_bytes"])
    assert bpt == g["bytes_per_token"]
    assert bpt * 8192 / GiB == g["seq_8192_GiB"]
    assert 32 * bpt * 8192 / GiB == g["batch_32_seq_8192_GiB"]
    assert g["video_frames"] * g["video_tokens_per_frame"] == g["video_tokens"]
    assert round(g["video_tokens"] * bpt / GiB, 2) == g["video_GiB"]


def test_held_ledger_explainer_window_case():
    """A grouped cache of 4096 tokens with R = G = 128 holds 3968 quantized
    positions plus a 128-token window: 124 MiB of 4-bit codes and 16 MiB of
    16-bit window over 32 layers x 8 heads, as in section 05."""
    led = O.held_ledger([4096], n_kv_heads=8, head_dim=128, residual_length=128, group=128,
                        qmax=7, window_element_bytes=2)
    assert 32 * led["code_bytes"] == 124 * MiB
    assert 32 * led["window_bytes"] == 16 * MiB
    # one Key scale per channel per group plus one Value scale per token
    assert 32 * led["n_scales"] == 32 * 8 * (31 * 128 + 3968) == 2_031_616


# --------------------------------------------------------------------------
# Quantizer ("KV Cache Quantization Strategies", Step 2 / Step 4)
# --------------------------------------------------------------------------

def test_quantizer_hand_example_axes_and_half_even():
    x = np.array([[1.0, -2.0], [0.5, 4.0]], dtype=np.float32)[None, None]   # [1,1,T=2,d=2]
    kq, ks = O.quantize_key_per_channel(x)
    assert ks.shape == (1, 1, 1, 2)
    np.testing.assert_array_equal(ks[0, 0, 0], np.float32([7.0, 1.75]))
    np.testing.assert_array_equal(kq[0, 0], [[7, -4], [4, 7]])          # 3.5 -> 4, -3.5 -> -4
    vq, vs = O.quantize_value_per_token(x)
    assert vs.shape == (1, 1, 2, 1)
    np.testing.assert_array_equal(vs[0, 0, :, 0], np.float32([3.5, 1.75]))
    np.testing.assert_array_equal(vq[0, 0], [[4, -7], [1, 7]])           # 0.875 -> 1


def test_round_half_to_even_and_clamp():
    # channel absmax 7 gives scale exactly 1: 2.5 -> 2, -2.5 -> -2, 0.5 -> 0, 1.5 -> 2
    x = np.array([7.0, 2.5, -2.5, 0.5, 1.5, -7.0], dtype=np.float32).reshape(1, 1, 6, 1)
    kq, ks = O.quantize_key_per_channel(x)
    assert ks.item() == 1.0
    np.testing.assert_array_equal(kq.ravel(), [7, 2, -2, 0, 2, -7])
    assert O.quantize_codes(np.float32([10.0, -10.0]), np.float32(1.0), 7).tolist() == [7, -7]
    assert O.quantize_codes(np.float32([300.0]), np.float32(1.0), 127).tolist() == [127]


def test_scale_is_correctly_rounded_division():
    rng = np.random.default_rng(3)
    absmax = (rng.random(20000) * 10 + 1e-3).astype(np.float32)
    s = O.scale_from_absmax(absmax, 7, 1e-8)
    exact = 7.0 / absmax.astype(np.float64)
    # correctly rounded: within half an ulp of the exact quotient
    ulp = np.spacing(s).astype(np.float64)
    assert np.all(np.abs(s.astype(np.float64) - exact) <= 0.5 * ulp)


def test_zero_range_gives_finite_scales_and_zero_codes():
    zeros = np.zeros((1, 1, 3, 4), dtype=np.float32)
    kq, ks = O.quantize_key_per_channel(zeros)
    vq, vs = O.quantize_value_per_token(zeros)
    assert np.isfinite(ks).all() and np.isfinite(vs).all()
    assert ks.ravel()[0] == np.float32(7) / np.float32(1e-8)
    assert not kq.any() and not vq.any()
    assert np.all(O.restore(kq, ks) == 0)


@pytest.mark.parametrize("qmax", [7, 127])
def test_quantizer_invariants_and_error_bound(qmax):
    rng = np.random.default_rng(qmax)
    x = (rng.standard_normal((2, 3, 48, 32)) * rng.uniform(0.05, 5, (1, 3, 1, 32))).astype(np.float32)
    for fn, axis in ((O.quantize_key_per_channel, -2), (O.quantize_value_per_token, -1)):
        q, s = fn(x, qmax)
        assert np.abs(q.astype(int)).max() <= qmax
        # every non-zero channel (K) / token (V) reaches the full code range
        assert np.all(np.abs(q.astype(int)).max(axis=axis) == qmax)
        restored = O.restore(q, s)
        absmax = np.abs(x).max(axis=axis, keepdims=True)
        bound = absmax / (2 * qmax) * (1 + 1e-5) + 1e-7
        assert np.all(np.abs(x - restored) <= bound)


def test_restore_divides_by_scale():
    assert O.restore(np.int8([4]), np.float32([7.0]))[0] == np.float32(4) / np.float32(7)
    assert O.restore(np.int8([-3]), np.float32([0.0]), eps=1e-8)[0] == np.float32(-3) / np.float32(1e-8)


def test_restore_is_correctly_rounded_division():
    # "54. KV Cache Quantization Strategies", Step 4 ``restore``: codes in fp32
    # divided by scale.clamp_min(eps).  One IEEE division rounds once, so every
    # result lies within half an ulp of the exact quotient code / max(scale, eps)
    # taken in fp64 (exact for these operands up to fp64 rounding).
    rng = np.random.default_rng(11)
    n = 50000
    codes = rng.integers(-127, 128, n).astype(np.int8)
    scales = np.exp(rng.uniform(np.log(1e-3), np.log(1e9), n)).astype(np.float32)
    scales[:64] = np.float32(3e-9)          # below eps: the clamp takes over
    scales[64:96] = np.float32(0.0)
    got = O.restore(codes, scales).astype(np.float64)
    eps32 = np.float64(np.float32(1e-8))
    exact = codes.astype(np.float64) / np.maximum(scales.astype(np.float64), eps32)
    ulp = np.spacing(np.abs(got).astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(got - exact) <= 0.5 * ulp)
    # the sample separates a true division from a reciprocal product: the
    # product 1/s * code rounds twice and misses the quotient on many pairs
    recip = (np.float32(1) / np.maximum(scales, np.float32(1e-8))) * codes.astype(np.float32)
    assert np.count_nonzero(recip != got.astype(np.float32)) > n // 50
    # the clamp: a scale below eps divides by eps
    assert got[0] == np.float64(np.float32(codes[0]) / np.float32(1e-8))


# --------------------------------------------------------------------------
# The datawhale page's eight mechanism checks, page rule (group=None)
# --------------------------------------------------------------------------

def _r(*shape, seed=0):
    return np.random.default_rng(seed).standard_normal(shape).astype(np.float32)


def test_page_scale_shapes():
    kq, ks = O.quantize_key_per_channel(_r(1, 2, 5, 8))
    vq, vs = O.quantize_value_per_token(_r(1, 2, 5, 8, seed=1))
    assert kq.shape == (1, 2, 5, 8) and ks.shape == (1, 2, 1, 8)
    assert vq.shape == (1, 2, 5, 8) and vs.shape == (1, 2, 5, 1)


def test_page_token_conservation():
    st = O.append_and_partition(None, _r(1, 2, 3, 8), _r(1, 2, 3, 8, seed=1), 4)
    st = O.append_and_partition(st, _r(1, 2, 2, 8, seed=2), _r(1, 2, 2, 8, seed=3), 4)
    assert st["total_tokens"] == 5
    assert st["quantized_tokens"] + st["key_residual"].shape[-2] == 5
    assert st["quantized_tokens"] + st["value_residual"].shape[-2] == 5


def test_page_partition_residual_two():
    st = O.append_and_partition(None, _r(1, 2, 3, 8), _r(1, 2, 3, 8, seed=1), 2)
    st = O.append_and_partition(st, _r(1, 2, 2, 8, seed=2), _r(1, 2, 2, 8, seed=3), 2)
    assert st["quantized_tokens"] == 3
    assert sum(s.shape[-2] for s in st["key_q_segments"]) == 3
    assert st["key_residual"].shape[-2] == 2 and st["value_residual"].shape[-2] == 2


def test_page_prefix_not_rewritten():
    st = O.append_and_partition(None, _r(1, 1, 3, 4), _r(1, 1, 3, 4, seed=1), 2)
    first = st["key_q_segments"][0].copy()
    first_scale = st["key_scale_segments"][0].copy()
    st = O.append_and_partition(st, _r(1, 1, 2, 4, seed=2) * 100, _r(1, 1, 2, 4, seed=3), 2)
    assert len(st["key_q_segments"]) == 2
    np.testing.assert_array_equal(st["key_q_segments"][0], first)
    np.testing.assert_array_equal(st["key_scale_segments"][0], first_scale)
    assert st["flushed_tokens"] == 2


def test_page_no_overflow():
    st = O.append_and_partition(None, _r(1, 1, 1, 4), _r(1, 1, 1, 4, seed=1), 4)
    st = O.append_and_partition(st, _r(1, 1, 1, 4, seed=2), _r(1, 1, 1, 4, seed=3), 4)
    assert st["quantized_tokens"] == 0 and st["flushed_tokens"] == 0
    assert st["key_residual"].shape[-2] == 2


def test_page_restore_and_budget():
    res = O.compare_bytes(_r(1, 2, 7, 8), _r(1, 2, 7, 8, seed=1), raw_element_bytes=4)
    assert math.isfinite(res["key_mse"]) and math.isfinite(res["value_mse"])
    assert res["packed_quantized_bytes"] < res["raw_bytes"]
    assert res["packed_quantized_bytes"] < res["container_quantized_bytes"]


@pytest.mark.parametrize("shape,raw_el,expect", [
    # [1, 2, 7, 8] fp32: 112 Key + 112 Value scalars; Key scales [1, 2, 1, 8] = 16
    # fp32 (64 B), Value scales [1, 2, 7, 1] = 14 fp32 (56 B).
    # raw 224 * 4 = 896; int8 container 224 + 120 = 344; packed (224 + 1) // 2 + 120 = 232
    ((1, 2, 7, 8), 4, (896, 344, 232)),
    # [2, 1, 3, 5] bf16: 30 + 30 scalars; Key scales 2 * 5 = 10 fp32 (40 B),
    # Value scales 2 * 3 = 6 fp32 (24 B).  raw 60 * 2 = 120; container 60 + 64 = 124;
    # packed 61 // 2 + 64 = 94
    ((2, 1, 3, 5), 2, (120, 124, 94)),
])
def test_compare_byte_ledger_hand_values(shape, raw_el, expect):
    # "54. KV Cache Quantization Strategies", Step 4 ``compare``: raw bytes are
    # numel * element_size of Key and Value; the int8 container adds one byte a
    # code plus the fp32 scales; packed 4-bit bytes are (nK + nV + 1) // 2 plus
    # the same fp32 scale bytes.  Values worked out by hand above.
    res = O.compare_bytes(_r(*shape), _r(*shape, seed=1), raw_element_bytes=raw_el)
    assert (res["raw_bytes"], res["container_quantized_bytes"], res["packed_quantized_bytes"]) == expect


def test_page_rule_rejects_bad_arguments():
    with pytest.raises(ValueError):
        O.append_and_partition(None, _r(1, 1, 1, 4), _r(1, 1, 1, 4), 0)
    with pytest.raises(ValueError):
        O.append_and_partition(None, _r(1, 1, 4), _r(1, 1, 4), 2)
    with pytest.raises(ValueError):
        O.append_and_partition(None, _r(1, 1, 1, 4), _r(1, 1, 2, 4), 2)


# --------------------------------------------------------------------------
# Grouped rule
# --------------------------------------------------------------------------

def test_grouped_counts_tiny_schedule():
    """Prefill 40 then 24 single-token appends, R = G = 8: 4 groups at once,
    then one group every 8 appends -> 7 groups, 56 quantized, window 8."""
    seq = O.GroupedSequence(heads=2, head_dim=16, residual_length=8, group=8)
    seq.append(_r(2, 40, 16), _r(2, 40, 16, seed=1))
    assert (seq.quantized, seq.window) == (32, 8)
    for i in range(24):
        seq.append(_r(2, 1, 16, seed=10 + i), _r(2, 1, 16, seed=100 + i))
    assert (seq.total, seq.quantized, seq.window) == (64, 56, 8)
    assert len(seq.state["key_q_segments"]) == 7


def test_group_of_one_is_the_page_rule():
    rng = np.random.default_rng(5)
    page = grouped = None
    for step in range(30):
        n = int(rng.integers(1, 6))
        k, v = _r(1, 1, n, 4, seed=step), _r(1, 1, n, 4, seed=1000 + step)
        page = O.append_and_partition(page, k, v, 5)
        grouped = O.append_and_partition(grouped, k, v, 5, group=1)
        assert page["flushed_tokens"] == grouped["flushed_tokens"]
        assert page["key_residual"].shape[-2] == grouped["key_residual"].shape[-2] == min(page["total_tokens"], 5)
        # Value scales are per token, so their codes agree whatever the segmentation
        np.testing.assert_array_equal(np.concatenate(page["value_q_segments"], -2) if page["value_q_segments"] else 0,
                                      np.concatenate(grouped["value_q_segments"], -2) if grouped["value_q_segments"] else 0)


def test_grouped_counts_closed_form_and_window_bounds():
    rng = np.random.default_rng(9)
    for R, G in ((8, 8), (128, 32), (5, 3), (1, 4)):
        seq = O.GroupedSequence(heads=1, head_dim=4, residual_length=R, group=G)
        for step in range(40):
            n = int(rng.integers(1, 3 * (R + G)))
            seq.append(_r(1, n, 4, seed=step), _r(1, n, 4, seed=500 + step))
            q, w = O.grouped_counts(seq.total, R, G)
            assert (seq.quantized, seq.window) == (q, w)
            assert seq.quantized % G == 0
            assert seq.window < R + G
            if seq.quantized:
                assert seq.window >= R


def test_grouped_chunking_invariance_and_no_rewrite():
    """Any chunking of the same token stream gives the same codes and scales,
    and codes already written never change."""
    H, D, R, G, T = 2, 16, 8, 8, 77
    k, v = _r(H, T, D, seed=1), _r(H, T, D, seed=2)
    ref = O.GroupedSequence(H, D, R, G)
    ref.append(k, v)
    for chunks in ([1] * T, [7] * 11, [40, 1, 1, 35], [3, 50, 24]):
        seq = O.GroupedSequence(H, D, R, G)
        pos = 0
        prev_codes = None
        for n in chunks:
            seq.append(k[:, pos:pos + n], v[:, pos:pos + n])
            pos += n
            codes = seq.key_codes()
            if prev_codes is not None:
                np.testing.assert_array_equal(codes[:, :prev_codes.shape[1]], prev_codes)
            prev_codes = codes
        np.testing.assert_array_equal(seq.key_codes(), ref.key_codes())
        np.testing.assert_array_equal(seq.value_codes(), ref.value_codes())
        np.testing.assert_array_equal(seq.key_scales(), ref.key_scales())
        np.testing.assert_array_equal(seq.value_scales(), ref.value_scales())
        np.testing.assert_array_equal(seq.window_kv()[0], ref.window_kv()[0])


def test_grouped_key_scale_is_per_group():
    """Each group's Key scale comes from that group's tokens only."""
    H, D, R, G = 1, 4, 4, 4
    k = np.zeros((H, 12, D), np.float32)
    k[:, :4] = 1.0
    k[:, 4:8] = 10.0
    seq = O.GroupedSequence(H, D, R, G)
    seq.append(k, k)
    ks = seq.key_scales()
    assert ks.shape == (1, 2, 4)
    np.testing.assert_array_equal(ks[0, 0], np.float32(7) / np.float32(1.0))
    np.testing.assert_array_equal(ks[0, 1], np.float32(7) / np.float32(10.0))


# --------------------------------------------------------------------------
# Attention ("KV Cache 与自回归视频生成" 3.1, section 04 attn_step)
# --------------------------------------------------------------------------

def test_attention_closed_forms():
    # equal keys -> plain mean of V
    V = _r(9, 1, 4).astype(np.float64)
    out = O.attn_step(_r(1, 4), np.ones((9, 1, 4)), V)
    np.testing.assert_allclose(out[0], V[:, 0].mean(axis=0), rtol=1e-13)
    # the 1/sqrt(d) factor: q = k1 = ones(4), k2 = 0 -> logits 2 and 0
    q = np.ones((1, 4))
    K = np.stack([np.ones(4), np.zeros(4)])[:, None, :]
    Vv = np.stack([np.full(4, 3.0), np.full(4, -1.0)])[:, None, :]
    p1 = math.exp(2) / (1 + math.exp(2))
    np.testing.assert_allclose(O.attn_step(q, K, Vv)[0], 3 * p1 - (1 - p1), rtol=1e-14)
    # a dominant key picks its value
    K2 = np.zeros((5, 1, 4))
    K2[3] = 100.0
    np.testing.assert_allclose(O.attn_step(np.ones((1, 4)), K2, V[:5])[0], V[3, 0], rtol=1e-12)


def test_attention_large_logits_stay_finite():
    """attn_step subtracts the row max before exponentiating, so logits in the
    thousands are exact rather than overflowing (softmax is shift invariant)."""
    q = np.full((1, 4), 100.0)
    K = np.zeros((3, 1, 4))
    K[1] = 50.0                                    # logit 1e4 against 0
    V = np.arange(12, dtype=np.float64).reshape(3, 1, 4)
    out = O.attn_step(q, K, V)
    assert np.isfinite(out).all()
    np.testing.assert_array_equal(out[0], V[1, 0])


def test_attention_gqa_head_mapping():
    """q head h reads KV head h // g (g = Hq / Hkv), not h % Hkv."""
    Hq, Hkv, S, d = 4, 2, 6, 8
    K = _r(S, Hkv, d).astype(np.float64)
    V = np.zeros((S, Hkv, d))
    V[:, 0] = 1.0
    V[:, 1] = -2.0
    out = O.attn_step(_r(Hq, d, seed=3), K, V)
    np.testing.assert_allclose(out[:2], 1.0, rtol=1e-14)
    np.testing.assert_allclose(out[2:], -2.0, rtol=1e-14)


def test_attention_matches_library_softmax():
    q, K, V = _r(3, 16).astype(np.float64), _r(20, 1, 16, seed=1), _r(20, 1, 16, seed=2)
    out = O.attn_step(q, K, V)
    for h in range(3):
        p = scipy.special.softmax(K[:, 0] @ q[h] / 4.0)
        np.testing.assert_allclose(out[h], p @ V[:, 0], rtol=1e-12, atol=1e-14)


def test_attention_empty_cache_is_zero():
    assert not O.attn_step(_r(2, 4), np.zeros((0, 1, 4)), np.zeros((0, 1, 4))).any()


def test_unflushed_cache_attends_raw_values():
    """While nothing has left the window the quantized cache is the plain cache."""
    seq = O.GroupedSequence(heads=2, head_dim=8, residual_length=16, group=8)
    k, v = _r(2, 20, 8), _r(2, 20, 8, seed=1)
    seq.append(k, v)
    assert seq.quantized == 0
    q = _r(4, 8, seed=2)
    np.testing.assert_array_equal(seq.attend(q), O.attn_step(q, k.transpose(1, 0, 2), v.transpose(1, 0, 2)))


def test_current_token_is_attended():
    """o_t sums j = 1..t: the token appended in this step takes part."""
    seq = O.GroupedSequence(heads=1, head_dim=4, residual_length=4, group=4)
    seq.append(np.zeros((1, 3, 4), np.float32), np.zeros((1, 3, 4), np.float32))
    big = np.full((1, 1, 4), 50.0, np.float32)
    seq.append(big, big)
    out = seq.attend(np.ones((1, 4), np.float32))
    np.testing.assert_allclose(out[0], 50.0, rtol=1e-12)


# --------------------------------------------------------------------------
# Storage layout encoder (include/kvq.h, group page)
# --------------------------------------------------------------------------

def test_layout_key_nibbles():
    # offset binary: nibble = code + 8, byte = code + 128
    codes = np.int8([[1, -1, -7, 7]])
    assert L.pack_key_codes(codes, 4) == bytes([0x79, 0xF1])
    assert L.pack_key_codes(codes, 8) == bytes([0x81, 0x7F, 0x79, 0x87])


def test_layout_two_bit_key_crumbs():
    # code + 2 in two bits, channel 4i + k at bits 2k of byte i
    codes = np.int8([[1, -1, 0, 1, -1, 0, 0, 1]])
    assert L.pack_key_codes(codes, 2) == bytes([0xE7, 0xE9])


def test_layout_two_bit_value_pieces():
    codes = np.int8([-1, 0, 1, -1, 0, 1, -1, 0]).reshape(8, 1)   # tokens 0..7 of one channel
    # low byte: tokens 0, 2, 4, 6 (crumbs 1, 3, 2, 1); high byte: tokens 1, 3, 5, 7 (2, 1, 3, 2)
    assert L.pack_value_codes(codes, 2) == bytes([0x6D, 0xB6])
    z = np.zeros((32, 16), np.int8)
    assert L.page_bytes(32, 16, 2) == 448
    assert len(L.pack_group_page(z, z, np.ones(16), np.ones(32), 2)) == 448


def test_code_bits():
    assert [O.code_bits(q) for q in (1, 2, 7, 8, 127)] == [2, 4, 4, 8, 8]


def test_held_ledger_two_bit_codes_halve_the_four_bit_ledger():
    """The section 05 case with 2-bit codes (qmax = 1): the code bytes halve,
    scales and window do not change."""
    four = O.held_ledger([4096], n_kv_heads=8, head_dim=128, residual_length=128, group=128,
                         qmax=7, window_element_bytes=2)
    two = O.held_ledger([4096], n_kv_heads=8, head_dim=128, residual_length=128, group=128,
                        qmax=1, window_element_bytes=2)
    assert 32 * two["code_bytes"] == 62 * MiB
    assert two["n_scales"] == four["n_scales"] and two["window_bytes"] == four["window_bytes"]


def test_layout_value_word_order():
    codes = np.arange(8, dtype=np.int8).reshape(8, 1)          # tokens 0..7 of one channel
    # nibbles hold tokens 0,2,4,6,1,3,5,7, each code + 8 -> word 0xFDB9ECA8
    assert L.pack_value_codes(codes, 4) == (0xFDB9ECA8).to_bytes(4, "little")
    codes2 = np.arange(64, dtype=np.int8).reshape(32, 2) - 32   # 32 tokens x 2 channels
    out = L.pack_value_codes(codes2, 8)
    assert out[:32] == bytes((int(c) + 128) for c in codes2[:, 0])
    assert out[32:] == bytes((int(c) + 128) for c in codes2[:, 1])
    assert len(L.pack_group_page(codes2, codes2, np.ones(2), np.ones(32), 8)) == L.page_bytes(32, 2, 8)
