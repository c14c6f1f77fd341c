"""Plain CPU oracle for the KIVI-style asymmetric KV-cache quantizer and the
single-query GQA decode attention that reads it.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA library (``quantized_kv_cache_02_gb300``): no kernels,
headers, helpers, tables or constant generators.

What it computes, and where each step is stated:

* Quantizer -- "54. KV Cache Quantization Strategies" (datawhale llm-algo-leetcode),
  Step 2 (quantization axes: Key per channel over the token axis, scale shape
  [..., 1, head_dim]; Value per token over head_dim, scale shape [..., tokens, 1])
  and Step 4, reference solution (``_quantize``, ``restore``,
  ``quantize_key_per_channel``, ``quantize_value_per_token``).
  Precision is the page's: fp32 (``x.float()``), ``torch.round`` (half to even),
  symmetric clamp to [-qmax, qmax], int8 container.
  Reading taken: ``qmax / max(absmax, eps)`` is the correctly rounded fp32
  quotient (PyTorch happens to evaluate ``int / tensor`` as reciprocal-then-
  multiply, which is a library artefact, not the stated formula).
* Residual window and flush -- same page, Step 3 (newest tokens stay in a
  high-precision window; on overflow only the oldest tokens move to a new
  quantized segment; the quantized prefix is never rewritten) and Step 4
  ``append_and_partition`` (flush = max(L - residual_length, 0)).
  Two modes:
    - ``group=None``: the page's rule verbatim, one segment per append.
    - ``group=G``: the grouped rule used by the GPU library: after an append the
      held tail L is flushed in whole groups of G tokens, F = floor((L - R) / G)
      groups when L >= R + G, each group one segment with its own Key scale.
      With G = 1 this is exactly the page's rule.
* Decode attention -- "KV Cache 与自回归视频生成" (jefxiong), section 3.1
  (o_t = sum_j softmax_j(q_t k_j^T / sqrt(d)) v_j, the current token included)
  and section 04 ``attn_step`` (GQA: query head h reads KV head h // g;
  max-subtract, exp, normalise).  Evaluated in float64 on the restored
  (dequantized, fp32) prefix followed by the fp32 window.
* Byte accounting -- "KV Cache 量化与压缩" (xuujii M005) sections 01 and 05;
  the datawhale page's ``compare`` (packed 4-bit bytes); the jefxiong page's
  section 3.3 (B_tok = 2 L n_kv d p).

Every function is written for clarity, not speed.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

F32 = np.float32


# --------------------------------------------------------------------------
# Quantizer  (KV Cache Quantization Strategies, Step 2 and Step 4)
# --------------------------------------------------------------------------

def quantize_codes(x: np.ndarray, scale: np.ndarray, qmax: int) -> np.ndarray:
    """``_quantize``: clamp(round(x.float() * scale), -qmax, qmax) as int8.

    The product is one fp32 multiply (rounded to nearest); ``np.rint`` rounds
    half to even like ``torch.round``.
    """
    prod = np.multiply(np.asarray(x, dtype=F32), np.asarray(scale, dtype=F32), dtype=F32)
    rounded = np.rint(prod)
    clamped = np.clip(rounded, -qmax, qmax)
    return clamped.astype(np.int8)


def scale_from_absmax(absmax: np.ndarray, qmax: int, eps: float) -> np.ndarray:
    """scale = qmax / max(absmax, eps), one correctly rounded fp32 division."""
    floor = np.maximum(np.asarray(absmax, dtype=F32), F32(eps))
    return np.divide(F32(qmax), floor, dtype=F32)


def quantize_key_per_channel(key: np.ndarray, qmax: int = 7, eps: float = 1e-8):
    """Key: absmax over the token axis (-2), keepdim -> scale [..., 1, head_dim]."""
    key = np.asarray(key, dtype=F32)
    absmax = np.max(np.abs(key), axis=-2, keepdims=True)
    scale = scale_from_absmax(absmax, qmax, eps)
    return quantize_codes(key, scale, qmax), scale


def quantize_value_per_token(value: np.ndarray, qmax: int = 7, eps: float = 1e-8):
    """Value: absmax over head_dim (-1), keepdim -> scale [..., tokens, 1]."""
    value = np.asarray(value, dtype=F32)
    absmax = np.max(np.abs(value), axis=-1, keepdims=True)
    scale = scale_from_absmax(absmax, qmax, eps)
    return quantize_codes(value, scale, qmax), scale


def restore(codes: np.ndarray, scale: np.ndarray, eps: float = 1e-8) -> np.ndarray:
    """``restore``: codes.to(fp32) / scale.clamp_min(eps), in fp32."""
    return np.divide(np.asarray(codes, dtype=F32),
                     np.maximum(np.asarray(scale, dtype=F32), F32(eps)), dtype=F32)


def quantize_on_grid(x: np.ndarray, step: float, qmax: int = 127) -> np.ndarray:
    """The explainer's worked examples put values on an integer grid of spacing
    ``step`` ("KV Cache 量化与压缩", section 03).  In the datawhale formulation
    the scale is a multiplier, so step s <-> scale 1/s; returns the restored
    values code / scale."""
    scale = np.full(np.shape(x), F32(1.0) / F32(step), dtype=F32)
    return restore(quantize_codes(x, scale, qmax), scale)


# --------------------------------------------------------------------------
# Residual window and flush  (KV Cache Quantization Strategies, Step 3/Step 4)
# --------------------------------------------------------------------------

def page_flush_tokens(held: int, new: int, residual_length: int) -> int:
    """flush_tokens = max(L - residual_length, 0) with L = held + new."""
    return max(held + new - residual_length, 0)


def grouped_flush_groups(held: int, new: int, residual_length: int, group: int) -> int:
    """Grouped rule: whole groups of ``group`` tokens leave the window once the
    held tail L = held + new reaches residual_length + group."""
    tail = held + new
    if tail < residual_length + group:
        return 0
    return (tail - residual_length) // group


def new_state(batch: int, heads: int, head_dim: int) -> dict:
    """The empty state dict of ``append_and_partition`` (segment lists plus an
    empty high-precision residual for Key and Value)."""
    empty = np.zeros((batch, heads, 0, head_dim), dtype=F32)
    return {
        "key_q_segments": [], "key_scale_segments": [],
        "value_q_segments": [], "value_scale_segments": [],
        "key_residual": empty.copy(), "value_residual": empty.copy(),
        "flushed_tokens": 0, "quantized_tokens": 0, "total_tokens": 0,
    }


def append_and_partition(state: dict | None, new_key: np.ndarray, new_value: np.ndarray,
                         residual_length: int, qmax: int = 7, eps: float = 1e-8,
                         group: int | None = None) -> dict:
    """Append new K/V ([batch, heads, tokens, head_dim]) and quantize only what
    overflows the residual window.

    ``group=None`` is the page's rule: the whole overflow becomes ONE new
    segment with one Key scale over its tokens.  ``group=G`` flushes whole
    groups of G tokens, oldest first, one segment (one Key scale) per group.
    Earlier segments are carried over untouched.
    """
    if residual_length <= 0:
        raise ValueError("residual_length must be positive")
    if group is not None and group <= 0:
        raise ValueError("group must be positive")
    new_key = np.asarray(new_key, dtype=F32)
    new_value = np.asarray(new_value, dtype=F32)
    if new_key.ndim != 4 or new_value.ndim != 4:
        raise ValueError("new_key and new_value must be four-dimensional")
    if new_key.shape != new_value.shape:
        raise ValueError("new_key and new_value must share the same shape")
    if state is None:
        b, h, _, d = new_key.shape
        state = new_state(b, h, d)

    key_all = np.concatenate([state["key_residual"], new_key], axis=-2)
    value_all = np.concatenate([state["value_residual"], new_value], axis=-2)
    held = state["key_residual"].shape[-2]
    n_new = new_key.shape[-2]

    if group is None:
        flush_tokens = page_flush_tokens(held, n_new, residual_length)
        spans = [(0, flush_tokens)] if flush_tokens else []
    else:
        n_groups = grouped_flush_groups(held, n_new, residual_length, group)
        flush_tokens = n_groups * group
        spans = [(i * group, (i + 1) * group) for i in range(n_groups)]

    key_q_segments = list(state["key_q_segments"])
    key_scale_segments = list(state["key_scale_segments"])
    value_q_segments = list(state["value_q_segments"])
    value_scale_segments = list(state["value_scale_segments"])
    for lo, hi in spans:
        key_q, key_scale = quantize_key_per_channel(key_all[..., lo:hi, :], qmax, eps)
        value_q, value_scale = quantize_value_per_token(value_all[..., lo:hi, :], qmax, eps)
        key_q_segments.append(key_q)
        key_scale_segments.append(key_scale)
        value_q_segments.append(value_q)
        value_scale_segments.append(value_scale)

    key_residual = key_all[..., flush_tokens:, :]
    value_residual = value_all[..., flush_tokens:, :]
    quantized_tokens = sum(seg.shape[-2] for seg in key_q_segments)
    return {
        "key_q_segments": key_q_segments,
        "key_scale_segments": key_scale_segments,
        "value_q_segments": value_q_segments,
        "value_scale_segments": value_scale_segments,
        "key_residual": key_residual,
        "value_residual": value_residual,
        "flushed_tokens": flush_tokens,
        "quantized_tokens": quantized_tokens,
        "total_tokens": quantized_tokens + key_residual.shape[-2],
    }


def restored_kv(state: dict, eps: float = 1e-8):
    """The cache as attention sees it: restored segments in token order, then
    the residual window.  Returns K, V as fp32 [batch, heads, tokens, head_dim]."""
    keys = [restore(q, s, eps) for q, s in zip(state["key_q_segments"], state["key_scale_segments"])]
    values = [restore(q, s, eps) for q, s in zip(state["value_q_segments"], state["value_scale_segments"])]
    keys.append(state["key_residual"])
    values.append(state["value_residual"])
    return np.concatenate(keys, axis=-2), np.concatenate(values, axis=-2)


# --------------------------------------------------------------------------
# Decode attention  (KV Cache 与自回归视频生成, section 3.1 and section 04)
# --------------------------------------------------------------------------

def attn_step(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """One decode step: q [Hq, Dh], K/V [S, Hkv, Dh] -> [Hq, Dh], float64.

    Query head h reads KV head h // g with g = Hq / Hkv; logits are q.k/sqrt(Dh);
    subtract the row max, exponentiate, normalise, weight V.
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    Hq, Dh = q.shape
    S, Hkv, _ = K.shape
    g = Hq // Hkv
    out = np.zeros((Hq, Dh), dtype=np.float64)
    if S == 0:
        return out
    for h in range(Hq):
        kv = h // g
        logits = (K[:, kv, :] @ q[h]) / math.sqrt(Dh)
        logits = logits - logits.max()
        p = np.exp(logits)
        p = p / p.sum()
        out[h] = p @ V[:, kv, :]
    return out


def decode_attention(state: dict, q: np.ndarray, eps: float = 1e-8) -> np.ndarray:
    """Attention of q [batch, Hq, d] over every held token of each sequence
    (restored prefix + window).  Returns float64 [batch, Hq, d]."""
    K, V = restored_kv(state, eps)               # [B, Hkv, S, d]
    q = np.asarray(q, dtype=F32)
    out = np.zeros(q.shape, dtype=np.float64)
    for b in range(q.shape[0]):
        out[b] = attn_step(q[b], np.transpose(K[b], (1, 0, 2)), np.transpose(V[b], (1, 0, 2)))
    return out


# --------------------------------------------------------------------------
# One sequence of a ragged batch, grouped rule (the GPU library's semantics)
# --------------------------------------------------------------------------

@dataclass
class GroupedSequence:
    """Per-sequence grouped-mode cache for heads x head_dim, fed one append at
    a time; the batch dimension of ``append_and_partition`` is 1."""
    heads: int
    head_dim: int
    residual_length: int
    group: int
    qmax: int = 7
    eps: float = 1e-8
    state: dict = field(default=None)

    def __post_init__(self):
        if self.state is None:
            self.state = new_state(1, self.heads, self.head_dim)

    def append(self, new_key: np.ndarray, new_value: np.ndarray) -> None:
        """new_key/new_value: [heads, n, head_dim]."""
        self.state = append_and_partition(self.state, new_key[None], new_value[None],
                                          self.residual_length, self.qmax, self.eps, self.group)

    @property
    def total(self) -> int:
        return self.state["total_tokens"]

    @property
    def quantized(self) -> int:
        return self.state["quantized_tokens"]

    @property
    def window(self) -> int:
        return self.state["key_residual"].shape[-2]

    def key_codes(self) -> np.ndarray:
        """[heads, quantized, head_dim] int8 in token order."""
        segs = [s[0] for s in self.state["key_q_segments"]]
        return np.concatenate(segs, axis=-2) if segs else np.zeros((self.heads, 0, self.head_dim), np.int8)

    def value_codes(self) -> np.ndarray:
        segs = [s[0] for s in self.state["value_q_segments"]]
        return np.concatenate(segs, axis=-2) if segs else np.zeros((self.heads, 0, self.head_dim), np.int8)

    def key_scales(self) -> np.ndarray:
        """[heads, n_groups, head_dim] fp32 (one row per flushed group)."""
        segs = [s[0, :, 0, :] for s in self.state["key_scale_segments"]]
        return np.stack(segs, axis=1) if segs else np.zeros((self.heads, 0, self.head_dim), F32)

    def value_scales(self) -> np.ndarray:
        """[heads, quantized] fp32 (one per token)."""
        segs = [s[0, :, :, 0] for s in self.state["value_scale_segments"]]
        return np.concatenate(segs, axis=-1) if segs else np.zeros((self.heads, 0), F32)

    def window_kv(self):
        return self.state["key_residual"][0], self.state["value_residual"][0]

    def attend(self, q: np.ndarray) -> np.ndarray:
        """q [Hq, head_dim] -> float64 [Hq, head_dim]."""
        return decode_attention(self.state, q[None], self.eps)[0]


# --------------------------------------------------------------------------
# Byte accounting
# --------------------------------------------------------------------------

def kv_bytes_per_token(n_layer: int, n_kv_head: int, d_head: int, dtype_bytes: int) -> int:
    """B_tok = 2 (K,V) x L x n_kv x d x p  ("KV Cache 与自回归视频生成", 3.3)."""
    return 2 * n_layer * n_kv_head * d_head * dtype_bytes


def cache_bytes(n_layer: int, n_kv_head: int, d_head: int, positions: int, bits: int,
                scale_bytes: int = 0, scalars_per_scale: int | None = None,
                window_positions: int = 0, window_bits: int = 16) -> dict:
    """Capacity ledger of "KV Cache 量化与压缩" sections 01 and 05.

    K and V scalars of the low-bit region are ``bits`` wide; the newest
    ``window_positions`` positions stay ``window_bits`` wide; optionally one
    ``scale_bytes`` scale per ``scalars_per_scale`` low-bit scalars.  Returns
    code bytes, window bytes, scale bytes and their total.
    """
    per_position = 2 * n_layer * n_kv_head * d_head          # K and V scalars
    low_scalars = per_position * (positions - window_positions)
    code_bytes = low_scalars * bits // 8
    window_bytes = per_position * window_positions * window_bits // 8
    scale = 0
    if scalars_per_scale:
        scale = (low_scalars // scalars_per_scale) * scale_bytes
    return {"code_bytes": code_bytes, "window_bytes": window_bytes,
            "scale_bytes": scale, "total": code_bytes + window_bytes + scale,
            "scalars": per_position * positions}


def compare_bytes(key: np.ndarray, value: np.ndarray, raw_element_bytes: int,
                  qmax: int = 7, eps: float = 1e-8) -> dict:
    """The datawhale page's ``compare`` ledger: raw bytes, int8-container bytes
    and packed 4-bit bytes ((nK + nV + 1) // 2 plus fp32 scale bytes)."""
    key_q, key_scale = quantize_key_per_channel(key, qmax, eps)
    value_q, value_scale = quantize_value_per_token(value, qmax, eps)
    scale_bytes = key_scale.size * 4 + value_scale.size * 4
    key_restored = restore(key_q, key_scale, eps)
    value_restored = restore(value_q, value_scale, eps)
    return {
        "key_scale_shape": key_scale.shape,
        "value_scale_shape": value_scale.shape,
        "key_mse": float(np.mean((np.asarray(key, F32) - key_restored) ** 2)),
        "value_mse": float(np.mean((np.asarray(value, F32) - value_restored) ** 2)),
        "raw_bytes": (key.size + value.size) * raw_element_bytes,
        "container_quantized_bytes": key_q.size + value_q.size + scale_bytes,
        "packed_quantized_bytes": (key_q.size + value_q.size + 1) // 2 + scale_bytes,
    }


def grouped_counts(total: int, residual_length: int, group: int):
    """Held partition of a sequence of ``total`` tokens under the grouped rule
    (independent of how the tokens were chunked into appends):
    returns (quantized, window)."""
    quantized = 0
    if total >= residual_length + group:
        quantized = ((total - residual_length) // group) * group
    return quantized, total - quantized


def code_bits(qmax: int) -> int:
    """Bits of one stored code: the fewest of 2, 4, 8 that hold the 2*qmax + 1
    levels -qmax..qmax."""
    return 2 if qmax <= 1 else 4 if qmax <= 7 else 8


def held_ledger(totals, n_kv_heads: int, head_dim: int, residual_length: int, group: int,
                qmax: int, window_element_bytes: int) -> dict:
    """Bytes a grouped-mode cache holds for sequences of the given lengths:
    codes (2-bit packed when qmax <= 1 -- KIVI's 2-bit codes, "KV Cache 量化与压缩"
    section 04 --, 4-bit packed when qmax <= 7, else int8), fp32 Key scales
    (one per channel per group), fp32 Value scales (one per token) and the
    window."""
    bits = code_bits(qmax)
    code = n_scales = window_elems = 0
    for total in totals:
        quantized, window = grouped_counts(int(total), residual_length, group)
        code += 2 * n_kv_heads * quantized * head_dim * bits // 8
        n_scales += n_kv_heads * ((quantized // group) * head_dim + quantized)
        window_elems += 2 * n_kv_heads * window * head_dim
    return {"code_bytes": code, "n_scales": n_scales, "scale_bytes": 4 * n_scales,
            "window_elems": window_elems, "window_bytes": window_elems * window_element_bytes,
            "total": code + 4 * n_scales + window_elems * window_element_bytes}
