"""Byte-level encoder of one flushed group ("group page") in the storage layout
that ``include/kvq.h`` defines, written from that definition alone.

TEST INFRASTRUCTURE ONLY (same rules as ``kvq_oracle``): the parity tests use
it to compare the GPU cache's raw bytes with the oracle's codes and scales.

Layout of one group page (G tokens, D channels, ``bits`` = 4 or 8):

Codes are stored offset binary: code + 2 in two bits (bits = 2, qmax <= 1),
code + 8 in a nibble, code + 128 in a byte.

1. Key codes, G rows in token order, D*bits/8 bytes each.  2-bit: byte i
   holds channel 4i + k in bits 2k..2k+1.  4-bit: byte i holds channel 2i in
   bits 0-3 and channel 2i+1 in bits 4-7.  8-bit: byte c is channel c.
2. Value codes, in sub-tiles of 32 tokens (the last sub-tile holds G mod 32
   tokens when G is not a multiple of 32).  A sub-tile of n tokens is D rows
   (channel order) of n*bits/8 bytes.  4-bit rows are little-endian 32-bit
   words; word w covers the sub-tile's tokens 8w..8w+7 and its nibble j
   (bits 4j..4j+3) holds token 8w+2j for j < 4 and token 8w+2(j-4)+1 for
   j >= 4.  2-bit rows are little-endian 16-bit pieces; piece p covers tokens
   8p..8p+7, bits 2f..2f+1 hold token 8p+2f and bits 8+2f..9+2f token
   8p+2f+1 (f = 0..3).  8-bit rows hold token i in byte i.
3. Key scales: D fp32, channel order.
4. Value scales: G fp32, token order.
"""

from __future__ import annotations

import numpy as np


def _nibble(code: int) -> int:
    return (int(code) + 8) & 0xF


def _byte(code: int) -> int:
    return (int(code) + 128) & 0xFF


def _crumb(code: int) -> int:
    return (int(code) + 2) & 0x3


def pack_key_codes(codes: np.ndarray, bits: int) -> bytes:
    """codes: int8 [G, D] -> key-code bytes of one page."""
    G, D = codes.shape
    out = bytearray()
    for t in range(G):
        if bits == 2:
            for i in range(D // 4):
                out.append(sum(_crumb(codes[t, 4 * i + k]) << (2 * k) for k in range(4)))
        elif bits == 4:
            for i in range(D // 2):
                out.append(_nibble(codes[t, 2 * i]) | (_nibble(codes[t, 2 * i + 1]) << 4))
        else:
            for c in range(D):
                out.append(_byte(codes[t, c]))
    return bytes(out)


def _value_word_tokens() -> list[int]:
    """Token offset (within an 8-token word) held by nibble j = 0..7."""
    return [2 * j if j < 4 else 2 * (j - 4) + 1 for j in range(8)]


def pack_value_codes(codes: np.ndarray, bits: int) -> bytes:
    """codes: int8 [G, D] -> value-code bytes of one page."""
    G, D = codes.shape
    order = _value_word_tokens()
    out = bytearray()
    for start in range(0, G, 32):
        n = min(32, G - start)
        for c in range(D):
            if bits == 2:
                for p in range(n // 8):
                    piece = 0
                    for f in range(4):
                        piece |= _crumb(codes[start + 8 * p + 2 * f, c]) << (2 * f)
                        piece |= _crumb(codes[start + 8 * p + 2 * f + 1, c]) << (8 + 2 * f)
                    out += piece.to_bytes(2, "little")
            elif bits == 4:
                for w in range(n // 8):
                    word = 0
                    for j in range(8):
                        word |= _nibble(codes[start + 8 * w + order[j], c]) << (4 * j)
                    out += word.to_bytes(4, "little")
            else:
                for i in range(n):
                    out.append(_byte(codes[start + i, c]))
    return bytes(out)


def pack_group_page(key_codes: np.ndarray, value_codes: np.ndarray,
                    key_scale: np.ndarray, value_scale: np.ndarray, bits: int) -> bytes:
    """One full page: key codes, value codes, key scales (D fp32), value scales (G fp32)."""
    return (pack_key_codes(key_codes, bits) + pack_value_codes(value_codes, bits)
            + np.asarray(key_scale, dtype="<f4").tobytes()
            + np.asarray(value_scale, dtype="<f4").tobytes())


def page_bytes(group: int, head_dim: int, bits: int) -> int:
    return 2 * group * head_dim * bits // 8 + 4 * head_dim + 4 * group
