"""Seeded synthetic inputs for the quantized KV cache: Key, Value and query
tensors with the value distributions of the workloads the library is measured
on.  This module holds none of the cache's arithmetic; both the CPU oracle (via
the numpy functions here) and the GPU runs (via the same numpy functions, or
the bit-identical CUDA fill in ``csrc/kvq_gen.cu``) consume its output.

Generator (counter based, so any (layer, sequence, head, token, channel)
element can be regenerated on its own):

* ``mix64`` is the SplitMix64 output function (Steele, Lea and Flood,
  "Fast splittable pseudorandom number generators", 2014; Stafford's variant-13
  constants); ``hash_at(key, i) = mix64(key + (i + 1) * 0x9E3779B97F4A7C15)``.
* A standard normal draw is ``NORMAL[h >> 48]``: 65536 equiprobable levels, the
  inverse normal CDF at (i + 0.5) / 65536 (|z| up to 4.3) rounded to fp32.
* Log-uniform draws use level tables computed once in float64 and rounded to
  fp32, so the device never evaluates exp/log and both sides agree bit for bit.

Distributions (per layer, sequence and KV head):

* K[t, c] = z * sigma_c, sigma_c log-uniform in [0.05, 5] per (layer, KV head,
  channel); in every block of 16 channels one seeded channel has sigma x 10
  (outlier channel).  Optional spikes: with probability 1/1000 per element the
  value is multiplied by 50.
* V[t, :] = z * tau_t, tau_t log-uniform in [0.5, 2] per (layer, sequence,
  KV head, token), 4096 levels.
* q = z.
* Every product is one fp32 multiply; bf16 inputs are then rounded to nearest
  even bf16 once.
"""

from __future__ import annotations

import math
from dataclasses import dataclass
from statistics import NormalDist

import numpy as np

U64 = np.uint64
GAMMA = 0x9E3779B97F4A7C15
MIX_A = 0xBF58476D1CE4E5B9
MIX_B = 0x94D049BB133111EB
MASK64 = (1 << 64) - 1
NORMAL_LEVELS = 65536
TAU_LEVELS = 4096
SPIKE_THRESHOLD = 4294967          # floor(0.001 * 2**32)
SPIKE_FACTOR = 50.0
OUTLIER_FACTOR = 10.0

STREAMS = {"K": 1, "V": 2, "q": 3, "tau": 4, "sigma": 5, "outlier": 6, "len": 7}


def mix64_int(z: int) -> int:
    z &= MASK64
    z = ((z ^ (z >> 30)) * MIX_A) & MASK64
    z = ((z ^ (z >> 27)) * MIX_B) & MASK64
    return z ^ (z >> 31)


def mix64(z: np.ndarray) -> np.ndarray:
    z = z.astype(U64, copy=True)
    with np.errstate(over="ignore"):
        z ^= z >> U64(30)
        z *= U64(MIX_A)
        z ^= z >> U64(27)
        z *= U64(MIX_B)
        z ^= z >> U64(31)
    return z


def stream_key(*parts: int) -> int:
    """Fold integer parts into one 64-bit key."""
    k = 0x243F6A8885A308D3
    for p in parts:
        k = mix64_int(k ^ mix64_int(int(p) + GAMMA))
    return k


def hash_at(key: int, idx: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = U64(key) + (idx.astype(U64) + U64(1)) * U64(GAMMA)
    return mix64(z)


def _normal_table() -> np.ndarray:
    nd = NormalDist()
    return np.array([nd.inv_cdf((i + 0.5) / NORMAL_LEVELS) for i in range(NORMAL_LEVELS)],
                    dtype=np.float32)


def _tau_table() -> np.ndarray:
    lo, hi = math.log(0.5), math.log(2.0)
    return np.array([math.exp(lo + (i + 0.5) / TAU_LEVELS * (hi - lo)) for i in range(TAU_LEVELS)],
                    dtype=np.float32)


NORMAL_TABLE = _normal_table()
TAU_TABLE = _tau_table()


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """fp32 -> nearest bf16 (ties to even), returned as fp32 values."""
    bits = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((bits >> np.uint32(16)) & np.uint32(1))
    out = ((bits + bias) & np.uint32(0xFFFF0000)).astype(np.uint32)
    return out.view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Upper 16 bits of fp32 values that are already bf16-representable."""
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


@dataclass(frozen=True)
class InputSpec:
    """Which synthetic workload to draw: ``seed`` separates workloads."""
    seed: int
    n_kv_heads: int
    n_q_heads: int
    head_dim: int
    bf16: bool = True
    spikes: bool = False

    # ---- per-stream keys --------------------------------------------------
    def key(self, stream: str, layer: int, seq: int, head: int) -> int:
        return stream_key(self.seed, STREAMS[stream], layer, seq, head)

    def sigma(self, layer: int) -> np.ndarray:
        """[n_kv_heads, head_dim] fp32 Key channel scales, outliers included."""
        H, D = self.n_kv_heads, self.head_dim
        out = np.empty((H, D), dtype=np.float32)
        lo, hi = math.log(0.05), math.log(5.0)
        for h in range(H):
            hs = hash_at(stream_key(self.seed, STREAMS["sigma"], layer, h), np.arange(D))
            u = (hs >> U64(11)).astype(np.float64) * 2.0 ** -53
            sig = np.exp(lo + u * (hi - lo))
            for blk in range(0, D, 16):
                width = min(16, D - blk)
                pick = int(hash_at(stream_key(self.seed, STREAMS["outlier"], layer, h), np.array([blk]))[0] % U64(width))
                sig[blk + pick] *= OUTLIER_FACTOR
            out[h] = sig.astype(np.float32)
        return out

    def _finish(self, x: np.ndarray) -> np.ndarray:
        return round_to_bf16(x) if self.bf16 else x

    # ---- host blocks --------------------------------------------------------
    def kv_block(self, layer: int, seqs, t0: int, n: int, heads=None):
        """K, V for tokens [t0, t0 + n) of the given sequences:
        fp32 arrays [len(seqs), n_kv_heads, n, head_dim], or
        [len(seqs), len(heads), n, head_dim] for a subset ``heads`` of the KV
        heads (each head's values do not depend on the others)."""
        seqs = list(seqs)
        H, D = self.n_kv_heads, self.head_dim
        heads = list(range(H)) if heads is None else list(heads)
        sig = self.sigma(layer)
        t = np.arange(t0, t0 + n, dtype=np.uint64)
        idx = (t[:, None] * U64(D) + np.arange(D, dtype=np.uint64)[None, :])
        K = np.empty((len(seqs), len(heads), n, D), dtype=np.float32)
        V = np.empty_like(K)
        for i, b in enumerate(seqs):
            for hi, h in enumerate(heads):
                hk = hash_at(self.key("K", layer, b, h), idx)
                k = np.multiply(NORMAL_TABLE[(hk >> U64(48)).astype(np.int64)], sig[h][None, :], dtype=np.float32)
                if self.spikes:
                    spike = (hk & U64(0xFFFFFFFF)) < U64(SPIKE_THRESHOLD)
                    k = np.where(spike, np.multiply(k, np.float32(SPIKE_FACTOR), dtype=np.float32), k)
                K[i, hi] = self._finish(k)
                hv = hash_at(self.key("V", layer, b, h), idx)
                tau = TAU_TABLE[(hash_at(self.key("tau", layer, b, h), t) >> U64(52)).astype(np.int64)]
                v = np.multiply(NORMAL_TABLE[(hv >> U64(48)).astype(np.int64)], tau[:, None], dtype=np.float32)
                V[i, hi] = self._finish(v)
        return K, V

    def q_block(self, layer: int, seqs, step: int) -> np.ndarray:
        """Queries of decode step ``step``: fp32 [len(seqs), n_q_heads, head_dim]."""
        seqs = list(seqs)
        D = self.head_dim
        idx = np.arange(D, dtype=np.uint64) + U64(step * D)
        out = np.empty((len(seqs), self.n_q_heads, D), dtype=np.float32)
        for i, b in enumerate(seqs):
            for h in range(self.n_q_heads):
                hq = hash_at(self.key("q", layer, b, h), idx)
                out[i, h] = self._finish(NORMAL_TABLE[(hq >> U64(48)).astype(np.int64)])
        return out

    def lengths(self, batch: int, lo: int, hi: int) -> list[int]:
        """Seeded per-sequence lengths, uniform on the integers [lo, hi]."""
        span = hi - lo + 1
        return [lo + int(hash_at(stream_key(self.seed, STREAMS["len"]), np.array([b]))[0] % U64(span))
                for b in range(batch)]
