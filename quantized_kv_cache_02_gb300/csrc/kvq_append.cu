// Append / flush / quantize / pack.
//
// One launch appends n tokens to each sequence of [seq_begin, seq_begin + n_seqs):
//   * flush blocks (blockIdx.x < flush_blocks): one CTA per (group, sequence, KV
//     head) quantizes the oldest G tokens of the held tail -- Key per channel
//     (absmax over the group's tokens), Value per token (absmax over head_dim),
//     scale = qmax / max(absmax, eps), code = clamp(rint(x * scale)) -- and writes
//     the group page once ("54. KV Cache Quantization Strategies", Step 2 and
//     the Step 4 reference solution; the grouped flush rule is in kvq.h);
//   * window block (the last blockIdx.x): copies the new tokens that stay in the
//     residual window into the per-unit ring (preallocated, written in place
//     rather than concatenated, as "KV Cache 与自回归视频生成" section 05 argues).
// Tokens being flushed come from the ring (old window) or straight from the
// input (new tokens), so a long prefill never passes through the ring.
// Bit exactness: absmax is exact, the division is __fdiv_rn, the product is a
// separately rounded __fmul_rn, rintf rounds half to even; no fast-math.

#include <cuda_bf16.h>

#include <type_traits>

#include "kvq_internal.h"

namespace kvq {
namespace {


__device__ __forceinline__ int quantize_one(float x, float scale, float qmax) {
  float r = rintf(__fmul_rn(x, scale));
  r = fminf(fmaxf(r, -qmax), qmax);
  return (int)r;
}

// The stored offset-binary code clamp(rint(x * scale), -qmax, qmax) +
// 2^(BITS-1), in the low BITS bits of the returned word.  The clamp never
// acts here: |x| <= absmax and scale = qmax / max(absmax, eps) (each rounded
// once) make |x * scale| <= qmax (1 + 2^-23) < qmax + 1/2, so rint already
// lies in [-qmax, qmax].  The product, rounded on its own, then gets one add
// of 1.5 * 2^23 + 2^(BITS-1): the sum's unit in the last place is 1, so the
// add rounds to the nearest integer with ties to even, which is rint(x *
// scale) + 2^(BITS-1) because the bias is even; the sum's mantissa field
// holds 2^22 plus that integer, and 2^22 being a multiple of 256, its low
// bits are the offset code (in [1, 2^BITS - 1]).  One FMA-pipe add stands for
// the conversion, the clamp and the bias.
template <int BITS>
__device__ __forceinline__ uint32_t quantize_bits(float x, float scale) {
  constexpr float kMagic = 12582912.f + (float)(1 << (BITS - 1));
  return __float_as_uint(__fadd_rn(__fmul_rn(x, scale), kMagic));
}

// The offset code in the low BITS bits of ``bits`` at field k of a word.
template <int BITS>
__device__ __forceinline__ uint32_t code_field(uint32_t bits, int k) {
  return (bits & ((1u << BITS) - 1u)) << (BITS * k);
}

// The low bytes of four words as the bytes 0..3 of one word.
__device__ __forceinline__ uint32_t low_bytes(uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3) {
  return __byte_perm(__byte_perm(b0, b1, 0x0040), __byte_perm(b2, b3, 0x0040), 0x5410);
}
// Eight 4-bit codes (low nibbles of the arguments) into one word: lo0..lo3
// go to the low nibbles of bytes 0..3, hi0..hi3 to their high nibbles.
__device__ __forceinline__ uint32_t pack_nibbles(uint32_t lo0, uint32_t lo1, uint32_t lo2, uint32_t lo3, uint32_t hi0,
                                                 uint32_t hi1, uint32_t hi2, uint32_t hi3) {
  const uint32_t lo = low_bytes(lo0, lo1, lo2, lo3), hi = low_bytes(hi0, hi1, hi2, hi3);
  return (lo & 0x0F0F0F0Fu) | ((hi << 4) & 0xF0F0F0F0u);
}

// Two consecutive elements of shared memory, kept packed until used.
struct PairF {
  float2 v;
  __device__ __forceinline__ void load(const float* p) { v = *reinterpret_cast<const float2*>(p); }
  __device__ __forceinline__ float get(int e) const { return e ? v.y : v.x; }
};
struct PairB {
  uint32_t v;  // two bf16, the first in the low half
  __device__ __forceinline__ void load(const __nv_bfloat16* p) { v = *reinterpret_cast<const uint32_t*>(p); }
  __device__ __forceinline__ float get(int e) const { return __uint_as_float(e ? (v & 0xFFFF0000u) : (v << 16)); }
};
template <typename T>
using PairOf = typename std::conditional<sizeof(T) == 4, PairF, PairB>::type;

template <typename T>
__device__ __forceinline__ float to_f32(T x) {
  if constexpr (sizeof(T) == 4) return x;
  else return __bfloat162float(x);
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
               : "memory");
}

// 16 bytes of elements -> fp32 values
__device__ __forceinline__ void unpack16(const uint4& raw, float (&x)[4]) {
  const float* f = reinterpret_cast<const float*>(&raw);
  x[0] = f[0];
  x[1] = f[1];
  x[2] = f[2];
  x[3] = f[3];
}
__device__ __forceinline__ void unpack16(const uint4& raw, float (&x)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __bfloat1622float2(h[e]);
    x[2 * e] = f.x;
    x[2 * e + 1] = f.y;
  }
}

// Absolute values of two bf16 packed in a word, as 16-bit unsigned integers:
// for values >= 0 the bit patterns order like the values, so a per-halfword
// unsigned max is the max of |x|, and the fp32 absmax of a half h is the float
// with bits h << 16.  Two channels (or tokens) a pair of instructions, with no
// conversion to fp32 until the final maximum.
__device__ __forceinline__ uint32_t abs_bf16x2(uint32_t w) { return w & 0x7FFF7FFFu; }
__device__ __forceinline__ uint32_t umax_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ float bf16_lo_f32(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi_f32(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// N consecutive elements of shared memory as fp32 (vector loads)
template <typename T, int N>
__device__ __forceinline__ void load_elems(const T* src, float (&x)[N]) {
  constexpr int kBytes = N * (int)sizeof(T);
  if constexpr (kBytes % 16 == 0) {
    constexpr int kPer = 16 / (int)sizeof(T);
#pragma unroll
    for (int i = 0; i < kBytes / 16; ++i) {
      float y[kPer];
      unpack16(reinterpret_cast<const uint4*>(src)[i], y);
#pragma unroll
      for (int e = 0; e < kPer; ++e) x[i * kPer + e] = y[e];
    }
  } else {
#pragma unroll
    for (int e = 0; e < N; ++e) x[e] = to_f32(src[e]);
  }
}

// DC: head_dim as a compile-time constant (64, 128), or 0 for any other.
// KB: rows a flush thread loads per batch (2 when the group is only a pass or
// two of rows deep, 4 for deeper groups), so that short groups do not issue
// predicated-off loads; four CTAs fit per SM.
template <typename T, int BITS, int DC, int KB>
__global__ void __launch_bounds__(kAppendThreads, 4) append_kernel(const AppendParams p) {
  extern __shared__ float smem[];
  pdl_wait();
  pdl_release();
  const int i = blockIdx.y;
  const int h = blockIdx.z;
  const int b = p.seq_begin + i;
  const int D = DC ? DC : p.D, G = p.G, Rcap = p.Rcap;
  // token counts fit in 32 bits (capacities are below 2^31)
  const int T0 = p.old[i].total;
  const int Q0 = p.old[i].quantized;
  const int n = (int)p.n;
  const int F = (int)flush_groups(T0 - Q0, n, p.R, G);
  const int Q1 = Q0 + F * G;
  const int T1 = T0 + n;
  const int64_t unit = (int64_t)b * p.Hkv + h;
  const T* in_k = reinterpret_cast<const T*>(p.new_k) + ((int64_t)i * p.Hkv + h) * n * D;
  const T* in_v = reinterpret_cast<const T*>(p.new_v) + ((int64_t)i * p.Hkv + h) * n * D;
  T* ring_k = reinterpret_cast<T*>(p.ring_k) + unit * Rcap * D;
  T* ring_v = reinterpret_cast<T*>(p.ring_v) + unit * Rcap * D;

  if ((int)blockIdx.x >= p.flush_blocks) {
    // Window block: the new tokens that stay in the residual window, copied
    // 16 bytes at a time, four rows in flight per thread; each thread keeps
    // one column and advances its ring row without a division.
    constexpr int kVec = 16 / sizeof(T);
    constexpr int kBatch = 4;
    const int per_row = D / kVec;
    const int rows_per_pass = kAppendThreads / per_row;
    if ((int)threadIdx.x >= rows_per_pass * per_row) return;
    const int r0 = threadIdx.x / per_row, c = (threadIdx.x - r0 * per_row) * kVec;
    const int t_lo = Q1 > T0 ? Q1 : T0;
    const int rows = T1 - t_lo;
    int ring_row = (t_lo + r0) % Rcap;
    const int step = rows_per_pass % Rcap;
    for (int r = r0; r < rows; r += kBatch * rows_per_pass) {
      uint4 kv[kBatch], vv[kBatch];
      int dst[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int rr = r + k * rows_per_pass;
        dst[k] = ring_row;
        ring_row += step;
        if (ring_row >= Rcap) ring_row -= Rcap;
        if (rr < rows) {
          const size_t src = (size_t)(t_lo + rr - T0) * D + c;
          kv[k] = *reinterpret_cast<const uint4*>(in_k + src);
          vv[k] = *reinterpret_cast<const uint4*>(in_v + src);
        }
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        if (r + k * rows_per_pass < rows) {
          *reinterpret_cast<uint4*>(ring_k + (size_t)dst[k] * D + c) = kv[k];
          *reinterpret_cast<uint4*>(ring_v + (size_t)dst[k] * D + c) = vv[k];
        }
      }
    }
    return;
  }

  const int j = blockIdx.x;
  if (j >= F) return;
  const int t_first = Q0 + j * G;
  const PageGeom& geom = p.geom;
  uint8_t* page;
  if (p.map.table) {
    // paged: this group's new block, entered in the block table once
    const int32_t blk = p.blk_ids[p.blk_first[i] + j];
    page = p.pages + (int64_t)blk * p.map.block_bytes + (int64_t)h * geom.page_bytes;
    if (h == 0 && threadIdx.x == 0) p.map.table[(int64_t)b * p.map.table_stride + t_first / G] = blk;
  } else {
    page = p.pages + page_offset(p.map, geom.page_bytes, b, h, t_first / G);
  }
  // The group's rows are staged in shared memory in the input dtype.  Each
  // thread loads one 16-byte column of kVec channels, stepping over rows with
  // four loads in flight, and keeps the column's Key absmax in registers; the
  // Value absmax of a row is reduced over the threads of the row with shuffles.
  constexpr int kVec = 16 / sizeof(T);
  constexpr int kBatch = KB;
  T* tileT = reinterpret_cast<T*>(smem);                         // [G][D]
  float* sK = reinterpret_cast<float*>(tileT + (size_t)G * D);   // [D] Key scales
  float* sV = sK + D;                                            // [G] Value scales
  float* part = sV + G;                                          // [rows_per_pass][D] partial Key maxima
  const float qmax = (float)p.qmax;
  const int per_row = D / kVec;
  const int rows_per_pass = kAppendThreads / per_row;
  const bool act = (int)threadIdx.x < rows_per_pass * per_row;
  const int r0 = act ? threadIdx.x / per_row : 0, col = act ? (threadIdx.x - r0 * per_row) * kVec : 0;
  const int ring_row0 = t_first % Rcap;
  // rows of a thread in one pass of the batch loop: the same count for every
  // lane of a warp, so the shuffles below see the whole warp
  auto load_rows = [&](const T* ring, const T* input, auto&& per_row_fn) {
    for (int base = 0; base < G; base += kBatch * rows_per_pass) {
      uint4 v[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int r = base + r0 + k * rows_per_pass;
        if (act && r < G) {
          const int t = t_first + r;
          const T* src = t < T0 ? ring + (size_t)(ring_row0 + r) * D + col : input + (size_t)(t - T0) * D + col;
          v[k] = *reinterpret_cast<const uint4*>(src);
        } else {
          v[k] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int r = base + r0 + k * rows_per_pass;
        if (act && r < G) *reinterpret_cast<uint4*>(tileT + (size_t)r * D + col) = v[k];
        float x[kVec];
        unpack16(v[k], x);
        per_row_fn(r, x);
      }
    }
  };

  // With room for a second tile both tiles are copied in at once (cp.async,
  // Keys then Values): the Value latency passes while the Keys are reduced and
  // packed.  Each thread copies the rows it reads back for the maxima.
  T* tileV = p.v_prefetch ? reinterpret_cast<T*>(reinterpret_cast<uint8_t*>(smem) + flush_smem_bytes(G, D, sizeof(T)))
                          : tileT;
  if (p.v_prefetch) {
#pragma unroll
    for (int kv = 0; kv < 2; ++kv) {
      const T* ring = kv ? ring_v : ring_k;
      const T* input = kv ? in_v : in_k;
      T* tile = kv ? tileV : tileT;
      if (act) {
        // rows below ``split`` come from the ring (contiguous from ring_row0),
        // the rest from the input (row r at element in_off + r * D)
        const int split = T0 - t_first;
        const T* ring_r = ring + (size_t)ring_row0 * D + col;
        const int64_t in_off = ((int64_t)t_first - T0) * D + col;
        for (int r = r0; r < G; r += rows_per_pass)
          cp_async16(tile + (size_t)r * D + col, r < split ? ring_r + (size_t)r * D : input + (in_off + (int64_t)r * D));
      }
      asm volatile("cp.async.commit_group;\n" ::: "memory");
    }
  }

  // ---- Key: per-channel absmax over the group's tokens --------------------
  {
    float amax[kVec];
#pragma unroll
    for (int e = 0; e < kVec; ++e) amax[e] = 0.f;
    if (p.v_prefetch) {
      asm volatile("cp.async.wait_group 1;\n" ::: "memory");  // this thread's Key rows
      if (act) {
        if constexpr (sizeof(T) == 2) {
          uint32_t am[4] = {0u, 0u, 0u, 0u};  // |x| of channels col + 2k (low half), + 2k + 1 (high)
          for (int r = r0; r < G; r += rows_per_pass) {
            const uint4 v = *reinterpret_cast<const uint4*>(tileT + (size_t)r * D + col);
            am[0] = umax_u16x2(am[0], abs_bf16x2(v.x));
            am[1] = umax_u16x2(am[1], abs_bf16x2(v.y));
            am[2] = umax_u16x2(am[2], abs_bf16x2(v.z));
            am[3] = umax_u16x2(am[3], abs_bf16x2(v.w));
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            amax[2 * k] = bf16_lo_f32(am[k]);
            amax[2 * k + 1] = bf16_hi_f32(am[k]);
          }
        } else {
          for (int r = r0; r < G; r += rows_per_pass) {
            float x[kVec];
            unpack16(*reinterpret_cast<const uint4*>(tileT + (size_t)r * D + col), x);
#pragma unroll
            for (int e = 0; e < kVec; ++e) amax[e] = fmaxf(amax[e], fabsf(x[e]));
          }
        }
      }
    } else {
      load_rows(ring_k, in_k, [&](int, const float (&x)[kVec]) {
#pragma unroll
        for (int e = 0; e < kVec; ++e) amax[e] = fmaxf(amax[e], fabsf(x[e]));
      });
    }
    if (act) {
#pragma unroll
      for (int e = 0; e < kVec; ++e) part[r0 * D + col + e] = amax[e];
    }
    __syncthreads();
    float kmx = 0.f;
    for (int c = threadIdx.x; c < D; c += kAppendThreads) {
      float a = 0.f;
      for (int r = 0; r < rows_per_pass; ++r) a = fmaxf(a, part[r * D + c]);
      sK[c] = __fdiv_rn(qmax, fmaxf(a, p.eps));
      kmx = fmaxf(kmx, a);
    }
    // the unit's largest flushed Key absmax (the decode's range guard)
    for (int o = 16; o > 0; o >>= 1) kmx = fmaxf(kmx, __shfl_xor_sync(0xffffffffu, kmx, o));
    if ((threadIdx.x & 31) == 0 && kmx > 0.f && p.range) atomicMax(p.range + 2 * unit, __float_as_uint(kmx));
    __syncthreads();
  }
  {
    // rows of D*BITS/8 bytes, written as 32-bit words; each thread keeps one
    // word column (and its scales) and steps over the token rows
    constexpr int kPerWord = 32 / BITS;  // codes per 32-bit word
    const int words_per_row = D / kPerWord;
    const int rows_pp = kAppendThreads / words_per_row;
    uint32_t* kc = reinterpret_cast<uint32_t*>(page);
    if ((int)threadIdx.x < rows_pp * words_per_row) {
      const int t0 = threadIdx.x / words_per_row, w = threadIdx.x - t0 * words_per_row;
      float sc[kPerWord];
#pragma unroll
      for (int k = 0; k < kPerWord; ++k) sc[k] = sK[w * kPerWord + k];
      for (int t = t0; t < G; t += rows_pp) {
        float x[kPerWord];
        load_elems<T, kPerWord>(tileT + (size_t)t * D + w * kPerWord, x);
        uint32_t c[kPerWord];
#pragma unroll
        for (int k = 0; k < kPerWord; ++k) c[k] = quantize_bits<BITS>(x[k], sc[k]);
        uint32_t word = 0;  // channel k of the word in field k
        if constexpr (BITS == 4) {
          word = pack_nibbles(c[0], c[2], c[4], c[6], c[1], c[3], c[5], c[7]);
        } else if constexpr (BITS == 8) {
          word = low_bytes(c[0], c[1], c[2], c[3]);
        } else {
#pragma unroll
          for (int k = 0; k < kPerWord; ++k) word |= code_field<BITS>(c[k], k);
        }
        kc[t * words_per_row + w] = word;
      }
    }
    float* ks = reinterpret_cast<float*>(page + geom.kscale_off);
    for (int c = threadIdx.x; c < D; c += kAppendThreads) ks[c] = sK[c];
  }
  __syncthreads();  // the tile is rewritten with the Values

  // ---- Value: per-token absmax over head_dim -----------------------------
  {
    const bool shuffle_rows = (per_row & (per_row - 1)) == 0 && per_row <= 32;
    uint32_t* rmax = reinterpret_cast<uint32_t*>(part);  // [G] bits of row maxima (other widths)
    if (!shuffle_rows) {
      for (int t = threadIdx.x; t < G; t += kAppendThreads) rmax[t] = 0u;
      __syncthreads();
    }
    auto row_max = [&](int r, const float (&x)[kVec]) {
      float a = 0.f;
#pragma unroll
      for (int e = 0; e < kVec; ++e) a = fmaxf(a, fabsf(x[e]));
      if (shuffle_rows) {
        for (int o = 1; o < per_row; o <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        if (act && r < G && col == 0) sV[r] = a;  // the row's absmax; its scale below
      } else if (act && r < G) {
        atomicMax(rmax + r, __float_as_uint(a));
      }
    };
    if (p.v_prefetch) {
      asm volatile("cp.async.wait_group 0;\n" ::: "memory");
      __syncthreads();
      // the same rows per thread as the copies, read back from the tile
      for (int base = 0; base < G; base += kBatch * rows_per_pass) {
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          const int r = base + r0 + k * rows_per_pass;
          const uint4 v = act && r < G ? *reinterpret_cast<const uint4*>(tileV + (size_t)r * D + col)
                                       : make_uint4(0u, 0u, 0u, 0u);
          if constexpr (sizeof(T) == 2) {
            // the row's |x| maximum over this thread's 8 channels, packed, then
            // as the same one-element row_max input
            const uint32_t m2 = umax_u16x2(umax_u16x2(abs_bf16x2(v.x), abs_bf16x2(v.y)),
                                           umax_u16x2(abs_bf16x2(v.z), abs_bf16x2(v.w)));
            float x[kVec];
            x[0] = fmaxf(bf16_lo_f32(m2), bf16_hi_f32(m2));
#pragma unroll
            for (int e = 1; e < kVec; ++e) x[e] = 0.f;
            row_max(r, x);
          } else {
            float x[kVec];
            unpack16(v, x);
            row_max(r, x);
          }
        }
      }
    } else {
      load_rows(ring_v, in_v, row_max);
    }
    __syncthreads();
    // one division per token, spread over the CTA (not inside the row loop)
    float vmx = 0.f;
    for (int t = threadIdx.x; t < G; t += kAppendThreads) {
      const float a = shuffle_rows ? sV[t] : __uint_as_float(rmax[t]);
      sV[t] = __fdiv_rn(qmax, fmaxf(a, p.eps));
      vmx = fmaxf(vmx, a);
    }
    for (int o = 16; o > 0; o >>= 1) vmx = fmaxf(vmx, __shfl_xor_sync(0xffffffffu, vmx, o));
    if ((threadIdx.x & 31) == 0 && vmx > 0.f && p.range) atomicMax(p.range + 2 * unit + 1, __float_as_uint(vmx));
    __syncthreads();
  }
  {
    // Value sub-tiles of 32 tokens, channel-major.  A work item is 8 tokens x 2
    // channels: eight 2-channel loads from the tile, both channels' codes packed
    // in registers (a word's token order is fixed), then one 4-bit word, one
    // 2-bit piece or two 8-bit words per channel.
    uint8_t* vbase = page + geom.code_bytes;
    const int n_cp = D / 2;
    for (int item = threadIdx.x; item < (G / 8) * n_cp; item += kAppendThreads) {
      const int oct = item / n_cp, c = 2 * (item - oct * n_cp), t8 = 8 * oct;
      const int st = t8 >> 5, n_st = min(32, G - 32 * st), o8 = (t8 & 31) >> 3;  // sub-tile, its length, octet
      PairOf<T> xp[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) xp[k].load(tileV + (size_t)(t8 + k) * D + c);
      uint8_t* sub = vbase + (int64_t)st * 32 * D * BITS / 8;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        uint32_t cv[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) cv[k] = quantize_bits<BITS>(xp[k].get(e), sV[t8 + k]);
        if (BITS == 4) {
          // nibbles 0..7 hold tokens 0, 2, 4, 6, 1, 3, 5, 7: bytes 0..3 pair
          // tokens (0, 2), (4, 6), (1, 3), (5, 7)
          reinterpret_cast<uint32_t*>(sub)[(c + e) * (n_st / 8) + o8] =
              pack_nibbles(cv[0], cv[4], cv[1], cv[5], cv[2], cv[6], cv[3], cv[7]);
        } else if (BITS == 2) {
          uint32_t piece = 0;  // token 2f in bits 2f, token 2f + 1 in bits 8 + 2f
#pragma unroll
          for (int k = 0; k < 8; ++k) piece |= code_field<2>(cv[k], (k & 1) * 4 + (k >> 1));
          reinterpret_cast<uint16_t*>(sub)[(c + e) * (n_st / 8) + o8] = (uint16_t)piece;
        } else {
          // byte k of word w holds token 4 w + k
          uint32_t* vc = reinterpret_cast<uint32_t*>(sub) + (c + e) * (n_st / 4) + 2 * o8;
          vc[0] = low_bytes(cv[0], cv[1], cv[2], cv[3]);
          vc[1] = low_bytes(cv[4], cv[5], cv[6], cv[7]);
        }
      }
    }
    float* vs = reinterpret_cast<float*>(page + geom.vscale_off);
    for (int t = threadIdx.x; t < G; t += kAppendThreads) vs[t] = sV[t];
  }
}

// The datawhale page's compare ("54. KV Cache Quantization Strategies",
// compare): quantize a Key/Value pair with the flush's quantizer (Key per
// channel over group_len tokens, Value per token over head_dim), restore
// (code / max(scale, eps)) and sum the squared errors (x - x_hat)^2, each
// difference and square rounded in fp32 as the page computes them, the sums
// in fp64.  One CTA per (Key-scale group, row); rows are the flattened
// [batch, heads] of the input.
constexpr int kCompareThreads = 256;

template <typename T>
__device__ __forceinline__ float load_f32(const T* p, int64_t i) {
  if constexpr (sizeof(T) == 2) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
  else return reinterpret_cast<const float*>(p)[i];
}

template <typename T>
__global__ void __launch_bounds__(kCompareThreads) compare_kernel(const CompareParams p) {
  __shared__ double red[2][kCompareThreads / 32];
  pdl_wait();
  pdl_release();
  const int D = p.D, L = p.group_len;
  const float qmax = (float)p.qmax;
  const int64_t base = ((int64_t)blockIdx.y * p.tokens + (int64_t)blockIdx.x * L) * D;
  const T* kx = reinterpret_cast<const T*>(p.key) + base;
  const T* vx = reinterpret_cast<const T*>(p.value) + base;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  double ek = 0.0, ev = 0.0;
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    float a = 0.f;
    for (int t = 0; t < L; ++t) a = fmaxf(a, fabsf(load_f32(kx, (int64_t)t * D + c)));
    const float scale = __fdiv_rn(qmax, fmaxf(a, p.eps));
    const float r = fmaxf(scale, p.eps);
    for (int t = 0; t < L; ++t) {
      const float x = load_f32(kx, (int64_t)t * D + c);
      const float e = __fsub_rn(x, __fdiv_rn((float)quantize_one(x, scale, qmax), r));
      ek += (double)__fmul_rn(e, e);
    }
  }
  for (int t = warp; t < L; t += nwarps) {
    float a = 0.f;
    for (int c = lane; c < D; c += 32) a = fmaxf(a, fabsf(load_f32(vx, (int64_t)t * D + c)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    const float scale = __fdiv_rn(qmax, fmaxf(a, p.eps));
    const float r = fmaxf(scale, p.eps);
    for (int c = lane; c < D; c += 32) {
      const float x = load_f32(vx, (int64_t)t * D + c);
      const float e = __fsub_rn(x, __fdiv_rn((float)quantize_one(x, scale, qmax), r));
      ev += (double)__fmul_rn(e, e);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    ek += __shfl_xor_sync(0xffffffffu, ek, o);
    ev += __shfl_xor_sync(0xffffffffu, ev, o);
  }
  if (lane == 0) {
    red[0][warp] = ek;
    red[1][warp] = ev;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double sk = 0.0, sv = 0.0;
    for (int w = 0; w < nwarps; ++w) {
      sk += red[0][w];
      sv += red[1][w];
    }
    atomicAdd(p.sums, sk);
    atomicAdd(p.sums + 1, sv);
  }
}

template <typename T, int BITS, int KB>
cudaError_t launch_kb(const AppendParams& p, const dim3& grid, size_t smem, cudaStream_t s) {
  if (p.D == 128) return launch_pdl(append_kernel<T, BITS, 128, KB>, grid, dim3(kAppendThreads), smem, s, p);
  if (p.D == 64) return launch_pdl(append_kernel<T, BITS, 64, KB>, grid, dim3(kAppendThreads), smem, s, p);
  return launch_pdl(append_kernel<T, BITS, 0, KB>, grid, dim3(kAppendThreads), smem, s, p);
}

template <typename T, int BITS>
cudaError_t launch_t(const AppendParams& p, cudaStream_t s) {
  const dim3 grid(p.flush_blocks + p.window_blocks, p.n_seqs, p.Hkv);
  const size_t smem = p.flush_blocks ? flush_launch_smem(p.G, p.D, (int)sizeof(T)) : 0;
  const int rows_per_pass = kAppendThreads / (p.D / (16 / (int)sizeof(T)));
  return p.G <= 2 * rows_per_pass ? launch_kb<T, BITS, 2>(p, grid, smem, s) : launch_kb<T, BITS, 4>(p, grid, smem, s);
}
template <typename T, int BITS, int KB>
cudaError_t configure_kb(size_t smem) {
  cudaError_t e = cudaFuncSetAttribute(append_kernel<T, BITS, 0, KB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(append_kernel<T, BITS, 64, KB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(append_kernel<T, BITS, 128, KB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  return e;
}
template <typename T, int BITS>
cudaError_t configure_t(size_t smem) {
  const cudaError_t e = configure_kb<T, BITS, 2>(smem);
  return e == cudaSuccess ? configure_kb<T, BITS, 4>(smem) : e;
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, int dtype, cudaStream_t s) {
  if (dtype == 0) {
    if (p.bits == 2) return launch_t<__nv_bfloat16, 2>(p, s);
    return p.bits == 4 ? launch_t<__nv_bfloat16, 4>(p, s) : launch_t<__nv_bfloat16, 8>(p, s);
  }
  if (p.bits == 2) return launch_t<float, 2>(p, s);
  return p.bits == 4 ? launch_t<float, 4>(p, s) : launch_t<float, 8>(p, s);
}

cudaError_t launch_compare(const CompareParams& p, int64_t rows, cudaStream_t s) {
  const dim3 grid((unsigned)(p.tokens / p.group_len), (unsigned)rows);
  if (p.dtype == 0) return launch_pdl(compare_kernel<__nv_bfloat16>, grid, dim3(kCompareThreads), 0, s, p);
  return launch_pdl(compare_kernel<float>, grid, dim3(kCompareThreads), 0, s, p);
}

cudaError_t configure_append(int dtype, int bits, size_t smem_bytes) {
  if (dtype == 0) {
    if (bits == 2) return configure_t<__nv_bfloat16, 2>(smem_bytes);
    return bits == 4 ? configure_t<__nv_bfloat16, 4>(smem_bytes) : configure_t<__nv_bfloat16, 8>(smem_bytes);
  }
  if (bits == 2) return configure_t<float, 2>(smem_bytes);
  return bits == 4 ? configure_t<float, 4>(smem_bytes) : configure_t<float, 8>(smem_bytes);
}

}  // namespace kvq
