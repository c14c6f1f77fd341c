// Segmented cache: the flush rule of "54. KV Cache Quantization Strategies"
// (append_and_partition) verbatim.  An append of n tokens to a window of L
// flushes max(L + n - R, 0) tokens -- the oldest -- as ONE new segment: Key
// quantized per channel over all of the segment's tokens, Value per token
// (Step 2; scale = qmax / max(absmax, eps), code = clamp(rint(x * scale))),
// and the newest min(L + n, R) tokens stay in the window.
//
// A segment may hold any number of tokens (a whole prefill), so its Key
// absmax is a reduction across CTAs: pass 1 takes each 32-token chunk's
// per-channel absmax into an atomicMax per channel (the float bits of values
// >= 0 order like unsigned integers) and, since Value scales are per token,
// writes the Value codes and scales at once; pass 2 quantizes the Keys with
// the final scales.  Codes are token-major rows packed like a group page's Key
// rows; a segment's Key scale row is stored once, in the row of its first
// token, and every token records that first token.

#include <cuda_bf16.h>

#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kSegThreads = 256;
constexpr int kSegChunk = 32;  // tokens per CTA

template <typename T>
__device__ __forceinline__ float ldf(const T* p, int64_t i) {
  if constexpr (sizeof(T) == 2) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
  else return reinterpret_cast<const float*>(p)[i];
}

__device__ __forceinline__ int quant(float x, float scale, float qmax) {
  float r = rintf(__fmul_rn(x, scale));
  return (int)fminf(fmaxf(r, -qmax), qmax);
}

template <int BITS>
__device__ __forceinline__ int row_code(const uint8_t* row, int c) {
  if (BITS == 2) return (int)((row[c >> 2] >> (2 * (c & 3))) & 0x3) - 2;
  if (BITS == 4) return (int)((row[c >> 1] >> (4 * (c & 1))) & 0xF) - 8;
  return (int)row[c] - 128;
}

// The chunk's tokens as fp32 rows in shared memory: tokens below T0 from the
// window ring (row t mod R), later ones from the input.
template <typename T>
__device__ void load_rows(float* tile, const SegFlushParams& p, int i, int h, int t_begin, int cnt, int T0) {
  const int D = p.D;
  const int b = p.seq_begin + i;
  const int64_t unit = (int64_t)b * p.Hkv + h;
  const T* ring_k = reinterpret_cast<const T*>(p.ring_k) + unit * p.R * D;
  const T* in_k = reinterpret_cast<const T*>(p.new_k) + ((int64_t)i * p.Hkv + h) * p.n * D;
  for (int idx = threadIdx.x; idx < cnt * D; idx += blockDim.x) {
    const int r = idx / D, c = idx - r * D;
    const int t = t_begin + r;
    tile[idx] = t < T0 ? ldf(ring_k, (int64_t)(t % p.R) * D + c) : ldf(in_k, (int64_t)(t - T0) * D + c);
  }
}

// Code rows of ``cnt`` tokens: 32-bit words of 32 / BITS codes, offset binary;
// per-channel scales (Keys) or one scale per token (Values).
template <int BITS>
__device__ void pack_rows(uint8_t* rows, int row_bytes, const float* tile, int cnt, int D, const float* scale,
                          bool per_token, float qmax) {
  constexpr int kPerWord = 32 / BITS;
  constexpr int kBias = BITS == 2 ? 2 : BITS == 4 ? 8 : 128;
  const int wpr = D / kPerWord;
  for (int idx = threadIdx.x; idx < cnt * wpr; idx += blockDim.x) {
    const int r = idx / wpr, w = idx - r * wpr;
    uint32_t word = 0;
#pragma unroll
    for (int k = 0; k < kPerWord; ++k) {
      const int c = w * kPerWord + k;
      const float s = per_token ? scale[r] : scale[c];
      word |= (uint32_t)(quant(tile[r * D + c], s, qmax) + kBias) << (BITS * k);
    }
    reinterpret_cast<uint32_t*>(rows + (int64_t)r * row_bytes)[w] = word;
  }
}

// the segment of sequence i in this append: [Q0, Q0 + F)
__device__ __forceinline__ void segment(const SegFlushParams& p, int i, int* T0, int* Q0, int* F) {
  *T0 = p.old[i].total;
  *Q0 = p.old[i].quantized;
  const int tail = *T0 - *Q0 + (int)p.n;
  *F = tail > p.R ? tail - p.R : 0;
}

template <typename T, int BITS>
__global__ void __launch_bounds__(kSegThreads) seg_pass1_kernel(const SegFlushParams p) {
  extern __shared__ float smem[];
  pdl_wait();
  pdl_release();
  const int i = blockIdx.y, h = blockIdx.z;
  int T0, Q0, F;
  segment(p, i, &T0, &Q0, &F);
  const int off = blockIdx.x * kSegChunk;
  if (off >= F) return;
  const int cnt = min(kSegChunk, F - off), t_begin = Q0 + off;
  const int D = p.D;
  const int64_t unit = (int64_t)(p.seq_begin + i) * p.Hkv + h;
  float* tile = smem;
  float* sV = tile + kSegChunk * D;
  const float qmax = (float)p.qmax;
  // ---- Keys: this chunk's per-channel absmax into the segment's maxima ------
  load_rows<T>(tile, p, i, h, t_begin, cnt, T0);
  __syncthreads();
  float amax = 0.f;
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    float a = 0.f;
    for (int r = 0; r < cnt; ++r) a = fmaxf(a, fabsf(tile[r * D + c]));
    atomicMax(p.kmax + unit * D + c, __float_as_uint(a));
    amax = fmaxf(amax, a);
  }
  // the unit's largest flushed Key absmax, for the decode's range test
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0 && amax > 0.f) atomicMax(p.range + 2 * unit, __float_as_uint(amax));
  __syncthreads();
  // ---- Values: per-token scale and codes --------------------------------
  SegFlushParams q = p;
  q.ring_k = p.ring_v;
  q.new_k = p.new_v;
  load_rows<T>(tile, q, i, h, t_begin, cnt, T0);
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int r = warp; r < cnt; r += blockDim.x >> 5) {
    float a = 0.f;
    for (int c = lane; c < D; c += 32) a = fmaxf(a, fabsf(tile[r * D + c]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    if (lane == 0) {
      sV[r] = __fdiv_rn(qmax, fmaxf(a, p.eps));
      p.seg.vscales[unit * p.seg.cap + t_begin + r] = sV[r];
      if (a > 0.f) atomicMax(p.range + 2 * unit + 1, __float_as_uint(a));
    }
  }
  __syncthreads();
  pack_rows<BITS>(p.seg.vcodes + (unit * p.seg.cap + t_begin) * p.seg.row_bytes, p.seg.row_bytes, tile, cnt, D,
                  sV, true, qmax);
}

template <typename T, int BITS>
__global__ void __launch_bounds__(kSegThreads) seg_pass2_kernel(const SegFlushParams p) {
  extern __shared__ float smem[];
  pdl_wait();
  pdl_release();
  const int i = blockIdx.y, h = blockIdx.z;
  int T0, Q0, F;
  segment(p, i, &T0, &Q0, &F);
  const int off = blockIdx.x * kSegChunk;
  if (off >= F) return;
  const int cnt = min(kSegChunk, F - off), t_begin = Q0 + off;
  const int D = p.D;
  const int64_t unit = (int64_t)(p.seq_begin + i) * p.Hkv + h;
  float* tile = smem;
  float* sK = tile + kSegChunk * D;
  const float qmax = (float)p.qmax;
  load_rows<T>(tile, p, i, h, t_begin, cnt, T0);
  for (int c = threadIdx.x; c < D; c += blockDim.x)
    sK[c] = __fdiv_rn(qmax, fmaxf(__uint_as_float(p.kmax[unit * D + c]), p.eps));
  __syncthreads();
  pack_rows<BITS>(p.seg.kcodes + (unit * p.seg.cap + t_begin) * p.seg.row_bytes, p.seg.row_bytes, tile, cnt, D,
                  sK, false, qmax);
  if (off == 0) {
    float* ks = p.seg.kscales + (unit * p.seg.cap + Q0) * D;
    for (int c = threadIdx.x; c < D; c += blockDim.x) ks[c] = sK[c];
  }
  if (h == 0) {
    int32_t* first = p.seg.first + (int64_t)(p.seq_begin + i) * p.seg.cap + t_begin;
    for (int r = threadIdx.x; r < cnt; r += blockDim.x) first[r] = Q0;
  }
}

// The new tokens that stay in the window, into their ring rows (t mod R).
template <typename T>
__global__ void __launch_bounds__(kSegThreads) seg_window_kernel(const SegFlushParams p) {
  pdl_wait();
  pdl_release();
  const int i = blockIdx.y, h = blockIdx.z;
  const int D = p.D;
  const int T0 = p.old[i].total, Q0 = p.old[i].quantized;
  const int T1 = T0 + (int)p.n;
  const int W1 = min(T0 - Q0 + (int)p.n, p.R);
  const int t_lo = max(T1 - W1, T0);
  const int64_t unit = (int64_t)(p.seq_begin + i) * p.Hkv + h;
  const T* in_k = reinterpret_cast<const T*>(p.new_k) + ((int64_t)i * p.Hkv + h) * p.n * D;
  const T* in_v = reinterpret_cast<const T*>(p.new_v) + ((int64_t)i * p.Hkv + h) * p.n * D;
  T* rk = reinterpret_cast<T*>(p.ring_k_out) + unit * p.R * D;
  T* rv = reinterpret_cast<T*>(p.ring_v_out) + unit * p.R * D;
  for (int idx = threadIdx.x; idx < (T1 - t_lo) * D; idx += blockDim.x) {
    const int r = idx / D, c = idx - r * D;
    const int t = t_lo + r;
    rk[(int64_t)(t % p.R) * D + c] = in_k[(int64_t)(t - T0) * D + c];
    rv[(int64_t)(t % p.R) * D + c] = in_v[(int64_t)(t - T0) * D + c];
  }
}

// restore of a segmented cache: one CTA per (32 rows, unit)
template <int BITS>
__global__ void __launch_bounds__(kSegThreads) seg_restore_kernel(const RestoreParams p) {
  pdl_wait();
  pdl_release();
  const int n_units = p.n_seqs * p.Hkv;
  const int col = blockIdx.x / n_units, u = blockIdx.x - col * n_units;
  const int i = u / p.Hkv, h = u - i * p.Hkv;
  const int D = p.D;
  const int T0 = p.ctr[i].total, Q0 = p.ctr[i].quantized;
  const int r0 = col * kSegChunk;
  if (r0 >= T0) return;
  const int cnt = min(kSegChunk, T0 - r0);
  const int64_t unit = (int64_t)(p.seq_begin + i) * p.Hkv + h;
  const int64_t out_unit = ((int64_t)i * p.Hkv + h) * p.t_stride;
  for (int idx = threadIdx.x; idx < cnt * D; idx += blockDim.x) {
    const int r = idx / D, c = idx - r * D;
    const int t = r0 + r;
    float kx, vx;
    if (t < Q0) {
      const int64_t row = unit * p.seg.cap + t;
      const int64_t srow = unit * p.seg.cap + p.seg.first[(int64_t)(p.seq_begin + i) * p.seg.cap + t];
      kx = __fdiv_rn((float)row_code<BITS>(p.seg.kcodes + row * p.seg.row_bytes, c),
                     fmaxf(p.seg.kscales[srow * D + c], p.eps));
      vx = __fdiv_rn((float)row_code<BITS>(p.seg.vcodes + row * p.seg.row_bytes, c), fmaxf(p.seg.vscales[row], p.eps));
    } else {
      const int64_t src = (unit * p.Rcap + t % p.Rcap) * D + c;
      if (p.in_dtype == 0) {
        kx = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.ring_k)[src]);
        vx = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.ring_v)[src]);
      } else {
        kx = reinterpret_cast<const float*>(p.ring_k)[src];
        vx = reinterpret_cast<const float*>(p.ring_v)[src];
      }
    }
    const int64_t dst = (out_unit + t) * D + c;
    if (p.out_dtype == 0) {
      reinterpret_cast<__nv_bfloat16*>(p.k_out)[dst] = __float2bfloat16_rn(kx);
      reinterpret_cast<__nv_bfloat16*>(p.v_out)[dst] = __float2bfloat16_rn(vx);
    } else {
      reinterpret_cast<float*>(p.k_out)[dst] = kx;
      reinterpret_cast<float*>(p.v_out)[dst] = vx;
    }
  }
}

template <typename T, int BITS>
cudaError_t flush_t(const SegFlushParams& p, int64_t max_tokens, cudaStream_t s) {
  const dim3 grid((unsigned)((max_tokens + kSegChunk - 1) / kSegChunk), p.n_seqs, p.Hkv);
  const size_t smem = ((size_t)kSegChunk * p.D + kSegChunk + p.D) * sizeof(float);
  cudaError_t e = launch_pdl(seg_pass1_kernel<T, BITS>, grid, dim3(kSegThreads), smem, s, p);
  if (e == cudaSuccess) e = launch_pdl(seg_pass2_kernel<T, BITS>, grid, dim3(kSegThreads), smem, s, p);
  return e;
}

template <typename T>
cudaError_t flush_b(const SegFlushParams& p, int64_t max_tokens, cudaStream_t s) {
  return p.bits == 2 ? flush_t<T, 2>(p, max_tokens, s) : p.bits == 4 ? flush_t<T, 4>(p, max_tokens, s)
                                                                      : flush_t<T, 8>(p, max_tokens, s);
}

}  // namespace

cudaError_t launch_seg_flush(const SegFlushParams& p, int dtype, int64_t max_tokens, cudaStream_t s) {
  if (max_tokens <= 0) return cudaSuccess;
  return dtype == 0 ? flush_b<__nv_bfloat16>(p, max_tokens, s) : flush_b<float>(p, max_tokens, s);
}

cudaError_t launch_seg_window(const SegFlushParams& p, int dtype, cudaStream_t s) {
  const dim3 grid(1, p.n_seqs, p.Hkv);
  return dtype == 0 ? launch_pdl(seg_window_kernel<__nv_bfloat16>, grid, dim3(kSegThreads), 0, s, p)
                    : launch_pdl(seg_window_kernel<float>, grid, dim3(kSegThreads), 0, s, p);
}

cudaError_t launch_seg_restore(const RestoreParams& p, int64_t max_tokens, cudaStream_t s) {
  const int cols = (int)((max_tokens + kSegChunk - 1) / kSegChunk);
  if (cols == 0) return cudaSuccess;
  const dim3 grid(cols * p.n_seqs * p.Hkv);
  if (p.bits == 2) return launch_pdl(seg_restore_kernel<2>, grid, dim3(kSegThreads), 0, s, p);
  if (p.bits == 4) return launch_pdl(seg_restore_kernel<4>, grid, dim3(kSegThreads), 0, s, p);
  return launch_pdl(seg_restore_kernel<8>, grid, dim3(kSegThreads), 0, s, p);
}

}  // namespace kvq
