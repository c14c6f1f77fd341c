// Dequantize a cache into dense Key/Value tensors (kvq_restore): the first
// half of the dequantize-to-HBM read path ("KV Cache 量化与压缩" section 06,
// path (a)), kept as the measured foil of the fused decode kernel.
//
// Row t < quantized of a unit is restore(code, scale) = code / max(scale, eps)
// in fp32 ("54. KV Cache Quantization Strategies", restore): Key codes over the
// page's per-channel scales, Value codes over the per-token scales; rows from
// quantized to total are the residual window as held.  A CTA per (run of four
// pages, unit) stages its pages in shared memory with cp.async, the next page
// in flight while the current one is decoded, decodes the
// offset-binary codes of the layout in kvq.h (the channel-major Value codes
// through a shared [G][D] tile) and writes 8 channels per thread (16- or
// 32-byte stores); the last grid column copies the window rows.

#include <cuda_bf16.h>

#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kRestoreThreads = 256;
constexpr int kRestorePages = 4;  // pages per CTA, double-buffered

__device__ __forceinline__ void cpa16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cpa_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cpa_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

// Key codes of channels c8 .. c8 + 7 of token t, as signed integers.
__device__ __forceinline__ void key_codes8(const uint8_t* page, int t, int c8, int D, int bits, int (&code)[8]) {
  if (bits == 2) {
    const uint32_t v = *reinterpret_cast<const uint16_t*>(page + t * (D / 4) + c8 / 4);
#pragma unroll
    for (int e = 0; e < 8; ++e) code[e] = (int)((v >> (2 * e)) & 0x3) - 2;
  } else if (bits == 4) {
    const uint32_t v = *reinterpret_cast<const uint32_t*>(page + t * (D / 2) + c8 / 2);
#pragma unroll
    for (int e = 0; e < 8; ++e) code[e] = (int)((v >> (4 * e)) & 0xF) - 8;
  } else {
    const uint2 v = *reinterpret_cast<const uint2*>(page + t * D + c8);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      code[e] = (int)((v.x >> (8 * e)) & 0xFF) - 128;
      code[4 + e] = (int)((v.y >> (8 * e)) & 0xFF) - 128;
    }
  }
}

__device__ __forceinline__ void store8(void* out, int64_t elem, const float (&x)[8], int out_dtype) {
  if (out_dtype == 0) {
    uint4 w;
    uint32_t* u = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
      u[e] = *reinterpret_cast<const uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(out) + elem) = w;
  } else {
    float4* o = reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + elem);
    o[0] = make_float4(x[0], x[1], x[2], x[3]);
    o[1] = make_float4(x[4], x[5], x[6], x[7]);
  }
}

__device__ __forceinline__ void load8(const void* in, int64_t elem, float (&x)[8], int in_dtype) {
  if (in_dtype == 0) {
    const uint4 w = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(in) + elem);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(h[e]);
      x[2 * e] = f.x;
      x[2 * e + 1] = f.y;
    }
  } else {
    const float4* f = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(in) + elem);
    const float4 a = f[0], b = f[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
}

__global__ void __launch_bounds__(kRestoreThreads) restore_kernel(const RestoreParams p) {
  extern __shared__ __align__(16) uint8_t page[];
  pdl_wait();
  pdl_release();
  const int n_units = p.n_seqs * p.Hkv;
  const int col = blockIdx.x / n_units;
  const int u = blockIdx.x - col * n_units;
  const int i = u / p.Hkv, h = u - i * p.Hkv;
  const int b = p.seq_begin + i;
  const int D = p.D, G = p.G;
  const int T0 = p.ctr[i].total, Q0 = p.ctr[i].quantized;
  const int64_t out_unit = ((int64_t)i * p.Hkv + h) * p.t_stride;  // first row of the unit in the output
  const int per_row = D / 8;

  if (col == p.page_cols) {
    // the window rows, as held in the ring
    const int64_t unit = (int64_t)b * p.Hkv + h;
    const int esz = p.in_dtype == 0 ? 2 : 4;
    const uint8_t* rk = reinterpret_cast<const uint8_t*>(p.ring_k) + unit * p.Rcap * D * esz;
    const uint8_t* rv = reinterpret_cast<const uint8_t*>(p.ring_v) + unit * p.Rcap * D * esz;
    for (int idx = threadIdx.x; idx < (T0 - Q0) * per_row; idx += blockDim.x) {
      const int r = idx / per_row, c8 = (idx - r * per_row) * 8;
      const int t = Q0 + r;
      const int64_t src = (int64_t)(t % p.Rcap) * D + c8;
      float x[8];
      load8(rk, src, x, p.in_dtype);
      store8(p.k_out, (out_unit + t) * D + c8, x, p.out_dtype);
      load8(rv, src, x, p.in_dtype);
      store8(p.v_out, (out_unit + t) * D + c8, x, p.out_dtype);
    }
    return;
  }
  const int P = Q0 / G;
  const int pg_begin = col * kRestorePages;
  if (pg_begin >= P) return;
  const int pg_end = min(P, pg_begin + kRestorePages);
  const PageGeom& geom = p.geom;
  const int pbytes = (int)geom.page_bytes;  // a multiple of 16

  uint8_t* buf[2] = {page, page + pbytes};
  float* vtile = reinterpret_cast<float*>(page + 2 * pbytes);  // [G][D]
  // Restored values m / max(scale, eps) for every magnitude m of a code (2 for
  // 2-bit, 8 for 4-bit codes): a code c restores to +-table[|c|], which is
  // exactly c / max(scale, eps) since IEEE division is sign-symmetric.  8-bit
  // codes (128 magnitudes) divide directly.
  const int nm = p.bits == 2 ? 2 : p.bits == 4 ? 8 : 0;
  float* ktab = vtile + G * D;  // [nm][D]
  float* vtab = ktab + nm * D;  // [G][nm]
  auto issue = [&](int pg, uint8_t* dst) {
    const uint8_t* src = p.pages + page_offset(p.map, pbytes, b, h, pg);
    for (int o = threadIdx.x * 16; o < pbytes; o += blockDim.x * 16) cpa16(dst + o, src + o);
    cpa_commit();
  };
  issue(pg_begin, buf[0]);
  for (int pg = pg_begin; pg < pg_end; ++pg) {
    uint8_t* cur = buf[(pg - pg_begin) & 1];
    if (pg + 1 < pg_end) {
      issue(pg + 1, buf[(pg + 1 - pg_begin) & 1]);
      cpa_wait<1>();
    } else {
      cpa_wait<0>();
    }
    __syncthreads();
    const float* ks = reinterpret_cast<const float*>(cur + geom.kscale_off);
    const float* vs = reinterpret_cast<const float*>(cur + geom.vscale_off);
    const uint8_t* vbase = cur + geom.code_bytes;
    for (int idx = threadIdx.x; idx < nm * D; idx += blockDim.x) {
      const int m = idx / D, c = idx - m * D;
      ktab[idx] = __fdiv_rn((float)m, fmaxf(ks[c], p.eps));
    }
    for (int idx = threadIdx.x; idx < nm * G; idx += blockDim.x) {
      const int t = idx / nm, m = idx - t * nm;
      vtab[idx] = __fdiv_rn((float)m, fmaxf(vs[t], p.eps));
    }
    __syncthreads();
    const int64_t row0 = out_unit + (int64_t)pg * G;
    // Value codes: one thread per (channel, 8-token unit of its sub-tile row: a
    // 32-bit word at 4 bits, a 16-bit piece at 2 bits; 4 tokens a word at 8
    // bits), the unit's tokens restored into a [G][D] tile (consecutive
    // threads, consecutive channels: no bank conflicts on the tile)
    const int tpu = p.bits == 8 ? 4 : 8;  // tokens per unit
    for (int idx = threadIdx.x; idx < G * D / tpu; idx += blockDim.x) {
      const int ui = idx / D, c = idx - ui * D;
      const int t0 = ui * tpu;
      const int st = t0 / 32, n_st = min(32, G - 32 * st);
      const uint8_t* row = vbase + (size_t)st * 32 * D * p.bits / 8 + (size_t)c * (n_st * p.bits / 8);
      const int uo = (t0 - 32 * st) / tpu;
      const uint32_t unit = p.bits == 2 ? (uint32_t)reinterpret_cast<const uint16_t*>(row)[uo]
                                        : reinterpret_cast<const uint32_t*>(row)[uo];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (j >= tpu) break;
        int t, code;
        if (p.bits == 2) {
          t = t0 + 2 * (j & 3) + (j >> 2);
          code = (int)((unit >> ((j >> 2) * 8 + 2 * (j & 3))) & 0x3) - 2;
        } else if (p.bits == 4) {
          t = t0 + (j < 4 ? 2 * j : 2 * (j - 4) + 1);
          code = (int)((unit >> (4 * j)) & 0xF) - 8;
        } else {
          t = t0 + j;
          code = (int)((unit >> (8 * j)) & 0xFF) - 128;
        }
        float x;
        if (nm) {
          const float r = vtab[t * nm + (code < 0 ? -code : code)];
          x = code < 0 ? -r : r;
        } else {
          x = __fdiv_rn((float)code, fmaxf(vs[t], p.eps));
        }
        vtile[t * D + c] = x;
      }
    }
    __syncthreads();
    // Key codes: one thread per (token, 8 channels); both rows go out as
    // 16-byte (bf16) or 32-byte (fp32) stores
    for (int idx = threadIdx.x; idx < G * per_row; idx += blockDim.x) {
      const int t = idx / per_row, c8 = (idx - t * per_row) * 8;
      int code[8];
      key_codes8(cur, t, c8, D, p.bits, code);
      float x[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (nm) {
          const float r = ktab[(code[e] < 0 ? -code[e] : code[e]) * D + c8 + e];
          x[e] = code[e] < 0 ? -r : r;
        } else {
          x[e] = __fdiv_rn((float)code[e], fmaxf(ks[c8 + e], p.eps));
        }
      }
      store8(p.k_out, (row0 + t) * D + c8, x, p.out_dtype);
      const float4 a = *reinterpret_cast<const float4*>(vtile + t * D + c8);
      const float4 b4 = *reinterpret_cast<const float4*>(vtile + t * D + c8 + 4);
      const float y[8] = {a.x, a.y, a.z, a.w, b4.x, b4.y, b4.z, b4.w};
      store8(p.v_out, (row0 + t) * D + c8, y, p.out_dtype);
    }
    __syncthreads();  // the tables, the tile and this buffer are rewritten next
  }
}

}  // namespace

cudaError_t launch_restore(const RestoreParams& p, cudaStream_t s) {
  const int nm = p.bits == 2 ? 2 : p.bits == 4 ? 8 : 0;
  const size_t smem = 2 * (size_t)p.geom.page_bytes +
                      ((size_t)p.G * p.D + (size_t)nm * (p.D + p.G)) * sizeof(float);
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(restore_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  RestoreParams q = p;
  q.page_cols = (p.page_cols + kRestorePages - 1) / kRestorePages;  // page-run columns
  return launch_pdl(restore_kernel, dim3((q.page_cols + 1) * p.n_seqs * p.Hkv), dim3(kRestoreThreads), smem, s, q);
}

}  // namespace kvq
