// CUDA-core split kernel and the combine kernel of the decode attention.
//
// Grid of the split kernel: x = split column (grid_splits quantized columns, then
// one residual-window column), y = (sequence, KV head) unit of this launch.
// The combine kernel merges a unit's partial softmax states, one CTA per
// (sequence, query head): M = max m_s, L = sum l_s 2^(m_s - M),
// o = sum o_s 2^(m_s - M) / L ("KV Cache 与自回归视频生成" section 05).

#include "kvq_simt.cuh"

namespace kvq {
namespace {

template <typename T, int BITS, int CPL, bool SEG>
__global__ void __launch_bounds__(kSimtThreads) decode_simt_kernel(const DecodeParams p) {
  pdl_wait();
  pdl_release();
  const int u = blockIdx.y;
  const int i = u / p.Hkv, h = u - i * p.Hkv;
  bool win;
  int pg0, pg1, slot;
  __shared__ float scratch[simt_scratch_floats<CPL>()];
  if (!split_item(p, blockIdx.x, i, &win, &pg0, &pg1, &slot)) return;
  simt_item<T, BITS, CPL, SEG>(p, i, h, win, pg0, pg1, slot, scratch);
}

template <typename T, int BITS, bool SEG>
cudaError_t launch_seg(const DecodeParams& p, cudaStream_t s) {
  const dim3 grid(p.grid_splits + 1, p.n_seqs * p.Hkv);
  const int cpl = (p.D + 31) / 32;
  const dim3 block(kSimtThreads);
  if (cpl <= 1) return launch_pdl(decode_simt_kernel<T, BITS, 1, SEG>, grid, block, 0, s, p);
  if (cpl <= 2) return launch_pdl(decode_simt_kernel<T, BITS, 2, SEG>, grid, block, 0, s, p);
  if (cpl <= 4) return launch_pdl(decode_simt_kernel<T, BITS, 4, SEG>, grid, block, 0, s, p);
  return launch_pdl(decode_simt_kernel<T, BITS, 8, SEG>, grid, block, 0, s, p);
}

template <typename T, int BITS>
cudaError_t launch_bits(const DecodeParams& p, cudaStream_t s) {
  return p.seg.kcodes ? launch_seg<T, BITS, true>(p, s) : launch_seg<T, BITS, false>(p, s);
}

constexpr int kCombineWarps = 4;
constexpr int kCombineChunk = 8;  // slots whose loads are in flight together

// Merge of the split partials (o[D], m, l) of one (sequence, query head):
// M = max m_s, L = sum l_s 2^(m_s - M), o = sum o_s 2^(m_s - M) / L
// ("KV Cache 与自回归视频生成" section 05, FlashDecoding).  One warp per
// (sequence, query head).  The slots are taken eight at a time: lane s reads
// slot s's (m, l) while every lane reads its 16-byte pieces of the eight o
// rows, so one round trip serves the whole chunk; the chunk is then folded
// into the running (M, L, o) with the usual rescale.  VPL = 16-byte pieces of
// o per lane (1 for head_dim <= 128, 2 up to 256).  A sequence without tokens
// gets zeros.
template <int VPL>
__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(const CombineParams p) {
  pdl_wait();
  pdl_release();
  const int lane = threadIdx.x & 31;
  const int item = blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
  if (item >= p.n_seqs * p.Hq) return;
  const int i = item / p.Hq;
  const int hq = item - i * p.Hq;
  const int b = p.seq_begin + i;
  const int h = hq / p.g, j = hq - h * p.g;
  const int T0 = p.ctr[i].total, Q0 = p.ctr[i].quantized;
  int nsplit = p.dense_chunk > 0 ? (T0 + p.dense_chunk - 1) / p.dense_chunk
                                 : (Q0 / p.G + p.chunk_pages - 1) / p.chunk_pages;
  int nslots = nsplit + (p.dense_chunk == 0 && T0 > Q0 ? 1 : 0);
  if (p.line_warps > 0) {
    // slots of the warps from the one holding the unit's first line position
    // to the one holding its last
    const int64_t C = p.line_start[p.n_seqs];
    const int64_t cost = Q0 / 32 + 2 * ((T0 - Q0 + 15) / 16);
    const int64_t s0 = p.line_start[i] + (int64_t)h * cost;
    const int N = p.line_warps;
    nslots = cost > 0 ? (int)(((s0 + cost) * N - 1) / C - ((s0 + 1) * N - 1) / C) + 1 : 0;
    nsplit = nslots;
  }
  const int D = p.D, nvec = D >> 2;
  const int64_t unit = (int64_t)b * p.Hkv + h;
  const int64_t stride = (int64_t)p.g * part_row(D);
  const float* base = p.partials + unit * p.max_splits * stride + (int64_t)j * part_row(D);
  // slot k < nsplit is split column k; the window's partial sits in the last column
  auto row = [&](int k) { return base + (k < nsplit ? k : p.max_splits - 1) * stride; };

  float M = -INFINITY, L = 0.f;
  float4 o[VPL];
#pragma unroll
  for (int e = 0; e < VPL; ++e) o[e] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k0 = 0; k0 < nslots; k0 += kCombineChunk) {
    const int n = min(kCombineChunk, nslots - k0);
    float2 ml = make_float2(-INFINITY, 0.f);
    if (lane < n) ml = __ldg(reinterpret_cast<const float2*>(row(k0 + lane) + D));
    float4 v[kCombineChunk][VPL];
#pragma unroll
    for (int s = 0; s < kCombineChunk; ++s)
#pragma unroll
      for (int e = 0; e < VPL; ++e) {
        const int c4 = lane + 32 * e;
        v[s][e] = (s < n && c4 < nvec) ? __ldg(reinterpret_cast<const float4*>(row(k0 + s)) + c4)
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    float cm = ml.x;
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, off));
    cm = __shfl_sync(0xffffffffu, cm, 0);
    const float Mn = fmaxf(M, cm);
    const float Ms = Mn == -INFINITY ? 0.f : Mn;
    const float corr = exp2f(M - Ms);
    const float f = exp2f(ml.x - Ms);  // lanes >= n: 0
    float ls = ml.y * f;
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, off);
    L = fmaf(L, corr, __shfl_sync(0xffffffffu, ls, 0));
#pragma unroll
    for (int e = 0; e < VPL; ++e) {
      o[e].x *= corr;
      o[e].y *= corr;
      o[e].z *= corr;
      o[e].w *= corr;
    }
#pragma unroll
    for (int s = 0; s < kCombineChunk; ++s) {
      const float fs = __shfl_sync(0xffffffffu, f, s);
#pragma unroll
      for (int e = 0; e < VPL; ++e) {
        o[e].x = fmaf(v[s][e].x, fs, o[e].x);
        o[e].y = fmaf(v[s][e].y, fs, o[e].y);
        o[e].z = fmaf(v[s][e].z, fs, o[e].z);
        o[e].w = fmaf(v[s][e].w, fs, o[e].w);
      }
    }
    M = Mn;
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  // the entry points accept only 16-byte aligned outputs
  float4* out = reinterpret_cast<float4*>(p.out + ((int64_t)b * p.Hq + hq) * D);
#pragma unroll
  for (int e = 0; e < VPL; ++e) {
    const int c4 = lane + 32 * e;
    if (c4 < nvec) out[c4] = make_float4(o[e].x * inv, o[e].y * inv, o[e].z * inv, o[e].w * inv);
  }
}

}  // namespace

cudaError_t launch_decode_simt(const DecodeParams& p, int dtype, cudaStream_t s) {
  if (dtype == 0) {
    if (p.bits == 2) return launch_bits<__nv_bfloat16, 2>(p, s);
    return p.bits == 4 ? launch_bits<__nv_bfloat16, 4>(p, s) : launch_bits<__nv_bfloat16, 8>(p, s);
  }
  if (p.bits == 2) return launch_bits<float, 2>(p, s);
  return p.bits == 4 ? launch_bits<float, 4>(p, s) : launch_bits<float, 8>(p, s);
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t s) {
  const dim3 grid((p.n_seqs * p.Hq + kCombineWarps - 1) / kCombineWarps);
  return p.D <= 128 ? launch_pdl(combine_kernel<1>, grid, dim3(kCombineWarps * 32), 0, s, p)
                    : launch_pdl(combine_kernel<2>, grid, dim3(kCombineWarps * 32), 0, s, p);
}

}  // namespace kvq
