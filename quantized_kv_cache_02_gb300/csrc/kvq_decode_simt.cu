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

template <typename T, int BITS, int CPL>
__global__ void __launch_bounds__(kSimtThreads) decode_simt_kernel(const DecodeParams p) {
  pdl_wait();
  pdl_release();
  const int u = blockIdx.y;
  const int i = u / p.Hkv, h = u - i * p.Hkv;
  bool win;
  int pg0, pg1, slot;
  __shared__ float scratch[simt_scratch_floats<CPL>()];
  if (!split_item(p, blockIdx.x, i, &win, &pg0, &pg1, &slot)) return;
  simt_item<T, BITS, CPL>(p, i, h, win, pg0, pg1, slot, scratch);
}

template <typename T, int BITS>
cudaError_t launch_bits(const DecodeParams& p, cudaStream_t s) {
  const dim3 grid(p.grid_splits + 1, p.n_seqs * p.Hkv);
  const int cpl = (p.D + 31) / 32;
  const dim3 block(kSimtThreads);
  if (cpl <= 1) return launch_pdl(decode_simt_kernel<T, BITS, 1>, grid, block, 0, s, p);
  if (cpl <= 2) return launch_pdl(decode_simt_kernel<T, BITS, 2>, grid, block, 0, s, p);
  if (cpl <= 4) return launch_pdl(decode_simt_kernel<T, BITS, 4>, grid, block, 0, s, p);
  return launch_pdl(decode_simt_kernel<T, BITS, 8>, grid, block, 0, s, p);
}

constexpr int kCombineThreads = 128;

// Merge of the split partials (o[D], m, l) of one (sequence, query head):
// M = max m_s, L = sum l_s 2^(m_s - M), o = sum o_s 2^(m_s - M) / L
// ("KV Cache 与自回归视频生成" section 05, FlashDecoding).  One CTA per
// (sequence, query head), one thread per channel; the slot loops are unrolled
// so their loads overlap.  A sequence without tokens gets zeros.
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const CombineParams p) {
  pdl_wait();
  pdl_release();
  const int i = blockIdx.x / p.Hq;
  const int hq = blockIdx.x - i * p.Hq;
  const int b = p.seq_begin + i;
  const int h = hq / p.g, j = hq - h * p.g;
  const int T0 = p.ctr[i].total, Q0 = p.ctr[i].quantized;
  const int nsplit = p.dense_chunk > 0 ? (T0 + p.dense_chunk - 1) / p.dense_chunk
                                      : (Q0 / p.G + p.chunk_pages - 1) / p.chunk_pages;
  const int nslots = nsplit + (p.dense_chunk == 0 && T0 > Q0 ? 1 : 0);
  const int D = p.D;
  const int64_t unit = (int64_t)b * p.Hkv + h;
  const float* base = p.partials + unit * p.max_splits * (int64_t)p.g * (D + 2) + (int64_t)j * (D + 2);
  const int64_t stride = (int64_t)p.g * (D + 2);
  auto row = [&](int k) { return base + (k < nsplit ? k : p.max_splits - 1) * stride; };
  float M = -INFINITY;
#pragma unroll 4
  for (int k = 0; k < nslots; ++k) M = fmaxf(M, row(k)[D]);
  const float Ms = M == -INFINITY ? 0.f : M;
  float L = 0.f;
  float o[2] = {0.f, 0.f};
#pragma unroll 4
  for (int k = 0; k < nslots; ++k) {
    const float* r = row(k);
    const float f = exp2f(r[D] - Ms);
    L = fmaf(r[D + 1], f, L);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int c = threadIdx.x + e * kCombineThreads;
      if (c < D) o[e] = fmaf(r[c], f, o[e]);
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  float* out = p.out + ((int64_t)b * p.Hq + hq) * D;
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int c = threadIdx.x + e * kCombineThreads;
    if (c < D) out[c] = o[e] * inv;
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
  return launch_pdl(combine_kernel, dim3(p.n_seqs * p.Hq), dim3(kCombineThreads), 0, s, p);
}

}  // namespace kvq
