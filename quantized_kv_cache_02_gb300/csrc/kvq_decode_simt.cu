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
  if (cpl <= 1) decode_simt_kernel<T, BITS, 1><<<grid, kSimtThreads, 0, s>>>(p);
  else if (cpl <= 2) decode_simt_kernel<T, BITS, 2><<<grid, kSimtThreads, 0, s>>>(p);
  else if (cpl <= 4) decode_simt_kernel<T, BITS, 4><<<grid, kSimtThreads, 0, s>>>(p);
  else decode_simt_kernel<T, BITS, 8><<<grid, kSimtThreads, 0, s>>>(p);
  return cudaGetLastError();
}

constexpr int kCombineThreads = 128;

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const CombineParams p) {
  const int i = blockIdx.x / p.Hq;
  const int hq = blockIdx.x - i * p.Hq;
  const int b = p.seq_begin + i;
  const int h = hq / p.g, j = hq - h * p.g;
  const int T0 = p.ctr[i].total, Q0 = p.ctr[i].quantized;
  const int P = Q0 / p.G;
  const int nsplit = (P + p.chunk_pages - 1) / p.chunk_pages;
  const bool has_win = T0 > Q0;
  const int D = p.D;
  const int64_t unit = (int64_t)b * p.Hkv + h;
  const float* base = p.partials + unit * p.max_splits * (int64_t)p.g * (D + 2) + (int64_t)j * (D + 2);
  const int64_t stride = (int64_t)p.g * (D + 2);
  float* out = p.out + ((int64_t)b * p.Hq + hq) * D;

  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, base[s * stride + D]);
  if (has_win) M = fmaxf(M, base[(p.max_splits - 1) * stride + D]);
  float L = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < nsplit; ++s) {
      const float ms = base[s * stride + D];
      if (ms != -INFINITY) L = fmaf(base[s * stride + D + 1], exp2f(ms - M), L);
    }
    if (has_win) {
      const float ms = base[(p.max_splits - 1) * stride + D];
      if (ms != -INFINITY) L = fmaf(base[(p.max_splits - 1) * stride + D + 1], exp2f(ms - M), L);
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    float o = 0.f;
    if (M != -INFINITY) {
      for (int s = 0; s < nsplit; ++s) {
        const float ms = base[s * stride + D];
        if (ms != -INFINITY) o = fmaf(base[s * stride + c], exp2f(ms - M), o);
      }
      if (has_win) {
        const float ms = base[(p.max_splits - 1) * stride + D];
        if (ms != -INFINITY) o = fmaf(base[(p.max_splits - 1) * stride + c], exp2f(ms - M), o);
      }
    }
    out[c] = o * inv;
  }
}

}  // namespace

cudaError_t launch_decode_simt(const DecodeParams& p, int dtype, cudaStream_t s) {
  if (dtype == 0) return p.bits == 4 ? launch_bits<__nv_bfloat16, 4>(p, s) : launch_bits<__nv_bfloat16, 8>(p, s);
  return p.bits == 4 ? launch_bits<float, 4>(p, s) : launch_bits<float, 8>(p, s);
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t s) {
  combine_kernel<<<p.n_seqs * p.Hq, kCombineThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace kvq
