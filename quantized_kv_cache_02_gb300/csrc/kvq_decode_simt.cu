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

// Merge of the split partials (o[D], m, l) of one (sequence, query head) by
// one warp each (merge_head), after a split launch that does not merge
// inside itself (DecodeParams::done null).  A sequence without tokens gets
// zeros.
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
  const int64_t unit = (int64_t)b * p.Hkv + h;
  const int64_t stride = (int64_t)p.g * part_row(p.D);
  const float* base = p.partials + unit * p.max_splits * stride + (int64_t)j * part_row(p.D);
  merge_head<VPL, false>(base, nsplit, nslots, p.max_splits, stride, p.D, p.out + ((int64_t)b * p.Hq + hq) * p.D,
                         lane);
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
