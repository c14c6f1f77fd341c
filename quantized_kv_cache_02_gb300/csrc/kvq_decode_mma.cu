// Tensor-core decode: the host-facing launchers.  The kernels live in
// kvq_decode_mma.cuh; the split kernel's instantiations are compiled one code
// width per translation unit (kvq_decode_mma_b2.cu, _b4.cu, _b8.cu) so that
// they build in parallel.

#include "kvq_decode_mma.cuh"

namespace kvq {

size_t decode_mma_smem_bytes(const DecodeParams& p) {
  return p.D == 64 ? smem_for<64>(p) : smem_for<128>(p);
}

cudaError_t launch_decode_dense(const DecodeParams& p, cudaStream_t s, int* supported) {
  *supported = (p.D == 64 || p.D == 128) && p.g <= kMaxGqa && p.dense_chunk > 0;
  if (!*supported) return cudaSuccess;
  int64_t tmax = 0;
  for (int i = 0; i < p.n_seqs; ++i) tmax = p.ctr[i].total > tmax ? p.ctr[i].total : tmax;
  const int cols = (int)((tmax + p.dense_chunk - 1) / p.dense_chunk);
  if (cols == 0) return cudaSuccess;
  return p.D == 64 ? launch_dense_g<64>(p, cols, s) : launch_dense_g<128>(p, cols, s);
}

bool decode_mma_supported(const DecodeParams& p) {
  // a segmented cache: 4-bit codes, split items of whole 32-token tiles
  const bool tiles = p.seg.kcodes ? p.bits == 4 && p.chunk_pages % 32 == 0 : p.G % 32 == 0;
  return (p.D == 64 || p.D == 128) && tiles && p.g >= 2 && p.g <= kMaxGqa && decode_mma_smem_bytes(p) <= kMaxSmem;
}

int decode_mma_resident_per_sm(const DecodeParams& p) {
  if (!decode_mma_supported(p)) return 0;
  return p.bits == 2 ? resident_mma_bits2(p) : p.bits == 4 ? resident_mma_bits4(p) : resident_mma_bits8(p);
}

cudaError_t decode_line(const DecodeParams& p, bool launch, cudaStream_t s, int* per_sm) {
  if (!decode_mma_supported(p) || p.seg.kcodes || p.step_k) {
    *per_sm = 0;
    return cudaSuccess;
  }
  return p.bits == 2 ? line_bits2(p, launch, s, per_sm)
         : p.bits == 4 ? line_bits4(p, launch, s, per_sm)
                       : line_bits8(p, launch, s, per_sm);
}

cudaError_t launch_decode_mma(const DecodeParams& p, cudaStream_t s, int* supported) {
  *supported = decode_mma_supported(p);
  if (!*supported) return cudaSuccess;
  return p.bits == 2 ? launch_mma_bits2(p, s) : p.bits == 4 ? launch_mma_bits4(p, s) : launch_mma_bits8(p, s);
}

}  // namespace kvq
