// Instantiations of the tensor-core split kernel for 8-bit codes (head_dim
// 64 and 128, every GQA padding and page mode); see kvq_decode_mma.cuh.

#include "kvq_decode_line.cuh"

namespace kvq {

int resident_mma_bits8(const DecodeParams& p) {
  return p.D == 64 ? resident_g<64, 8>(p) : resident_g<128, 8>(p);
}

cudaError_t launch_mma_bits8(const DecodeParams& p, cudaStream_t s) {
  return p.D == 64 ? launch_g<64, 8>(p, s) : launch_g<128, 8>(p, s);
}

cudaError_t line_bits8(const DecodeParams& p, bool launch, cudaStream_t s, int* per_sm) {
  return p.D == 64 ? line_g<64, 8>(p, launch, s, per_sm) : line_g<128, 8>(p, launch, s, per_sm);
}

}  // namespace kvq
