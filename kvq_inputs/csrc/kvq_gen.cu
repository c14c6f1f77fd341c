// Device-side fill of the seeded synthetic inputs described in kvq_inputs/gen.py.
// Bit-identical to the numpy generator: integer hashing, table lookups and single
// fp32 multiplies (no contraction), then one round-to-nearest-even to bf16.
// Test and benchmark infrastructure only; not part of the cache library.

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;
constexpr uint64_t kMixA = 0xBF58476D1CE4E5B9ull;
constexpr uint64_t kMixB = 0x94D049BB133111EBull;
constexpr uint32_t kSpikeThreshold = 4294967u;

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * kMixA;
  z = (z ^ (z >> 27)) * kMixB;
  return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t hash_at(uint64_t key, uint64_t idx) {
  return mix64(key + (idx + 1ull) * kGamma);
}

__device__ __forceinline__ void store(void* out, size_t i, float x, int bf16) {
  if (bf16)
    reinterpret_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(x);
  else
    reinterpret_cast<float*>(out)[i] = x;
}

__global__ void gen_kv_kernel(const uint64_t* __restrict__ k_keys, const uint64_t* __restrict__ v_keys,
                              const uint64_t* __restrict__ tau_keys, const float* __restrict__ sigma,
                              const float* __restrict__ normal, const float* __restrict__ tau_table,
                              int n_units, int n_kv_heads, int D, long long t0, long long n_tokens,
                              int bf16, int spikes, void* out_k, void* out_v) {
  const size_t total = (size_t)n_units * (size_t)n_tokens * (size_t)D;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const int c = (int)(i % D);
    const size_t rest = i / D;
    const long long t = (long long)(rest % (size_t)n_tokens) + t0;
    const int unit = (int)(rest / (size_t)n_tokens);
    const int h = unit % n_kv_heads;
    const uint64_t idx = (uint64_t)t * (uint64_t)D + (uint64_t)c;

    const uint64_t hk = hash_at(k_keys[unit], idx);
    float k = __fmul_rn(normal[hk >> 48], sigma[h * D + c]);
    if (spikes && (uint32_t)(hk & 0xFFFFFFFFull) < kSpikeThreshold) k = __fmul_rn(k, 50.0f);
    store(out_k, i, k, bf16);

    const uint64_t hv = hash_at(v_keys[unit], idx);
    const float tau = tau_table[hash_at(tau_keys[unit], (uint64_t)t) >> 52];
    store(out_v, i, __fmul_rn(normal[hv >> 48], tau), bf16);
  }
}

__global__ void gen_q_kernel(const uint64_t* __restrict__ q_keys, const float* __restrict__ normal,
                             int n_rows, int D, long long step, int bf16, void* out) {
  const size_t total = (size_t)n_rows * D;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const int c = (int)(i % D);
    const int row = (int)(i / D);
    const uint64_t hq = hash_at(q_keys[row], (uint64_t)step * (uint64_t)D + (uint64_t)c);
    store(out, i, normal[hq >> 48], bf16);
  }
}

int grid_for(size_t total) {
  size_t blocks = (total + 255) / 256;
  if (blocks > 152 * 32) blocks = 152 * 32;
  return blocks ? (int)blocks : 1;
}

}  // namespace

extern "C" int kvq_gen_kv(const uint64_t* k_keys, const uint64_t* v_keys, const uint64_t* tau_keys,
                          const float* sigma, const float* normal_table, const float* tau_table,
                          int n_units, int n_kv_heads, int head_dim, long long t0, long long n_tokens,
                          int bf16, int spikes, void* out_k, void* out_v, void* stream) {
  if (n_units <= 0 || n_tokens <= 0 || head_dim <= 0 || n_kv_heads <= 0) return 1;
  const size_t total = (size_t)n_units * (size_t)n_tokens * (size_t)head_dim;
  gen_kv_kernel<<<grid_for(total), 256, 0, (cudaStream_t)stream>>>(
      k_keys, v_keys, tau_keys, sigma, normal_table, tau_table, n_units, n_kv_heads, head_dim, t0,
      n_tokens, bf16, spikes, out_k, out_v);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

extern "C" int kvq_gen_q(const uint64_t* q_keys, const float* normal_table, int n_rows, int head_dim,
                         long long step, int bf16, void* out, void* stream) {
  if (n_rows <= 0 || head_dim <= 0) return 1;
  const size_t total = (size_t)n_rows * head_dim;
  gen_q_kernel<<<grid_for(total), 256, 0, (cudaStream_t)stream>>>(q_keys, normal_table, n_rows,
                                                                  head_dim, step, bf16, out);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}
