// Tensor-core split kernel of the decode attention over the quantized prefix.
//
// Work item: a run of group pages of one (sequence, KV head) unit; the CTA's
// warps take pages round robin, each warp streaming its pages through its own
// ring of shared-memory slots with cp.async.bulk (the TMA engine) and one
// mbarrier per slot, so no warp ever waits on another.  All waits are bounded:
// a wait that gives up sets the device status word and the warp stops.
//
// Per 32-token sub-tile the warp computes, for the g <= 8 query heads of the
// KV head (GQA: they share every K/V tile):
//   S[t][h] = sum_c code_K[t][c] * (q[h][c] / sK[c]) * log2(e)/sqrt(d)
//   online softmax in base 2 (running max m, sum l)
//   O^T[c][h] += sum_t code_V[t][c] * (p[h][t] / sV[t])
// which is q.k/sqrt(d) and p.v over restored values k = code/sK, v = code/sV
// ("KV Cache Quantization Strategies", restore; "KV Cache 与自回归视频生成"
// 3.1 and attn_step) with both scales folded into the f16 MMA operand that
// is not the code (q/sK as an f16 hi + lo pair, p/sV as one f16).  Codes
// enter the MMA as f16 subnormals cut straight out of the stored word (see
// "codes as f16 subnormals" below); the bias and the 2^-24 are undone once per
// page for S and once per run for O.
// Matrix shapes: S = A(K codes: 16 tokens x 16 channels) * B(q: 16 x 8 heads),
// O^T = A(V codes^T: 16 channels x 16 tokens) * B(P^T: 16 tokens x 8 heads);
// P goes from the S accumulator layout to the B layout with movmatrix.trans.
// Token and channel orders inside a k-step are permuted to match the packed
// byte layout; both operands of every MMA use the same permutation.

#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>
#include <type_traits>

#include "kvq_simt.cuh"

namespace kvq {
namespace {

constexpr int kMmaWarps = 4;
constexpr int kMmaThreads = kMmaWarps * 32;
constexpr uint32_t kSpinLimit = 1u << 24;

// ---- PTX helpers -----------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// Fire-and-forget copy of [src, src + bytes) from HBM into L2 (16-byte
// aligned address and size).
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Bounded wait on phase ``parity`` of an mbarrier; false if it gave up.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (uint32_t it = 0; it < kSpinLimit; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t transpose8x8(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- codes as f16 subnormals --------------------------------------------
// A stored code is offset binary: u = code + bias (bias 8 for 4-bit, 128 for
// 8-bit), u in [1, 2*bias).  A 16-bit half whose bits are just u (exponent 0)
// is the binary16 subnormal u * 2^-24, exactly; u << 4 is 16 * u * 2^-24.  So
// masking the stored word yields MMA operands without any floating-point
// conversion; the 2^-24, the x16 of the second nibble position (cancelled by a
// 1/16 on the matching B rows) and the bias are undone after the MMA:
// S = 2^24 * S' - bias * sum(B),  O = 2^24 * O' - bias * sum(p').

// 4-bit: word of eight nibbles -> r[j] = (nibble j, nibble j + 4) as f16x2;
// r[1] and r[3] carry an extra factor 16.
__device__ __forceinline__ void nibble_regs(uint32_t w, uint32_t (&r)[4]) {
  const uint32_t w2 = w >> 8;
  r[0] = w & 0x000F000Fu;
  r[1] = w & 0x00F000F0u;
  r[2] = w2 & 0x000F000Fu;
  r[3] = w2 & 0x00F000F0u;
}

// 2-bit: word of sixteen 2-bit fields (four per byte) -> r[j] = (field j of
// byte 0, field j of byte 2), r[4 + j] = (field j of byte 1, of byte 3), each
// carrying a factor 4^j.
__device__ __forceinline__ void crumb_regs(uint32_t w, uint32_t (&r)[8]) {
  const uint32_t w2 = w >> 8;
  r[0] = w & 0x00030003u;
  r[1] = w & 0x000C000Cu;
  r[2] = w & 0x00300030u;
  r[3] = w & 0x00C000C0u;
  r[4] = w2 & 0x00030003u;
  r[5] = w2 & 0x000C000Cu;
  r[6] = w2 & 0x00300030u;
  r[7] = w2 & 0x00C000C0u;
}

// 2-bit registers hold u * 4^j * 2^-24 with u = code + 2; subtracting
// 2 * 4^j * 2^-24 (f16 subnormal arithmetic on small integers is exact) leaves
// code * 4^j * 2^-24.  With codes of -1..1 and per-group absmax scales, a
// channel holding one huge outlier adds 2 * q / sK to every token's biased
// score, and the fp32 accumulation of that term would cost more precision
// than the subtraction here.
__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ void unbias_crumbs(uint32_t (&r)[8]) {
#pragma unroll
  for (int m = 0; m < 8; ++m) r[m] = hsub2(r[m], 0x00020002u << (2 * (m & 3)));
}

// 2-bit Value piece (16 bits: even tokens of an 8-token span in the low byte,
// odd tokens in the high byte) -> r[j] = (token 2j, token 2j + 1), factor 4^j.
__device__ __forceinline__ void piece_regs(uint32_t piece, uint32_t (&r)[4]) {
  const uint32_t x = __byte_perm(piece, 0u, 0x4140);  // bytes (b0, 0, b1, 0)
  r[0] = x & 0x00030003u;
  r[1] = x & 0x000C000Cu;
  r[2] = x & 0x00300030u;
  r[3] = x & 0x00C000C0u;
#pragma unroll
  for (int j = 0; j < 4; ++j) r[j] = hsub2(r[j], 0x00020002u << (2 * j));
}

// The same for 4-bit registers (u = code + 8; registers 1 and 3 carry x16)
// and 8-bit ones (u = code + 128): afterwards they hold code * 2^-24 (x16).
__device__ __forceinline__ void unbias_nibbles(uint32_t (&r)[4]) {
  r[0] = hsub2(r[0], 0x00080008u);
  r[1] = hsub2(r[1], 0x00800080u);
  r[2] = hsub2(r[2], 0x00080008u);
  r[3] = hsub2(r[3], 0x00800080u);
}

// 8-bit: word of four bytes -> r[0] = (byte 0, byte 2), r[1] = (byte 1, byte 3).
__device__ __forceinline__ void byte_regs(uint32_t w, uint32_t (&r)[2]) {
  r[0] = w & 0x00FF00FFu;
  r[1] = (w >> 8) & 0x00FF00FFu;
}

// f16 hi of (x0, x1), and the f16 of hi - x = -(lo) from the mixed-precision
// add (f16 + f32 -> f32, exact here: hi and x agree to within an f16 ulp), so
// that hi + lo carries x to about 22 bits.
__device__ __forceinline__ void split_hi_neglo(float x0, float x1, uint32_t& hi, uint32_t& nlo) {
  const __half2 h = __floats2half2_rn(x0, x1);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  float d0, d1;
  asm("{\n .reg .b16 a, b;\n mov.b32 {a, b}, %2;\n add.rn.f32.f16 %0, a, %3;\n add.rn.f32.f16 %1, b, %4;\n}\n"
      : "=f"(d0), "=f"(d1)
      : "r"(hi), "f"(-x0), "f"(-x1));
  const __half2 l = __floats2half2_rn(d0, d1);
  nlo = *reinterpret_cast<const uint32_t*>(&l);
}

__device__ __forceinline__ float fast_rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void mma16816_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// 16-byte global -> shared copy; src_bytes = 0 fills the 16 bytes with zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

template <int N>
__device__ __forceinline__ void lds_words(const uint8_t* p, uint32_t (&w)[N]) {
  static_assert(N == 1 || N % 2 == 0, "word count");
  if constexpr (N == 1) {
    w[0] = *reinterpret_cast<const uint32_t*>(p);
  } else if constexpr (N % 4 == 0) {
#pragma unroll
    for (int i = 0; i < N / 4; ++i) {
      const uint4 v = reinterpret_cast<const uint4*>(p)[i];
      w[4 * i] = v.x;
      w[4 * i + 1] = v.y;
      w[4 * i + 2] = v.z;
      w[4 * i + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
      const uint2 v = reinterpret_cast<const uint2*>(p)[i];
      w[2 * i] = v.x;
      w[2 * i + 1] = v.y;
    }
  }
}

// ---- range of the f16 operands ------------------------------------------
// The pages hold any finite scale, so q / sK and p / sV can leave the f16
// range (65504), the fp32 bias sums of large q / sK lose the scores'
// precision, one f16 p / sV (11 bits) keeps the output error near 2^-12 of
// the p-weighted |v| only while |v| is small, and a scale can drop below eps,
// where the page's restore divides by eps.  A tensor-core item therefore
// runs only when the unit's flushed maxima bound every group: all Key scales
// at least kthr (|q / sK| <= 2^9, 2^14 at 2 bits where the codes enter
// signed and only the f16 range limits) and every Value absmax at most
// kVWideAbs.  Other items take the CUDA-core path (fp32, IEEE division with
// the eps clamp) inside the same kernel.
constexpr float kVWideAbs = 16.f;
// split items of at most this many pages prefetch their first pages to L2
constexpr int kShortItemPages = 16;
constexpr int kMaxRangeShift = 100;

// Binary exponent of a positive finite float (floor(log2 x)); 0 gives -127.
__device__ __forceinline__ int float_exp2i(float x) { return (int)((__float_as_uint(x) >> 23) & 0xFFu) - 127; }
// 2^-e for 0 <= e <= 126, exactly.
__device__ __forceinline__ float pow2_neg(int e) { return __uint_as_float((uint32_t)(127 - e) << 23); }
// 2^e for -126 <= e <= 127 (0 below, infinity above).
__device__ __forceinline__ float pow2i(int e) {
  return e < -126 ? 0.f : e > 127 ? INFINITY : __uint_as_float((uint32_t)(e + 127) << 23);
}

// GP = query heads per KV head rounded up to 2, 4 or 8.  The MMA's 8 columns
// hold GP heads of each of PB = 8 / GP pages, so one B operand (q / sK) and one
// softmax update serve PB pages ("streams"); column n belongs to stream n / GP.
template <int D, int BITS, int GP>
struct Shape {
  static constexpr int PB = 8 / GP;
  static constexpr int kSteps = D / 16;          // k-steps of the S MMA, m-tiles of the O MMA
  static constexpr int kRowBytes = D * BITS / 8;
  static constexpr int kWords = kRowBytes / 16;  // 32-bit words of a K row per thread
  static constexpr int kChan = D / 4;            // channels of a K row per thread
  static constexpr int kSubBytes = 32 * D * BITS / 8;
  static constexpr int kChunks = D / 4;          // float4 chunks of a page's Key scales
  static constexpr float kBias = BITS == 2 ? 2.f : BITS == 4 ? 8.f : 128.f;
  // 2-bit: the B operand carries 16 * 4^-j for a code in field j, so that no
  // q / sK term drops into the f16 subnormals; S is divided by it afterwards
  static constexpr float kBScale = BITS == 2 ? 16.f : 1.f;
};

// Channel (in the thread's slice) of element e of k-step kk's B operand:
// e = 0, 1 -> register 0 (k-slots 2tig, 2tig+1); e = 2, 3 -> register 1.
// 2-bit: k-step kk = 4i + s takes registers R[2s] (a0) and R[2s + 1] (a2) of
// word i, R as crumb_regs returns them.
template <int BITS>
__device__ __forceinline__ constexpr int kslot_channel(int kk, int e) {
  if (BITS == 2) {
    const int m = 2 * (kk & 3) + (e >> 1);
    return 16 * (kk >> 2) + 4 * (m >> 2) + (m & 3) + 8 * (e & 1);
  }
  return BITS == 4 ? 8 * (kk >> 1) + 2 * (kk & 1) + (e == 0 ? 0 : e == 1 ? 4 : e == 2 ? 1 : 5)
                   : 4 * kk + (e == 0 ? 0 : e == 1 ? 2 : e == 2 ? 1 : 3);
}

// Token row (inside a 32-token sub-tile) of S rows gid (r0) and gid + 8 (r1)
// of m-block mb; these orders match how the conversions pair tokens.
template <int BITS>
__device__ __forceinline__ int token_row0(int gid, int mb) {
  return BITS <= 4 ? 8 * (gid >> 1) + 4 * mb + (gid & 1) : 8 * (gid >> 1) + 4 * mb + 2 * (gid & 1);
}
template <int BITS>
__device__ __forceinline__ constexpr int token_row_gap() {
  return BITS <= 4 ? 2 : 1;
}

template <int D>
struct WarpState {
  float O[D / 16][4];  // O'^T accumulators (biased codes, scaled by 2^-24)
  float C[4];          // 2^-24 * sum of the p / sV each column fed to O' (for the bias)
  float m0, m1;        // running max of the thread's two columns (base 2)
  float l0, l1;        // running sum of p (partial over this thread's rows)
};

// A group of PB pages (FULL) or of npages < PB pages (the tail of a warp's
// run), already in shared memory.  TOKV (4-bit only): the pages are 32-token
// tiles of a segmented cache, whose Value codes are token-major rows like the
// Key rows.  Their Value A operand pairs two tokens of one channel from two
// rows with a byte permute; lane (gid, tig) takes the channels
// [gid D/8, (gid + 1) D/8) (O'^T row gid of m-tile mt is channel
// gid D/8 + 2 mt, row gid + 8 the next one, whose odd nibble comes x16) and
// the tokens 8 tig .. 8 tig + 7 that its P columns hold.
template <int D, int BITS, int GP, bool FULL, bool TOKV = false>
__device__ __forceinline__ void mma_group(const uint8_t* const (&pg)[Shape<D, BITS, GP>::PB], int npages_rt,
                                          const PageGeom& geom, int G, const float4* q4, float* rsc, int lane,
                                          int gid, int tig, WarpState<D>& st) {
  using S = Shape<D, BITS, GP>;
  constexpr float kTwo24 = 16777216.f;
  const int npages = FULL ? S::PB : npages_rt;
  // ---- reciprocal Key scales, cooperatively, in a bank-friendly order -------
  // chunk i (channels tig*kChan + 4i .. +3) of slice tig goes to float4 slot
  // i*4 + tig.  For 4-bit codes the odd channels meet the x16 registers, so
  // their reciprocals carry the compensating 1/16.
  static_assert((S::PB * S::kChunks) % 32 == 0 || S::PB * S::kChunks < 32, "chunk split");
#pragma unroll
  for (int it = 0; it < (S::PB * S::kChunks + 31) / 32; ++it) {
    const int q = lane + 32 * it;
    const int j = q / S::kChunks, cc = q - j * S::kChunks;
    if (q < S::PB * S::kChunks && j < npages) {
      const float4 s4 = reinterpret_cast<const float4*>(pg[j] + geom.kscale_off)[cc];
      // the factor that undoes each channel's position in its code word
      constexpr float f0 = BITS == 2 ? 16.f : 1.f, f1 = BITS == 2 ? 4.f : BITS == 4 ? 0.0625f : 1.f;
      constexpr float f2 = 1.f, f3 = BITS == 2 ? 0.25f : BITS == 4 ? 0.0625f : 1.f;
      const float4 r4 = make_float4(fast_rcp(s4.x) * f0, fast_rcp(s4.y) * f1, fast_rcp(s4.z) * f2,
                                    fast_rcp(s4.w) * f3);
      const int tg = cc / (S::kChan / 4), i = cc - tg * (S::kChan / 4);
      reinterpret_cast<float4*>(rsc + j * D)[i * 4 + tg] = r4;
    }
  }
  __syncwarp();
  // ---- B operand of S: q / sK for (head gid % GP, page gid / GP), hi + lo ---
  uint32_t bh[S::kSteps][2], bl[S::kSteps][2];
  float beta0, beta1;
  {
    const int jb = FULL ? gid / GP : min(gid / GP, npages - 1);
    const float4* rj = reinterpret_cast<const float4*>(rsc + jb * D);
    float qk[S::kChan];
    float bs[4] = {0.f, 0.f, 0.f, 0.f};  // sums over channels 4i + k
    const int hq = gid % GP;
#pragma unroll
    for (int i = 0; i < S::kChan / 4; ++i) {
      const float4 r = rj[i * 4 + tig];
      const float4 qv = q4[(i * GP + hq) * 4 + tig];
      qk[4 * i + 0] = qv.x * r.x;
      qk[4 * i + 1] = qv.y * r.y;
      qk[4 * i + 2] = qv.z * r.z;
      qk[4 * i + 3] = qv.w * r.w;
      bs[0] += qk[4 * i + 0];
      bs[1] += qk[4 * i + 1];
      bs[2] += qk[4 * i + 2];
      bs[3] += qk[4 * i + 3];
    }
    // sum of q / sK with the position factors taken back out
    if constexpr (BITS == 2) {
      // 2-bit codes enter the MMA already signed: no bias to take out
      beta0 = beta1 = 0.f;
    } else {
      float beta = BITS == 4 ? (bs[0] + bs[2]) + 16.f * (bs[1] + bs[3]) : (bs[0] + bs[2]) + (bs[1] + bs[3]);
      beta += __shfl_xor_sync(0xffffffffu, beta, 1);
      beta += __shfl_xor_sync(0xffffffffu, beta, 2);
      beta0 = S::kBias * __shfl_sync(0xffffffffu, beta, 4 * (2 * tig));
      beta1 = S::kBias * __shfl_sync(0xffffffffu, beta, 4 * (2 * tig + 1));
    }
#pragma unroll
    for (int kk = 0; kk < S::kSteps; ++kk) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float x0 = qk[kslot_channel<BITS>(kk, 2 * r)], x1 = qk[kslot_channel<BITS>(kk, 2 * r + 1)];
        // bl holds the lo parts negated (hi - x, exact in fp32), taken off the
        // hi products where the scores are summed; 8-bit codes share one
        // accumulator for both, so their lo parts get the sign back here
        split_hi_neglo(x0, x1, bh[kk][r], bl[kk][r]);
        if (BITS == 8) bl[kk][r] ^= 0x80008000u;
      }
    }
  }
  const int sj = (2 * tig) / GP;                  // this thread's stream (both columns)
  const int vpage = FULL ? sj : min(sj, npages - 1);  // a valid page for its Value scales
  const uint8_t* vpg = pg[0];
#pragma unroll
  for (int j = 1; j < S::PB; ++j)
    if (j == vpage) vpg = pg[j];
  constexpr int kGap = token_row_gap<BITS>();
  // A operand of the p/sV counter: the value 1 (or 16 on the x16 k-slots) in
  // every element, as 2^-24-scaled subnormals like the codes
  constexpr uint32_t kOneLo = 0x00010001u;
  constexpr uint32_t kOneHi = BITS == 4 && !TOKV ? 0x00100010u : 0x00010001u;
  static_assert(!TOKV || BITS == 4, "token-major Value codes: 4-bit only");

  for (int sub = 0; sub < G / 32; ++sub) {
    // ---- scores of every page; keep each column's own page ------------------
    float ss[2][4];
#pragma unroll
    for (int mb = 0; mb < 2; ++mb) ss[mb][0] = ss[mb][1] = ss[mb][2] = ss[mb][3] = -INFINITY;
#pragma unroll
    for (int j = 0; j < S::PB; ++j) {
      if (!FULL && j >= npages) break;
      const uint8_t* kc = pg[j] + sub * 32 * S::kRowBytes;
      uint32_t wa[2][S::kWords], wb[2][S::kWords];
      // hi and (negated) lo halves of q accumulate separately: two dependent
      // MMA chains of half the length, combined once per sub-tile
      float s[2][4], s2[2][4];
#pragma unroll
      for (int mb = 0; mb < 2; ++mb) {
        const int r0 = token_row0<BITS>(gid, mb);
        lds_words<S::kWords>(kc + r0 * S::kRowBytes + tig * (S::kRowBytes / 4), wa[mb]);
        lds_words<S::kWords>(kc + (r0 + kGap) * S::kRowBytes + tig * (S::kRowBytes / 4), wb[mb]);
        s[mb][0] = s[mb][1] = s[mb][2] = s[mb][3] = 0.f;
        s2[mb][0] = s2[mb][1] = s2[mb][2] = s2[mb][3] = 0.f;
      }
      if (BITS == 2) {
#pragma unroll
        for (int i = 0; i < S::kWords; ++i) {
#pragma unroll
          for (int mb = 0; mb < 2; ++mb) {
            uint32_t ra[8], rb[8];
            crumb_regs(wa[mb][i], ra);
            crumb_regs(wb[mb][i], rb);
            unbias_crumbs(ra);
            unbias_crumbs(rb);
#pragma unroll
            for (int st2 = 0; st2 < 4; ++st2) {
              const int kk = 4 * i + st2;
              mma16816(s[mb], ra[2 * st2], rb[2 * st2], ra[2 * st2 + 1], rb[2 * st2 + 1], bh[kk][0], bh[kk][1]);
              mma16816(s2[mb], ra[2 * st2], rb[2 * st2], ra[2 * st2 + 1], rb[2 * st2 + 1], bl[kk][0], bl[kk][1]);
            }
          }
        }
#pragma unroll
        for (int mb = 0; mb < 2; ++mb)
#pragma unroll
          for (int e = 0; e < 4; ++e) s[mb][e] -= s2[mb][e];
      } else if (BITS == 4) {
#pragma unroll
        for (int i = 0; i < S::kWords; ++i) {
#pragma unroll
          for (int mb = 0; mb < 2; ++mb) {
            uint32_t ra[4], rb[4];
            nibble_regs(wa[mb][i], ra);
            nibble_regs(wb[mb][i], rb);
            mma16816(s[mb], ra[0], rb[0], ra[1], rb[1], bh[2 * i][0], bh[2 * i][1]);
            mma16816(s2[mb], ra[0], rb[0], ra[1], rb[1], bl[2 * i][0], bl[2 * i][1]);
            mma16816(s[mb], ra[2], rb[2], ra[3], rb[3], bh[2 * i + 1][0], bh[2 * i + 1][1]);
            mma16816(s2[mb], ra[2], rb[2], ra[3], rb[3], bl[2 * i + 1][0], bl[2 * i + 1][1]);
          }
        }
#pragma unroll
        for (int mb = 0; mb < 2; ++mb)
#pragma unroll
          for (int e = 0; e < 4; ++e) s[mb][e] -= s2[mb][e];
      } else {
#pragma unroll
        for (int kk = 0; kk < S::kWords; ++kk) {
#pragma unroll
          for (int mb = 0; mb < 2; ++mb) {
            uint32_t ra[2], rb[2];
            byte_regs(wa[mb][kk], ra);
            byte_regs(wb[mb][kk], rb);
            mma16816(s[mb], ra[0], rb[0], ra[1], rb[1], bh[kk][0], bh[kk][1]);
            mma16816(s[mb], ra[0], rb[0], ra[1], rb[1], bl[kk][0], bl[kk][1]);
          }
        }
      }
      const bool mine = sj == j;
#pragma unroll
      for (int mb = 0; mb < 2; ++mb) {
        constexpr float kUnscale = kTwo24 / S::kBScale;
        ss[mb][0] = mine ? fmaf(s[mb][0], kUnscale, -beta0) : ss[mb][0];
        ss[mb][1] = mine ? fmaf(s[mb][1], kUnscale, -beta1) : ss[mb][1];
        ss[mb][2] = mine ? fmaf(s[mb][2], kUnscale, -beta0) : ss[mb][2];
        ss[mb][3] = mine ? fmaf(s[mb][3], kUnscale, -beta1) : ss[mb][3];
      }
    }
    // ---- online softmax (base 2) over the 32 tokens of each column ----------
    // Lazy rescaling: the reference max m moves only when a score exceeds it
    // by more than kSlack (weights then stay below 2^kSlack, well inside f16);
    // l and O always share the same m, so the final o = O / l is exact.  Each
    // lane tests its own scores; the column maxima are reduced across the
    // warp only when some lane asks for a move.
    constexpr float kSlack = 8.f;
    float mx0 = fmaxf(fmaxf(ss[0][0], ss[0][2]), fmaxf(ss[1][0], ss[1][2]));
    float mx1 = fmaxf(fmaxf(ss[0][1], ss[0][3]), fmaxf(ss[1][1], ss[1][3]));
    if (__any_sync(0xffffffffu, mx0 > st.m0 + kSlack || mx1 > st.m1 + kSlack)) {
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      const float mn0 = fmaxf(st.m0, mx0), mn1 = fmaxf(st.m1, mx1);
      const float a0 = st.m0 == -INFINITY ? 0.f : fast_exp2(st.m0 - mn0);
      const float a1 = st.m1 == -INFINITY ? 0.f : fast_exp2(st.m1 - mn1);
      st.m0 = mn0;
      st.m1 = mn1;
      st.l0 *= a0;
      st.l1 *= a1;
#pragma unroll
      for (int mt = 0; mt < S::kSteps; ++mt) {
        st.O[mt][0] *= a0;
        st.O[mt][1] *= a1;
        st.O[mt][2] *= a0;
        st.O[mt][3] *= a1;
      }
      st.C[0] *= a0;
      st.C[1] *= a1;
      st.C[2] *= a0;
      st.C[3] *= a1;
    }
    const float ms0 = st.m0 == -INFINITY ? 0.f : st.m0, ms1 = st.m1 == -INFINITY ? 0.f : st.m1;
    float pr[2][4];
#pragma unroll
    for (int mb = 0; mb < 2; ++mb) {
      pr[mb][0] = fast_exp2(ss[mb][0] - ms0);
      pr[mb][1] = fast_exp2(ss[mb][1] - ms1);
      pr[mb][2] = fast_exp2(ss[mb][2] - ms0);
      pr[mb][3] = fast_exp2(ss[mb][3] - ms1);
    }
    st.l0 += (pr[0][0] + pr[0][2]) + (pr[1][0] + pr[1][2]);
    st.l1 += (pr[0][1] + pr[0][3]) + (pr[1][1] + pr[1][3]);
    // ---- p / sV (Value scale of this thread's stream page), f16 -------------
    const float* vscale = reinterpret_cast<const float*>(vpg + geom.vscale_off) + sub * 32;
    uint32_t pk[2][2];
#pragma unroll
    for (int mb = 0; mb < 2; ++mb) {
      const int r0 = token_row0<BITS>(gid, mb);
      // undo the code's position factor: 4-bit x16 on the second row of each
      // pair; 2-bit x1, x4 (m-block 0) and x16, x64 (m-block 1)
      const float f0 = BITS == 2 ? (mb == 0 ? 1.f : 0.0625f) : 1.f;
      const float f1 = BITS == 2 ? (mb == 0 ? 0.25f : 0.015625f) : BITS == 4 && !TOKV ? 0.0625f : 1.f;
      const float i0 = fast_rcp(vscale[r0]) * f0;
      const float i1 = fast_rcp(vscale[r0 + kGap]) * f1;
      pk[mb][0] = pack_f16x2(pr[mb][0] * i0, pr[mb][1] * i0);
      pk[mb][1] = pack_f16x2(pr[mb][2] * i1, pr[mb][3] * i1);
    }
    // ---- O'^T += V'^T P' for every page, P' masked to the page's columns ------
#pragma unroll
    for (int j = 0; j < S::PB; ++j) {
      if (!FULL && j >= npages) break;
      const bool mine = sj == j;
      uint32_t bp[2][2];
#pragma unroll
      for (int mb = 0; mb < 2; ++mb) {
        bp[mb][0] = transpose8x8(mine ? pk[mb][0] : 0u);
        bp[mb][1] = transpose8x8(mine ? pk[mb][1] : 0u);
        // the p / sV sum for the Value bias (2-bit codes enter signed: none)
        if (BITS != 2) mma16816(st.C, kOneLo, kOneLo, kOneHi, kOneHi, bp[mb][0], bp[mb][1]);
      }
      const uint8_t* vc = pg[j] + geom.code_bytes + sub * S::kSubBytes;
      if constexpr (TOKV) {
        // this lane's D/16 bytes (channels gid D/8 ..) of token rows 8 tig + r,
        // one 32-bit word of each row at a time (four m-tiles).  Lanes of odd
        // tig load each pair of rows the other way round (w[2i] = row 2i + 1),
        // so the four tig lanes of a gid fall on two banks, not one; their P
        // halves are swapped to match (same dot products).
        constexpr int kLaneBytes = D / 16;
        const uint8_t* vrow = vc + 8 * tig * S::kRowBytes + gid * kLaneBytes;
        const int rflip = tig & 1;
        uint32_t bq[2][2];
#pragma unroll
        for (int mb = 0; mb < 2; ++mb) {
          bq[mb][0] = __byte_perm(bp[mb][0], 0u, rflip ? 0x1032u : 0x3210u);
          bq[mb][1] = __byte_perm(bp[mb][1], 0u, rflip ? 0x1032u : 0x3210u);
        }
#pragma unroll
        for (int wd = 0; wd < kLaneBytes / 4; ++wd) {
          uint32_t w[8];
#pragma unroll
          for (int r = 0; r < 8; ++r)
            w[r] = *reinterpret_cast<const uint32_t*>(vrow + (r ^ rflip) * S::kRowBytes + 4 * wd);
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const int mt = 4 * wd + m;
            // bytes (m of row a, m of row a, m of row b, m of row b): the low
            // nibbles are channel 2 mt of tokens a, b, the high ones channel 2 mt + 1
            constexpr uint32_t kSel[4] = {0x4400u, 0x5511u, 0x6622u, 0x7733u};
#pragma unroll
            for (int mb = 0; mb < 2; ++mb) {
              const uint32_t x01 = __byte_perm(w[4 * mb], w[4 * mb + 1], kSel[m]);
              const uint32_t x23 = __byte_perm(w[4 * mb + 2], w[4 * mb + 3], kSel[m]);
              mma16816(st.O[mt], x01 & 0x000F000Fu, x01 & 0x00F000F0u, x23 & 0x000F000Fu, x23 & 0x00F000F0u,
                       bq[mb][0], bq[mb][1]);
            }
          }
        }
        continue;
      }
#pragma unroll
      for (int mt = 0; mt < S::kSteps; ++mt) {
        const int c_lo = 16 * mt + gid, c_hi = c_lo + 8;
        if (BITS == 2) {
          const uint32_t pl = *reinterpret_cast<const uint16_t*>(vc + c_lo * 8 + 2 * tig);
          const uint32_t ph = *reinterpret_cast<const uint16_t*>(vc + c_hi * 8 + 2 * tig);
          uint32_t rl[4], rh[4];
          piece_regs(pl, rl);
          piece_regs(ph, rh);
          mma16816(st.O[mt], rl[0], rh[0], rl[1], rh[1], bp[0][0], bp[0][1]);
          mma16816(st.O[mt], rl[2], rh[2], rl[3], rh[3], bp[1][0], bp[1][1]);
        } else if (BITS == 4) {
          const uint32_t wl = *reinterpret_cast<const uint32_t*>(vc + c_lo * 16 + 4 * tig);
          const uint32_t wh = *reinterpret_cast<const uint32_t*>(vc + c_hi * 16 + 4 * tig);
          uint32_t rl[4], rh[4];
          nibble_regs(wl, rl);
          nibble_regs(wh, rh);
          mma16816(st.O[mt], rl[0], rh[0], rl[1], rh[1], bp[0][0], bp[0][1]);
          mma16816(st.O[mt], rl[2], rh[2], rl[3], rh[3], bp[1][0], bp[1][1]);
        } else {
          const uint2 vl = *reinterpret_cast<const uint2*>(vc + c_lo * 32 + 8 * tig);
          const uint2 vh = *reinterpret_cast<const uint2*>(vc + c_hi * 32 + 8 * tig);
          uint32_t rl[2], rh[2];
          byte_regs(vl.x, rl);
          byte_regs(vh.x, rh);
          mma16816(st.O[mt], rl[0], rh[0], rl[1], rh[1], bp[0][0], bp[0][1]);
          byte_regs(vl.y, rl);
          byte_regs(vh.y, rh);
          mma16816(st.O[mt], rl[0], rh[0], rl[1], rh[1], bp[1][0], bp[1][1]);
        }
      }
    }
  }
}

// A run of bf16 Key/Value rows on the tensor cores: the residual window of a
// unit (rows in its ring) or a range of a dense restored cache.  Steps of 16
// tokens: the rows are copied into a per-warp shared buffer with cp.async
// (16-byte chunks XOR-swizzled by row so ldmatrix is conflict free; rows past
// the run are zero-filled), double-buffered so the next step's copy overlaps
// this step's math when NBUF = 2; then S = K q with bf16 MMAs (q is the bf16 input, so every
// product is exact), the same online softmax as the pages, and O^T += V^T P
// with V^T read by ldmatrix.trans and P as a bf16 hi + lo pair.  Row t of the
// run is row (row0 + t) mod ring of kbase / vbase (RING), else row0 + t.
// Column n holds head (n % GP) % g of the unit; only n < g is kept.
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

template <int D, int GP, int NBUF, bool RING>
__device__ __forceinline__ void rows_mma(const DecodeParams& p, const __nv_bfloat16* kbase,
                                         const __nv_bfloat16* vbase, int64_t row0, int ring, int n,
                                         const __nv_bfloat16* qunit, int lane, int warp, int gid, int tig,
                                         uint8_t* wbuf, WarpState<D>& st, const __nv_bfloat16* last_k = nullptr,
                                         const __nv_bfloat16* last_v = nullptr) {
  constexpr int kRow = D * 2;             // bytes of one bf16 row
  constexpr int kChunks = kRow / 16;      // 16-byte chunks per row
  constexpr int kBuf = 32 * kRow;         // one step: 16 K rows + 16 V rows
  uint32_t bq[D / 16][2];
  {
    const __nv_bfloat16* q = qunit + (int64_t)((gid % GP) % p.g) * D;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      bq[kk][0] = *reinterpret_cast<const uint32_t*>(q + 16 * kk + 2 * tig);
      bq[kk][1] = *reinterpret_cast<const uint32_t*>(q + 16 * kk + 2 * tig + 8);
    }
  }
  const uint32_t buf_s = smem_addr(wbuf);
  const int nsteps = (n + 15) / 16;
  // copies of step stp into buffer half ``half``
  auto issue = [&](int stp, int half) {
    const int t0 = stp * 16;
    const uint32_t kb = buf_s + half * kBuf, vb = kb + 16 * kRow;
    for (int idx = lane; idx < 16 * kChunks; idx += 32) {
      const int r = idx / kChunks, c = idx - r * kChunks;
      const bool valid = t0 + r < n;
      const int64_t t = row0 + t0 + (valid ? r : 0);
      const int64_t row = RING ? t % ring : t;
      const uint32_t off = r * kRow + ((c ^ (r & 7)) * 16);
      // the run's last row may come from elsewhere (this step's input token)
      const bool last = last_k != nullptr && valid && t0 + r == n - 1;
      cp_async16(kb + off, last ? last_k + c * 8 : kbase + row * D + c * 8, valid ? 16u : 0u);
      cp_async16(vb + off, last ? last_v + c * 8 : vbase + row * D + c * 8, valid ? 16u : 0u);
    }
    cp_async_commit();
  };
  if (NBUF == 2 && warp < nsteps) issue(warp, 0);
  int half = 0;
  for (int stp = warp; stp < nsteps; stp += kMmaWarps, half ^= (NBUF - 1)) {
    if (NBUF == 1) {
      issue(stp, 0);
      cp_async_wait_group<0>();
    } else if (stp + kMmaWarps < nsteps) {
      issue(stp + kMmaWarps, half ^ 1);
      cp_async_wait_group<1>();
    } else {
      cp_async_wait_group<0>();
    }
    __syncwarp();
    const int t0 = stp * 16;
    const uint32_t kb_s = buf_s + half * kBuf, vb_s = kb_s + 16 * kRow;
    float s[4] = {0.f, 0.f, 0.f, 0.f};
    {
      const int r = (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t a[4];
        ldmatrix_x4(a, kb_s + r * kRow + (((2 * kk + (lane >> 4)) ^ (r & 7)) * 16));
        mma16816_bf16(s, a[0], a[1], a[2], a[3], bq[kk][0], bq[kk][1]);
      }
    }
    const bool v0 = t0 + gid < n, v1 = t0 + gid + 8 < n;
    s[0] = v0 ? s[0] * p.qk_scale : -INFINITY;
    s[1] = v0 ? s[1] * p.qk_scale : -INFINITY;
    s[2] = v1 ? s[2] * p.qk_scale : -INFINITY;
    s[3] = v1 ? s[3] * p.qk_scale : -INFINITY;
    float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float mn0 = fmaxf(st.m0, mx0), mn1 = fmaxf(st.m1, mx1);
    const float a0 = fast_exp2(st.m0 - mn0), a1 = fast_exp2(st.m1 - mn1);  // mn is finite: row 0 is valid
    st.m0 = mn0;
    st.m1 = mn1;
    const float p0 = fast_exp2(s[0] - mn0), p1 = fast_exp2(s[1] - mn1);
    const float p2 = fast_exp2(s[2] - mn0), p3 = fast_exp2(s[3] - mn1);
    st.l0 = fmaf(st.l0, a0, p0 + p2);
    st.l1 = fmaf(st.l1, a1, p1 + p3);
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      st.O[mt][0] *= a0;
      st.O[mt][1] *= a1;
      st.O[mt][2] *= a0;
      st.O[mt][3] *= a1;
    }
    uint32_t bh[2], bl[2];
    {
      const uint32_t h0 = pack_bf16x2(p0, p1), h1 = pack_bf16x2(p2, p3);
      const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&h0));
      const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&h1));
      bh[0] = transpose8x8(h0);
      bh[1] = transpose8x8(h1);
      bl[0] = transpose8x8(pack_bf16x2(p0 - f0.x, p1 - f0.y));
      bl[1] = transpose8x8(pack_bf16x2(p2 - f1.x, p3 - f1.y));
    }
    {
      const int r = (lane & 7) + 8 * (lane >> 4);
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        uint32_t a[4];
        ldmatrix_x4_trans(a, vb_s + r * kRow + (((2 * mt + ((lane >> 3) & 1)) ^ (r & 7)) * 16));
        mma16816_bf16(st.O[mt], a[0], a[1], a[2], a[3], bh[0], bh[1]);
        mma16816_bf16(st.O[mt], a[0], a[1], a[2], a[3], bl[0], bl[1]);
      }
    }
    __syncwarp();  // the buffer is refilled by a later step
  }
  // sums over the thread's rows -> over the warp's rows
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    st.l0 += __shfl_xor_sync(0xffffffffu, st.l0, off);
    st.l1 += __shfl_xor_sync(0xffffffffu, st.l1, off);
  }
}

// Merge the thread's (m, l, O) of its two columns with lane ^ off (same heads,
// another stream of pages).
template <int D>
__device__ __forceinline__ void merge_streams(WarpState<D>& st, int off) {
  const float m0o = __shfl_xor_sync(0xffffffffu, st.m0, off), m1o = __shfl_xor_sync(0xffffffffu, st.m1, off);
  const float l0o = __shfl_xor_sync(0xffffffffu, st.l0, off), l1o = __shfl_xor_sync(0xffffffffu, st.l1, off);
  const float M0 = fmaxf(st.m0, m0o), M1 = fmaxf(st.m1, m1o);
  const float s0 = M0 == -INFINITY ? 0.f : M0, s1 = M1 == -INFINITY ? 0.f : M1;
  const float fa0 = fast_exp2(st.m0 - s0), fb0 = fast_exp2(m0o - s0);
  const float fa1 = fast_exp2(st.m1 - s1), fb1 = fast_exp2(m1o - s1);
  st.l0 = st.l0 * fa0 + l0o * fb0;
  st.l1 = st.l1 * fa1 + l1o * fb1;
  st.m0 = M0;
  st.m1 = M1;
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) {
    const float o0 = __shfl_xor_sync(0xffffffffu, st.O[mt][0], off);
    const float o1 = __shfl_xor_sync(0xffffffffu, st.O[mt][1], off);
    const float o2 = __shfl_xor_sync(0xffffffffu, st.O[mt][2], off);
    const float o3 = __shfl_xor_sync(0xffffffffu, st.O[mt][3], off);
    st.O[mt][0] = st.O[mt][0] * fa0 + o0 * fb0;
    st.O[mt][1] = st.O[mt][1] * fa1 + o1 * fb1;
    st.O[mt][2] = st.O[mt][2] * fa0 + o2 * fb0;
    st.O[mt][3] = st.O[mt][3] * fa1 + o3 * fb1;
  }
}

// Fold the four warps' (m, l, O) of the stream-0 columns into one partial
// (o = sum O, m, l per query head) of slot ``slot`` of ``unit``.  ``buf`` is
// shared memory no warp still reads (kMmaWarps * kMaxGqa * (D + 2) floats).
// tokv: O'^T rows hold the channels of mma_group's token-major Value path.
template <int D, int GP>
__device__ __forceinline__ void write_partial(const DecodeParams& p, int64_t unit, int slot, int warp,
                                              int gid, int tig, const WarpState<D>& st, uint8_t* buf,
                                              bool tokv = false) {
  const int g = p.g;

  float* mrg = reinterpret_cast<float*>(buf);  // [kMmaWarps][kMaxGqa][D + 2]
  const int hd0 = 2 * tig, hd1 = 2 * tig + 1;  // heads of the stream-0 columns
  float* mw = mrg + (size_t)warp * kMaxGqa * (D + 2);
  const bool stream0 = 2 * tig < GP && warp < kMmaWarps;  // a fifth (control) warp holds no rows
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) {
    const int c_lo = tokv ? gid * (D / 8) + 2 * mt : 16 * mt + gid;
    const int c_hi = tokv ? c_lo + 1 : c_lo + 8;
    if (stream0 && hd0 < g) {
      mw[hd0 * (D + 2) + c_lo] = st.O[mt][0];
      mw[hd0 * (D + 2) + c_hi] = st.O[mt][2];
    }
    if (stream0 && hd1 < g) {
      mw[hd1 * (D + 2) + c_lo] = st.O[mt][1];
      mw[hd1 * (D + 2) + c_hi] = st.O[mt][3];
    }
  }
  if (gid == 0 && stream0) {
    if (hd0 < g) {
      mw[hd0 * (D + 2) + D] = st.m0;
      mw[hd0 * (D + 2) + D + 1] = st.l0;
    }
    if (hd1 < g) {
      mw[hd1 * (D + 2) + D] = st.m1;
      mw[hd1 * (D + 2) + D + 1] = st.l1;
    }
  }
  __syncthreads();
  float* part = p.partials + (unit * p.max_splits + slot) * (int64_t)g * part_row(D);
  for (int idx = threadIdx.x; idx < g * D; idx += blockDim.x) {
    const int j = idx / D, c = idx - j * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kMmaWarps; ++w) M = fmaxf(M, mrg[((size_t)w * kMaxGqa + j) * (D + 2) + D]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kMmaWarps; ++w) {
        const float* r = mrg + ((size_t)w * kMaxGqa + j) * (D + 2);
        if (r[D] == -INFINITY) continue;
        const float f = exp2f(r[D] - M);
        L = fmaf(r[D + 1], f, L);
        O = fmaf(r[c], f, O);
      }
    }
    part[(int64_t)j * part_row(D) + c] = O;
    if (c == 0) {
      part[(int64_t)j * part_row(D) + D] = M;
      part[(int64_t)j * part_row(D) + D + 1] = L;
    }
  }
}

// Per-warp shared bytes of rows_mma: NBUF steps of 16 Key + 16 Value bf16 rows.
template <int D, int NBUF>
constexpr int kRowsBuf = NBUF * 32 * D * 2;

// Page modes of the split kernel: contiguous pages of G = 32, paged pages of
// G = 32, any larger G (either map) staged in 32-token units, and the
// 32-token tiles of a segmented cache (4-bit; token-major Value rows).
constexpr int kFlat32 = 0, kPaged32 = 1, kStaged = 2, kSeg32 = 3;

// A tile of a segmented cache that the tensor cores cannot take: its tokens
// span more than one segment (so more than one Key scale row), or it is the
// unit's last, partial tile (nvalid < 32 tokens).  Its tokens go through the
// CUDA cores in fp32: lane r scores token t0 + r against every head with its
// own segment's Key scale row; the warp then folds the tile into stream 0 of
// the tensor-core state (mma_group, token-major Value path): the same lazy
// running max (moved only past 2^8), l, and O' -- unbiased codes x 2^-24, x16
// on the odd-channel rows, so the bias counter C takes nothing.  pw: 32 x GP
// floats of this warp's shared memory.
template <int D, int GP>
__device__ __noinline__ void seg_tile_cuda_cores(const DecodeParams& p, const uint8_t* tile, int64_t unit_row,
                                                 const int32_t* first, int t0, int nvalid, const float4* q4,
                                                 float* pw, WarpState<D>& st, int lane) {
  using S = Shape<D, 4, GP>;
  constexpr float kTwo24i = 1.f / 16777216.f;
  constexpr float kSlack = 8.f;  // as mma_group's lazy rescaling
  const PageGeom ug = make_geom(32, D, 4);
  const int gid = lane >> 2, tig = lane & 3;
  const float* qf = reinterpret_cast<const float*>(q4);
  // ---- scores of token t0 + lane, every head (base 2, q pre-scaled)
  float sc[GP];
#pragma unroll
  for (int n = 0; n < GP; ++n) sc[n] = -INFINITY;
  if (lane < nvalid) {
    const float4* ks = reinterpret_cast<const float4*>(p.seg.kscales + (unit_row + first[t0 + lane]) * D);
    const uint32_t* kr = reinterpret_cast<const uint32_t*>(tile + lane * S::kRowBytes);
#pragma unroll
    for (int n = 0; n < GP; ++n) sc[n] = 0.f;
    for (int w8 = 0; w8 < D / 8; ++w8) {
      const uint32_t w = kr[w8];
      const float4 sa = __ldg(ks + 2 * w8), sb = __ldg(ks + 2 * w8 + 1);
      const float sk[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int c = 8 * w8 + e;
        const float kv = (float)((int)((w >> (4 * e)) & 0xFu) - 8) * fast_rcp(fmaxf(sk[e], p.eps));
        const int tg = c / S::kChan, i4 = (c - tg * S::kChan) >> 2;
#pragma unroll
        for (int n = 0; n < GP; ++n) sc[n] = fmaf(qf[((i4 * GP + n) * 4 + tg) * 4 + (c & 3)], kv, sc[n]);
      }
    }
  }
  // ---- per-head maxima; the lazy max of this thread's stream-0 columns
  float mx[GP];
#pragma unroll
  for (int n = 0; n < GP; ++n) {
    mx[n] = sc[n];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx[n] = fmaxf(mx[n], __shfl_xor_sync(0xffffffffu, mx[n], off));
  }
  const bool own = 2 * tig < GP;  // this thread's columns are stream 0's heads 2 tig, 2 tig + 1
  float mxa = -INFINITY, mxb = -INFINITY;
#pragma unroll
  for (int n = 0; n < GP; n += 2)
    if (2 * tig == n) {
      mxa = mx[n];
      mxb = mx[n + 1];
    }
  if (own && mxa > st.m0 + kSlack) {
    const float mn = fmaxf(st.m0, mxa), a = st.m0 == -INFINITY ? 0.f : fast_exp2(st.m0 - mn);
    st.m0 = mn;
    st.l0 *= a;
    st.C[0] *= a;
    st.C[2] *= a;
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      st.O[mt][0] *= a;
      st.O[mt][2] *= a;
    }
  }
  if (own && mxb > st.m1 + kSlack) {
    const float mn = fmaxf(st.m1, mxb), a = st.m1 == -INFINITY ? 0.f : fast_exp2(st.m1 - mn);
    st.m1 = mn;
    st.l1 *= a;
    st.C[1] *= a;
    st.C[3] *= a;
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      st.O[mt][1] *= a;
      st.O[mt][3] *= a;
    }
  }
  // ---- weights p = 2^(s - m) of token lane, head n (column n's m sits in lane n / 2)
#pragma unroll
  for (int n = 0; n < GP; ++n) {
    const float m = __shfl_sync(0xffffffffu, (n & 1) ? st.m1 : st.m0, n >> 1);
    const float pv = lane < nvalid ? fast_exp2(sc[n] - m) : 0.f;
    pw[lane * GP + n] = pv;
    float ls = pv;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, off);
    // l is summed over a column's rows (gid) at the end: count it once
    if (gid == 0 && 2 * tig == n) st.l0 += ls;
    if (gid == 0 && 2 * tig + 1 == n) st.l1 += ls;
  }
  __syncwarp();
  // ---- O'^T += V^T p / sV on this thread's channels and columns
  if (own) {
    const float* vscale = reinterpret_cast<const float*>(tile + ug.vscale_off);
    const uint8_t* vrows = tile + ug.code_bytes + gid * (D / 16);
    for (int r = 0; r < nvalid; ++r) {
      const float iv = fast_rcp(vscale[r]) * kTwo24i;
      const float w0 = pw[r * GP + 2 * tig] * iv, w1 = pw[r * GP + 2 * tig + 1] * iv;
#pragma unroll
      for (int wd = 0; wd < D / 64; ++wd) {
        const uint32_t word = *reinterpret_cast<const uint32_t*>(vrows + r * S::kRowBytes + 4 * wd);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int mt = 4 * wd + m;
          const float vlo = (float)((int)((word >> (8 * m)) & 0xFu) - 8);
          const float vhi = 16.f * (float)((int)((word >> (8 * m + 4)) & 0xFu) - 8);
          st.O[mt][0] = fmaf(vlo, w0, st.O[mt][0]);
          st.O[mt][1] = fmaf(vlo, w1, st.O[mt][1]);
          st.O[mt][2] = fmaf(vhi, w0, st.O[mt][2]);
          st.O[mt][3] = fmaf(vhi, w1, st.O[mt][3]);
        }
      }
    }
  }
  __syncwarp();
}

// A short split item (a few pages a warp, as at batch 1) spends most of its
// time waiting: its first copies are issued only after the query set-up,
// which itself waits on global loads.  Lane 0 of each warp therefore asks L2
// for the warp's first pages before that set-up (whole pages of a contiguous
// G = 32 cache), so the copies then hit L2.
__device__ __forceinline__ void prefetch_first_pages(const uint8_t* unit_pages, int64_t stored, int pg0, int pg1,
                                                     int warp, int n) {
  for (int k = 0; k < n; ++k) {
    const int pg = pg0 + warp + k * kMmaWarps;
    if (pg >= pg1) break;
    prefetch_l2(unit_pages + (int64_t)pg * stored, (uint32_t)stored);
  }
}

// The CUDA-core path of an item the range test sends there, kept out of line
// so that the page loop's code stays compact (the layer's split 76.2 -> 75.8
// us, measured).
template <int BITS, int D, bool SEG>
__device__ __noinline__ void range_fallback(const DecodeParams& p, int i, int h, int pg0, int pg1, int slot,
                                            float* scratch) {
  simt_item<__nv_bfloat16, BITS, D / 32, SEG>(p, i, h, false, pg0, pg1, slot, scratch);
}

// The combine inside the split launch (DecodeParams::done): after its partial
// is written, a CTA counts itself finished for its unit, and the CTA that
// finishes the unit's last item merges the unit's g query heads (one warp
// each, merge_head) into the output and sets the count back to 0 for the
// next launch.  The count is one device-scope acquire-release atomic: the
// barrier before it orders every thread's partial writes ahead of its
// release, and for the last CTA its acquire (passed on by the barrier after
// it) orders the others' partials ahead of the merge's loads, which read L2.
// No CTA waits for another.
__device__ __forceinline__ uint32_t arrive_acq_rel(uint32_t* counter) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(counter) : "memory");
  return old;
}

template <int D>
__device__ __noinline__ void finish_unit(const DecodeParams& p, int i, int h) {
  __shared__ uint32_t last;
  const int b = p.seq_begin + i;
  const int64_t unit = (int64_t)b * p.Hkv + h;
  const int T0 = p.ctr[i].total, Q0 = p.ctr[i].quantized;
  const int nsplit = (Q0 / p.G + p.chunk_pages - 1) / p.chunk_pages;
  const int nslots = nsplit + (T0 > Q0 ? 1 : 0);
  __syncthreads();
  if (threadIdx.x == 0) last = arrive_acq_rel(p.done + unit) + 1u == (uint32_t)nslots;
  __syncthreads();
  if (!last) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t stride = (int64_t)p.g * part_row(D);
  const float* base = p.partials + unit * p.max_splits * stride;
  for (int j = warp; j < p.g; j += kMmaWarps)
    merge_head<D <= 128 ? 1 : 2, true>(base + (int64_t)j * part_row(D), nsplit, nslots, p.max_splits, stride, D,
                                       p.out + ((int64_t)b * p.Hq + (int64_t)h * p.g + j) * D, lane);
  if (threadIdx.x == 0) p.done[unit] = 0u;
}

// The residual-window item of unit (sequence i of the launch, KV head h): its
// ring rows on the tensor cores (plus, for kvq_decode_step, this step's token,
// which it also stores into its ring row).  ``buf`` holds kRowsBuf<D, 2> bytes
// per warp: each warp's next 16 rows are copied in while it works on these.
template <int D, int GP>
__device__ __forceinline__ void window_rows(const DecodeParams& p, int i, int h, int lane, int warp, int gid, int tig,
                                            uint8_t* buf, WarpState<D>& st) {
  const int b = p.seq_begin + i;
  const int64_t unit = (int64_t)b * p.Hkv + h;
  const int64_t T0 = p.ctr[i].total, Q0 = p.ctr[i].quantized;
  __nv_bfloat16* rk = reinterpret_cast<__nv_bfloat16*>(const_cast<void*>(p.ring_k)) + unit * p.Rcap * D;
  __nv_bfloat16* rv = reinterpret_cast<__nv_bfloat16*>(const_cast<void*>(p.ring_v)) + unit * p.Rcap * D;
  const __nv_bfloat16* lk = nullptr;
  const __nv_bfloat16* lv = nullptr;
  if (p.step_k) {
    // this step's token: attended from the input and stored in its ring row
    // (row (T0 - 1) mod Rcap holds no other token of the window, so no copy
    // of this launch reads it)
    lk = reinterpret_cast<const __nv_bfloat16*>(p.step_k) + ((int64_t)i * p.Hkv + h) * D;
    lv = reinterpret_cast<const __nv_bfloat16*>(p.step_v) + ((int64_t)i * p.Hkv + h) * D;
    const int64_t row = ((T0 - 1) % p.Rcap) * D;
    for (int c = threadIdx.x; c < D / 8; c += blockDim.x) {
      reinterpret_cast<uint4*>(rk + row)[c] = reinterpret_cast<const uint4*>(lk)[c];
      reinterpret_cast<uint4*>(rv + row)[c] = reinterpret_cast<const uint4*>(lv)[c];
    }
  }
  rows_mma<D, GP, 2, true>(p, rk, rv, Q0, p.Rcap, (int)(T0 - Q0),
                           reinterpret_cast<const __nv_bfloat16*>(p.q) + ((int64_t)b * p.Hq + h * p.g) * D, lane,
                           warp, gid, tig, buf + (size_t)warp * kRowsBuf<D, 2>, st, lk, lv);
}

// A window item whole, out of line: its state, its rows and its partial, so
// that the page path's code stays compact and no state crosses the call (the
// layer's split 76.2 -> 74.9 us, measured).
template <int D, int GP>
__device__ __noinline__ void window_item(const DecodeParams& p, int i, int h, int slot, uint8_t* buf) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gid = lane >> 2, tig = lane & 3;
  WarpState<D> st;
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) st.O[mt][0] = st.O[mt][1] = st.O[mt][2] = st.O[mt][3] = 0.f;
  st.C[0] = st.C[1] = st.C[2] = st.C[3] = 0.f;
  st.m0 = st.m1 = -INFINITY;
  st.l0 = st.l1 = 0.f;
  window_rows<D, GP>(p, i, h, lane, warp, gid, tig, buf, st);
  __syncthreads();  // every warp is done with its buffers: reuse them for the merge
  write_partial<D, GP>(p, (int64_t)(p.seq_begin + i) * p.Hkv + h, slot, warp, gid, tig, st, buf, false);
}

template <int D, int BITS, int GP, int MODE>
__global__ void __launch_bounds__(kMmaThreads, 3) decode_mma_kernel(const DecodeParams p, int slots) {
  using S = Shape<D, BITS, GP>;
  extern __shared__ __align__(128) uint8_t smem[];
  pdl_wait();
  pdl_release();
  // column-major over (split column, unit): every unit's first chunk, then
  // every unit's second, ..., the windows last, so the last wave holds the
  // shortest items
  const int n_units = p.n_seqs * p.Hkv;
  const int col = blockIdx.x / n_units;
  const int u = blockIdx.x - col * n_units;
  const int i = u / p.Hkv, h = u - i * p.Hkv;
  const int b = p.seq_begin + i;
  bool win;
  int pg0, pg1, slot;
  if (p.done && col == 0 && p.ctr[i].total == 0) {
    // a unit without tokens: zeros (no item of it runs)
    float* o = p.out + ((int64_t)(p.seq_begin + i) * p.Hq + (int64_t)h * p.g) * D;
    for (int idx = threadIdx.x; idx < p.g * D; idx += blockDim.x) o[idx] = 0.f;
    return;
  }
  if (!split_item(p, col, i, &win, &pg0, &pg1, &slot)) return;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gid = lane >> 2, tig = lane & 3;
  const int g = p.g;
  // Ring slots hold 32-token units.  With G = 32 a unit is a whole page (one
  // bulk copy); with a larger G it is the unit's Key rows, Value sub-tile,
  // the page's Key scales and the unit's Value scales (four copies) laid out
  // as a G = 32 page, so shared memory and the math do not depend on G.
  const PageGeom geom = p.geom;                                      // a stored page
  const int upp = MODE == kStaged ? p.G / 32 : 1;                    // units per page
  const PageGeom ug = MODE == kStaged || MODE == kSeg32 ? make_geom(32, D, BITS) : geom;  // a staged unit
  const uint32_t page_bytes = (uint32_t)ug.page_bytes;              // bytes of a slot
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  float* scratch = reinterpret_cast<float*>(smem + 128 * ((kMmaWarps * slots * 8 + 127) / 128));
  float* my_rsc = scratch + warp * S::PB * D;
  float4* q4 = reinterpret_cast<float4*>(scratch + kMmaWarps * S::PB * D);  // GP * D floats
  uint8_t* buf = reinterpret_cast<uint8_t*>(scratch + kMmaWarps * S::PB * D + GP * D + 32);
  uint8_t* my_buf = buf + (size_t)warp * slots * page_bytes;
  const uint32_t my_bar = smem_addr(bars + warp * slots);

  WarpState<D> st;
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) st.O[mt][0] = st.O[mt][1] = st.O[mt][2] = st.O[mt][3] = 0.f;
  st.C[0] = st.C[1] = st.C[2] = st.C[3] = 0.f;
  st.m0 = st.m1 = -INFINITY;
  st.l0 = st.l1 = 0.f;
  bool ok = true;

  // (8-bit codes keep the window inline: with the call their page loop
  // spills more, and the 8-bit ragged decode measured 158.7 against 154.6 us)
  if (BITS == 8 && win) {
    window_rows<D, GP>(p, i, h, lane, warp, gid, tig, buf, st);
  } else if (win) {
    window_item<D, GP>(p, i, h, slot, buf);
    if (p.done) finish_unit<D>(p, i, h);
    return;
  } else {
  // The loads that depend only on the unit go out first, all at once: the
  // unit's flushed maxima, this thread's 8 query channels and (contiguous
  // G = 32) its page base; a short decode would otherwise wait on each in turn.
  uint2 rng = make_uint2(0u, 0u);
  if (p.range) rng = __ldg(reinterpret_cast<const uint2*>(p.range + 2 * ((int64_t)b * p.Hkv + h)));
  static_assert(GP * D / 8 <= kMmaThreads, "one 16-byte query load a thread");
  uint4 qraw = make_uint4(0u, 0u, 0u, 0u);
  if (threadIdx.x < GP * D / 8) {
    const int n = threadIdx.x / (D / 8), c0 = (threadIdx.x - n * (D / 8)) * 8;
    qraw = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p.q) +
                                                ((int64_t)b * p.Hq + (int64_t)h * g + n % g) * D + c0));
  }
  int64_t unit_base = 0;
  if (MODE == kFlat32) unit_base = p.map.layout[b].page_base + h * p.map.layout[b].unit_stride;
  if (MODE == kFlat32 && lane == 0 && pg1 - pg0 <= kShortItemPages)
    prefetch_first_pages(p.pages + unit_base, (int64_t)p.geom.page_bytes, pg0, pg1, warp, slots);
  // the unit's flushed maxima, for the range test below
  const float kabs = __uint_as_float(rng.x), vabs = __uint_as_float(rng.y);
  // queries of the GP column heads (head n % g for the padding columns, so every
  // value stays finite), pre-scaled, in shared memory: channel c of head n goes
  // to float4 ((i * GP + n) * 4 + tig) with tig = c / (D/4), i = (c % (D/4)) / 4,
  // so the lanes that read together hit distinct banks
  // (8 channels a thread from one 16-byte load, every load of the CTA in
  // flight at once)
  float qa = 0.f;
  {
    const int x = threadIdx.x;
    if (x < GP * D / 8) {
      const int n = x / (D / 8), c0 = (x - n * (D / 8)) * 8;
      const __nv_bfloat162* q2 = reinterpret_cast<const __nv_bfloat162*>(&qraw);
      float qv[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(q2[e]);
        qv[2 * e] = f.x * p.qk_scale;
        qv[2 * e + 1] = f.y * p.qk_scale;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) qa = fmaxf(qa, fabsf(qv[e]));
      const int tg = c0 / S::kChan, i4 = (c0 - tg * S::kChan) >> 2;  // channels c0 .. c0 + 3, then i4 + 1
      q4[(i4 * GP + n) * 4 + tg] = make_float4(qv[0], qv[1], qv[2], qv[3]);
      q4[((i4 + 1) * GP + n) * 4 + tg] = make_float4(qv[4], qv[5], qv[6], qv[7]);
    }
  }
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) qa = fmaxf(qa, __shfl_xor_sync(0xffffffffu, qa, off));
  float* qred = reinterpret_cast<float*>(q4) + GP * D;  // kMmaWarps floats
  if (lane == 0) qred[warp] = qa;
  __syncthreads();
  {
    // the range test (see kVWideAbs): every flushed Key scale is at least
    // qmax / max(largest Key absmax, eps) rounded, which is >= kthr when the
    // product below stays under qmax by more than its rounding
#pragma unroll
    for (int w = 0; w < kMmaWarps; ++w) qa = fmaxf(qa, qred[w]);
    const int qexp = float_exp2i(qa);
    const float kthr = fmaxf(pow2i(BITS == 2 ? qexp + 1 + 4 - 14 : qexp + 1 - 9), p.eps);
    if (!(fmaxf(kabs, p.eps) * kthr <= (float)p.qmax * 0.9999f && vabs <= kVWideAbs * 0.999f)) {
      range_fallback<BITS, D, MODE == kSeg32>(p, i, h, pg0, pg1, slot, reinterpret_cast<float*>(buf));
      if (p.done) finish_unit<D>(p, i, h);
      return;
    }
  }

  // source of this warp's pos-th unit (units u0 + warp, + 4, ...), through
  // the block table for a paged cache
  const int64_t stored = geom.page_bytes;
  const uint8_t* unit_pages = MODE == kFlat32 ? p.pages + unit_base : p.pages;
  auto page_src = [&](int pg) {
    return MODE == kFlat32 ? unit_pages + (int64_t)pg * stored : p.pages + page_offset(p.map, stored, b, h, pg);
  };
  auto src_of = [&](int pos) { return page_src(pg0 + warp + pos * kMmaWarps); };  // G = 32
  const int npg = MODE == kSeg32 ? (pg1 - pg0 + 31) / 32 : (pg1 - pg0) * upp;  // units of this CTA
  const int my_n = warp < npg ? (npg - warp + kMmaWarps - 1) / kMmaWarps : 0;
  // segmented cache: the warp's tiles pg0 / 32 + warp + 4 pos; per tile the
  // first token of its first token's segment (whose row holds the segment's
  // Key scales) and whether every token is in that segment and below Q,
  // loaded by the lanes for 32 positions at a time (lane k: position
  // seg_base + k); lane 0 marks each slot's tile (seg_flag) as it issues it
  const int64_t unit_row = ((int64_t)b * p.Hkv + h) * p.seg.cap;
  const int32_t* seg_first = MODE == kSeg32 ? p.seg.first + (int64_t)b * p.seg.cap : nullptr;
  const int Qseg = p.ctr[i].quantized;
  int seg_base = -64, seg_f = 0;
  bool seg_u = false;
  uint8_t* seg_flag = my_buf + (size_t)(kMmaWarps - warp) * slots * page_bytes + (size_t)warp * 8;
  float* seg_pw = reinterpret_cast<float*>(my_buf + (size_t)(kMmaWarps - warp) * slots * page_bytes + 32) +
                  warp * 32 * GP;
  auto seg_tile = [&](int pos) { return pg0 / 32 + warp + pos * kMmaWarps; };
  auto seg_load = [&](int pos) {  // all lanes: the 32 positions from pos's block
    seg_base = pos & ~31;
    const int t = seg_tile(seg_base + lane);
    seg_f = 0;
    seg_u = false;
    if (seg_base + lane < my_n) {
      seg_f = seg_first[32 * t];
      seg_u = 32 * t + 31 < Qseg && seg_first[32 * t + 31] == seg_f;
    }
  };
  // the copies of unit pos into slot s (lane 0); f, u: its tile's scale row and mark (segmented)
  auto issue = [&](int pos, int s, int f, bool u) {
    const uint32_t bar = my_bar + 8 * s, dst = smem_addr(my_buf + (size_t)s * page_bytes);
    if constexpr (MODE == kSeg32) seg_flag[s] = u ? 1 : 0;
    mbar_expect_tx(bar, page_bytes);
    if constexpr (MODE == kSeg32) {
      const int64_t row = unit_row + 32 * (int64_t)seg_tile(pos);
      const int rb = S::kRowBytes;
      bulk_load(dst, p.seg.kcodes + row * rb, 32 * rb, bar);
      bulk_load(dst + (uint32_t)ug.code_bytes, p.seg.vcodes + row * rb, 32 * rb, bar);
      bulk_load(dst + (uint32_t)ug.kscale_off, p.seg.kscales + (unit_row + f) * D, 4 * D, bar);
      bulk_load(dst + (uint32_t)ug.vscale_off, p.seg.vscales + row, 128, bar);
    } else if constexpr (MODE != kStaged) {
      bulk_load(dst, src_of(pos), page_bytes, bar);
    } else {
      const int u = pg0 * upp + warp + pos * kMmaWarps;
      const int pg = u / upp, sub = u - pg * upp;
      const uint8_t* src = page_src(pg);
      bulk_load(dst, src + sub * 32 * S::kRowBytes, 32 * S::kRowBytes, bar);
      bulk_load(dst + (uint32_t)ug.code_bytes, src + geom.code_bytes + sub * S::kSubBytes, S::kSubBytes, bar);
      bulk_load(dst + (uint32_t)ug.kscale_off, src + geom.kscale_off, 4 * D, bar);
      bulk_load(dst + (uint32_t)ug.vscale_off, src + geom.vscale_off + 128 * sub, 128, bar);
    }
  };
  if (MODE == kSeg32) seg_load(0);
  if (lane == 0) {
    for (int s = 0; s < slots; ++s) mbar_init(my_bar + 8 * s, 1);
    fence_mbar_init();
    fence_proxy_async();
  }
  for (int s = 0; s < slots && s < my_n; ++s) {
    int f = 0;
    bool u = false;
    if (MODE == kSeg32) {
      f = __shfl_sync(0xffffffffu, seg_f, s);
      u = __shfl_sync(0xffffffffu, seg_u, s);
    }
    if (lane == 0) issue(s, s, f, u);
  }
  __syncwarp();
  // Pages are consumed in issue order; page k sits in slot k mod slots, and
  // bit t of ``phases`` is the parity slot t's barrier completes next.  Every
  // lane keeps the same counters; lane 0 issues the copies.
  int k = 0, sidx = 0, consumed = 0, issued = slots < my_n ? slots : my_n;
  uint32_t phases = 0;
  // contiguous G = 32: the source pointer advances by whole runs
  const uint8_t* next_src = MODE == kFlat32 ? src_of(issued) : nullptr;
  for (; k < my_n; k += S::PB) {
    const int np = min(S::PB, my_n - k);
    int sl[S::PB];
    const uint8_t* pgs[S::PB];
#pragma unroll
    for (int j = 0; j < S::PB; ++j) {
      int t = sidx + (j < np ? j : np - 1);
      if (t >= slots) t -= slots;
      sl[j] = t;
      pgs[j] = my_buf + (size_t)t * page_bytes;
    }
#pragma unroll
    for (int j = 0; j < S::PB; ++j) {
      if (j < np && ok) {
        ok = mbar_wait(my_bar + 8 * sl[j], (phases >> sl[j]) & 1u);
        if (ok) {
          phases ^= 1u << sl[j];
          ++consumed;
        }
      }
    }
    if (!ok) break;
    if constexpr (MODE == kSeg32) {
      if constexpr (BITS == 4) {
        bool all = true;
#pragma unroll
        for (int j = 0; j < S::PB; ++j)
          if (j < np) all = all && seg_flag[sl[j]] != 0;
        if (all && np == S::PB) {
          mma_group<D, BITS, GP, true, true>(pgs, np, ug, 32, q4, my_rsc, lane, gid, tig, st);
        } else if (all) {
          mma_group<D, BITS, GP, false, true>(pgs, np, ug, 32, q4, my_rsc, lane, gid, tig, st);
        } else {
#pragma unroll
          for (int j = 0; j < S::PB; ++j) {
            if (j >= np) break;
            if (seg_flag[sl[j]]) {
              const uint8_t* one[S::PB];
#pragma unroll
              for (int jj = 0; jj < S::PB; ++jj) one[jj] = pgs[j];
              mma_group<D, BITS, GP, false, true>(one, 1, ug, 32, q4, my_rsc, lane, gid, tig, st);
            } else {
              const int t0 = 32 * seg_tile(k + j);
              seg_tile_cuda_cores<D, GP>(p, pgs[j], unit_row, seg_first, t0, min(32, Qseg - t0), q4, seg_pw, st,
                                         lane);
            }
            __syncwarp();
          }
        }
      }
    } else if (np == S::PB) {
      mma_group<D, BITS, GP, true>(pgs, np, ug, MODE == kStaged ? p.G / upp : p.G, q4, my_rsc, lane, gid, tig, st);
    } else {
      mma_group<D, BITS, GP, false>(pgs, np, ug, MODE == kStaged ? p.G / upp : p.G, q4, my_rsc, lane, gid, tig, st);
    }
    __syncwarp();
    // refill the freed slots with the next pages of this warp's run
    const int refill = min(np, my_n - issued);
    int seg_fs[S::PB];
    bool seg_us[S::PB];
    if (MODE == kSeg32) {
#pragma unroll
      for (int j = 0; j < S::PB; ++j) {
        if (j < refill && issued + j >= seg_base + 32) seg_load(issued + j);
        seg_fs[j] = __shfl_sync(0xffffffffu, seg_f, (issued + j) & 31);
        seg_us[j] = __shfl_sync(0xffffffffu, seg_u, (issued + j) & 31);
      }
    }
    if (lane == 0 && refill > 0) {
      fence_proxy_async();
#pragma unroll
      for (int j = 0; j < S::PB; ++j) {
        if (j < refill) {
          if (MODE != kFlat32) {
            issue(issued + j, sl[j], MODE == kSeg32 ? seg_fs[j] : 0, MODE == kSeg32 ? seg_us[j] : false);
          } else {
            mbar_expect_tx(my_bar + 8 * sl[j], page_bytes);
            bulk_load(smem_addr(my_buf + (size_t)sl[j] * page_bytes), next_src + (int64_t)j * kMmaWarps * page_bytes,
                      page_bytes, my_bar + 8 * sl[j]);
          }
        }
      }
    }
    if (MODE == kFlat32) next_src += (int64_t)refill * kMmaWarps * page_bytes;
    issued += refill;
    sidx += np;
    if (sidx >= slots) sidx -= slots;
  }
  if (!ok) {
    // drain the copies still in flight (bounded), report, and contribute nothing
    for (int kk = consumed; kk < issued; ++kk) {
      const int t = kk % slots;
      mbar_wait(my_bar + 8 * t, (phases >> t) & 1u);
      phases ^= 1u << t;
    }
    if (lane == 0) atomicOr(p.status, kStatusWaitTimeout);
    st.m0 = st.m1 = -INFINITY;
    st.l0 = st.l1 = 0.f;
    st.C[0] = st.C[1] = st.C[2] = st.C[3] = 0.f;
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) st.O[mt][0] = st.O[mt][1] = st.O[mt][2] = st.O[mt][3] = 0.f;
  }
  // sums over the thread's rows -> over the warp's rows; undo the code bias
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    st.l0 += __shfl_xor_sync(0xffffffffu, st.l0, off);
    st.l1 += __shfl_xor_sync(0xffffffffu, st.l1, off);
  }
  {
    // C holds 2^-24 * sum of p/sV per column (every row of the counter MMA
    // carries the full sum), so the bias term is bias * 2^24 * C
    constexpr float kTwo24 = 16777216.f;
    const float c0 = S::kBias * kTwo24 * st.C[0], c1 = S::kBias * kTwo24 * st.C[1];
    // (segmented tiles: the second row of each m-tile, an odd channel, came x16)
    constexpr float kTwo24hi = MODE == kSeg32 ? kTwo24 / 16.f : kTwo24;
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      st.O[mt][0] = fmaf(st.O[mt][0], kTwo24, -c0);
      st.O[mt][1] = fmaf(st.O[mt][1], kTwo24, -c1);
      st.O[mt][2] = fmaf(st.O[mt][2], kTwo24hi, -c0);
      st.O[mt][3] = fmaf(st.O[mt][3], kTwo24hi, -c1);
    }
  }
  // fold the page streams onto stream 0 (columns 0 .. GP-1)
#pragma unroll
  for (int off = GP / 2; off < 4; off <<= 1) merge_streams<D>(st, off);
  }  // page path
  __syncthreads();  // every warp is done with its slots: reuse them for the merge
  write_partial<D, GP>(p, (int64_t)b * p.Hkv + h, slot, warp, gid, tig, st, buf, MODE == kSeg32 && !win);
  if (p.done) finish_unit<D>(p, i, h);
}

// Decode attention over a dense bf16 Key/Value cache ([batch][Hkv][t_stride][D],
// as kvq_restore writes it): the second half of the dequantize-to-HBM read
// path, kept as the measured foil of the fused kernel.  One CTA per
// (token chunk, unit), column-major like the fused kernel; its four warps take
// 16-token steps round robin through rows_mma (double-buffered) and the CTA
// writes the chunk's partial to slot ``chunk``.
template <int D, int GP>
__global__ void __launch_bounds__(kMmaThreads) decode_dense_kernel(const DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  pdl_wait();
  pdl_release();
  const int n_units = p.n_seqs * p.Hkv;
  const int col = blockIdx.x / n_units;
  const int u = blockIdx.x - col * n_units;
  const int i = u / p.Hkv, h = u - i * p.Hkv;
  const int64_t T0 = p.ctr[i].total;
  const int64_t t_begin = (int64_t)col * p.dense_chunk;
  if (t_begin >= T0) return;
  const int n = T0 - t_begin < p.dense_chunk ? (int)(T0 - t_begin) : p.dense_chunk;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gid = lane >> 2, tig = lane & 3;
  const int b = p.seq_begin + i;
  const int64_t unit = (int64_t)b * p.Hkv + h;
  WarpState<D> st;
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) st.O[mt][0] = st.O[mt][1] = st.O[mt][2] = st.O[mt][3] = 0.f;
  st.C[0] = st.C[1] = st.C[2] = st.C[3] = 0.f;
  st.m0 = st.m1 = -INFINITY;
  st.l0 = st.l1 = 0.f;
  rows_mma<D, GP, 2, false>(p, reinterpret_cast<const __nv_bfloat16*>(p.dense_k) + unit * p.t_stride * D,
                            reinterpret_cast<const __nv_bfloat16*>(p.dense_v) + unit * p.t_stride * D, t_begin, 0,
                            n, reinterpret_cast<const __nv_bfloat16*>(p.q) + ((int64_t)b * p.Hq + h * p.g) * D, lane,
                            warp, gid, tig, smem + (size_t)warp * kRowsBuf<D, 2>, st);
  __syncthreads();  // every warp is done with its buffers: reuse them for the merge
  write_partial<D, GP>(p, unit, col, warp, gid, tig, st, smem);
}

template <int D>
size_t dense_smem() {
  const size_t rows = (size_t)kMmaWarps * kRowsBuf<D, 2>;
  const size_t merge = (size_t)kMmaWarps * kMaxGqa * (D + 2) * sizeof(float);
  return rows > merge ? rows : merge;
}

template <int D, int GP>
cudaError_t launch_dense_t(const DecodeParams& p, int cols, cudaStream_t s) {
  const size_t smem = dense_smem<D>();
  int dev = 0;
  cudaGetDevice(&dev);
  static size_t configured[64] = {};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (smem > configured[dev]) {
    const cudaError_t e =
        cudaFuncSetAttribute(decode_dense_kernel<D, GP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured[dev] = smem;
  }
  return launch_pdl(decode_dense_kernel<D, GP>, dim3(cols * p.n_seqs * p.Hkv), dim3(kMmaThreads), smem, s, p);
}

int gqa_pad(int g) { return g <= 2 ? 2 : g <= 4 ? 4 : 8; }

template <int D>
cudaError_t launch_dense_g(const DecodeParams& p, int cols, cudaStream_t s) {
  switch (gqa_pad(p.g)) {
    case 2: return launch_dense_t<D, 2>(p, cols, s);
    case 4: return launch_dense_t<D, 4>(p, cols, s);
    default: return launch_dense_t<D, 8>(p, cols, s);
  }
}

// Shared-memory page slots per warp: about 60 KB of pages per CTA, at least
// one group (8 / padded g pages) and at most 8.  Slots above 6 KB (8-bit
// codes) get one page beyond a group even though the CTA then needs more
// shared memory (2 CTAs per SM instead of 3): with one group's slots only,
// no copy is in flight while a group is computed (the 8-bit ragged decode:
// 171.5 -> 155.1 us).
int mma_slots(int64_t page_bytes, int g) {
  const int pb = 8 / gqa_pad(g);
  int slots = (int)(60 * 1024 / (kMmaWarps * page_bytes));
  if (slots < pb) slots = pb;
  if (page_bytes > 6144 && slots < pb + 1) slots = pb + 1;
  if (slots > 8) slots = 8;
  return slots;
}

constexpr size_t kMaxSmem = 227 * 1024;

// Bytes of one ring slot: a whole page at G = 32, else a 32-token unit (the
// layout of a G = 32 page).
int64_t unit_bytes(const DecodeParams& p) {
  return p.G == 32 ? p.geom.page_bytes : make_geom(32, p.D, p.bits).page_bytes;
}

template <int D>
size_t smem_for(const DecodeParams& p) {
  const int slots = mma_slots(unit_bytes(p), p.g);
  size_t pages = (size_t)kMmaWarps * slots * unit_bytes(p);
  // segmented tiles: each warp's slot marks (8 bytes) and CUDA-core weights
  if (p.seg.kcodes) pages += 32 + (size_t)kMmaWarps * 32 * gqa_pad(p.g) * sizeof(float);
  const size_t merge = (size_t)kMmaWarps * kMaxGqa * (D + 2) * sizeof(float);
  const size_t window = (size_t)kMmaWarps * kRowsBuf<D, 2>;
  if (pages < merge) pages = merge;
  if (pages < window) pages = window;
  const size_t scratch = ((size_t)kMmaWarps * (8 / gqa_pad(p.g)) * D + (size_t)gqa_pad(p.g) * D + 32) * sizeof(float);
  return 128 * ((kMmaWarps * slots * 8 + 127) / 128) + scratch + pages;
}

// Allows the split kernel instance ``smem`` bytes of dynamic shared memory
// on the current device (once per device and size).
template <int D, int BITS, int GP, int MODE>
cudaError_t configure_t(size_t smem) {
  int dev = 0;
  cudaGetDevice(&dev);
  static size_t configured[64] = {};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (smem > configured[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel<D, BITS, GP, MODE>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured[dev] = smem;
  }
  return cudaSuccess;
}

// CTAs of the split kernel one SM holds at once for these parameters (0 on
// error).  The answer depends only on the device and the shared memory size,
// so the last one is kept per device: the query costs more host time than a
// batch-1 decode takes on the GPU.
template <int D, int BITS, int GP, int MODE>
int resident_t(const DecodeParams& p) {
  const size_t smem = smem_for<D>(p);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  // (shared memory bytes << 8 | CTAs per SM), one word so that concurrent
  // callers never see one query's size with another's answer
  static std::atomic<uint64_t> known[64];
  const uint64_t k = known[dev].load(std::memory_order_relaxed);
  if ((k & 0xFFu) != 0 && (k >> 8) == (uint64_t)smem) return (int)(k & 0xFFu);
  int per_sm = 0;
  if (configure_t<D, BITS, GP, MODE>(smem) != cudaSuccess) return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_mma_kernel<D, BITS, GP, MODE>, kMmaThreads,
                                                    smem) != cudaSuccess)
    return 0;
  if (per_sm > 0 && per_sm < 256) known[dev].store((uint64_t)smem << 8 | (uint64_t)per_sm, std::memory_order_relaxed);
  return per_sm;
}

template <int D, int BITS>
int resident_g(const DecodeParams& p) {
  auto pick = [&](auto gp) {
    constexpr int GP = decltype(gp)::value;
    if constexpr (BITS == 4)
      if (p.seg.kcodes) return resident_t<D, BITS, GP, kSeg32>(p);
    if (p.G != 32) return resident_t<D, BITS, GP, kStaged>(p);
    return p.map.table ? resident_t<D, BITS, GP, kPaged32>(p) : resident_t<D, BITS, GP, kFlat32>(p);
  };
  switch (gqa_pad(p.g)) {
    case 2: return pick(std::integral_constant<int, 2>{});
    case 4: return pick(std::integral_constant<int, 4>{});
    default: return pick(std::integral_constant<int, 8>{});
  }
}

template <int D, int BITS, int GP, int MODE>
cudaError_t launch_t(const DecodeParams& p, cudaStream_t s) {
  const size_t smem = smem_for<D>(p);
  const cudaError_t e = configure_t<D, BITS, GP, MODE>(smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((p.grid_splits + 1) * p.n_seqs * p.Hkv);
  return launch_pdl(decode_mma_kernel<D, BITS, GP, MODE>, grid, dim3(kMmaThreads), smem, s, p,
                    mma_slots(unit_bytes(p), p.g));
}

template <int D, int BITS, int GP>
cudaError_t launch_m(const DecodeParams& p, cudaStream_t s) {
  if constexpr (BITS == 4)
    if (p.seg.kcodes) return launch_t<D, BITS, GP, kSeg32>(p, s);
  if (p.G != 32) return launch_t<D, BITS, GP, kStaged>(p, s);
  return p.map.table ? launch_t<D, BITS, GP, kPaged32>(p, s) : launch_t<D, BITS, GP, kFlat32>(p, s);
}

template <int D, int BITS>
cudaError_t launch_g(const DecodeParams& p, cudaStream_t s) {
  switch (gqa_pad(p.g)) {
    case 2: return launch_m<D, BITS, 2>(p, s);
    case 4: return launch_m<D, BITS, 4>(p, s);
    default: return launch_m<D, BITS, 8>(p, s);
  }
}

}  // namespace
}  // namespace kvq
