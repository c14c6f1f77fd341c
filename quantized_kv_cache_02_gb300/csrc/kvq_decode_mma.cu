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
// is not the code (q/sK as an f16 hi + lo pair, p/sV as one f16).  Codes are
// exact small integers in f16; the nibble to f16 conversion writes the biased
// nibble into the mantissa of 1024.0 and subtracts 1032.0 (IEEE binary16:
// 0x6400 | u == 1024 + u for u < 1024).
// Matrix shapes: S = A(K codes: 16 tokens x 16 channels) * B(q: 16 x 8 heads),
// O^T = A(V codes^T: 16 channels x 16 tokens) * B(P^T: 16 tokens x 8 heads);
// P goes from the S accumulator layout to the B layout with movmatrix.trans.
// Token and channel orders inside a k-step are permuted to match the packed
// byte layout; both operands of every MMA use the same permutation.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

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

__device__ __forceinline__ uint32_t f16x2_sub(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Eight signed nibbles of ``w`` -> four f16x2 registers; register j holds
// nibble j (low half) and nibble j + 4 (high half).  The lop3 builds
// 0x6400 | (nibble ^ 8) in each half: truth table 0x6A over
// (a = shifted word, b = 0x000F000F, c = 0x64086408) keeps a where b & ~c,
// inverts it where b & c (the nibble's top bit) and sets the bits of c
// outside b.  Subtracting 1032.0 leaves the signed value exactly.
__device__ __forceinline__ void nibbles_to_f16(uint32_t w, uint32_t (&r)[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t t;
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(t) : "r"(w >> (4 * j)), "r"(0x000F000Fu), "r"(0x64086408u));
    r[j] = f16x2_sub(t, 0x64086408u);
  }
}

// Four signed bytes of ``w`` -> two f16x2 registers: (byte0, byte1), (byte2, byte3).
__device__ __forceinline__ void bytes_to_f16(uint32_t w, uint32_t (&r)[2]) {
  const uint32_t t = w ^ 0x80808080u;
  uint32_t x0, x1;
  asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(x0) : "r"(t), "r"(0x64646464u));
  asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(x1) : "r"(t), "r"(0x64646464u));
  r[0] = f16x2_sub(x0, 0x64806480u);
  r[1] = f16x2_sub(x1, 0x64806480u);
}

template <int N>
__device__ __forceinline__ void lds_words(const uint8_t* p, uint32_t (&w)[N]) {
  static_assert(N % 2 == 0, "word count");
  if constexpr (N % 4 == 0) {
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

template <int D, int BITS>
struct Shape {
  static constexpr int kSteps = D / 16;        // k-steps of the S MMA, m-tiles of the O MMA
  static constexpr int kRowBytes = D * BITS / 8;
  static constexpr int kWords = kRowBytes / 16;  // 32-bit words of a K row per thread
  static constexpr int kChan = D / 4;          // channels of a K row per thread
  static constexpr int kSubBytes = 32 * D * BITS / 8;
};

// Channel (relative to the thread's slice) of element e (0..3) of k-step kk:
// e = 0, 1 -> B register 0 (k-slots 2tig, 2tig+1); e = 2, 3 -> register 1.
template <int BITS>
__device__ __forceinline__ int kslot_channel(int kk, int e) {
  if (BITS == 4) {
    const int base = 8 * (kk >> 1) + 2 * (kk & 1);
    const int off[4] = {0, 4, 1, 5};
    return base + off[e];
  } else {
    return 4 * kk + e;
  }
}

template <int D, int BITS>
struct WarpState {
  float O[D / 16][4];
  float m0, m1, l0, l1;
};

// One group page (G tokens) in shared memory.
template <int D, int BITS>
__device__ __forceinline__ void mma_page(const uint8_t* pg, const PageGeom& geom, int G, bool qlive,
                                         const float (&qreg)[Shape<D, BITS>::kChan], int gid, int tig,
                                         WarpState<D, BITS>& st) {
  using S = Shape<D, BITS>;
  // ---- B operand of S: q / sK per channel as an f16 pair hi + lo ---------
  // (hi = f16(x), lo = f16(x - hi)): two MMAs against the same code operand
  // give the scores to ~2^-22 relative instead of f16's 2^-12, which matters
  // because outlier channels make the softmax very peaked.
  uint32_t bq[S::kSteps][2], bl[S::kSteps][2];
  {
    const float* ks = reinterpret_cast<const float*>(pg + geom.kscale_off) + tig * S::kChan;
    float qk[S::kChan];
#pragma unroll
    for (int i = 0; i < S::kChan / 4; ++i) {
      const float4 s4 = reinterpret_cast<const float4*>(ks)[i];
      qk[4 * i + 0] = __fdividef(qreg[4 * i + 0], s4.x);
      qk[4 * i + 1] = __fdividef(qreg[4 * i + 1], s4.y);
      qk[4 * i + 2] = __fdividef(qreg[4 * i + 2], s4.z);
      qk[4 * i + 3] = __fdividef(qreg[4 * i + 3], s4.w);
    }
#pragma unroll
    for (int kk = 0; kk < S::kSteps; ++kk) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float x0 = qk[kslot_channel<BITS>(kk, 2 * r)], x1 = qk[kslot_channel<BITS>(kk, 2 * r + 1)];
        const __half2 hi = __floats2half2_rn(x0, x1);
        const float2 back = __half22float2(hi);
        const __half2 lo = __floats2half2_rn(x0 - back.x, x1 - back.y);
        bq[kk][r] = qlive ? *reinterpret_cast<const uint32_t*>(&hi) : 0u;
        bl[kk][r] = qlive ? *reinterpret_cast<const uint32_t*>(&lo) : 0u;
      }
    }
  }
  const float* vscale = reinterpret_cast<const float*>(pg + geom.vscale_off);
  const int r_base = 8 * (gid >> 1) + (gid & 1);  // token row of m-block 0 inside a sub-tile

  for (int sub = 0; sub < G / 32; ++sub) {
    const uint8_t* kc = pg + sub * 32 * S::kRowBytes;
    const uint8_t* vc = pg + geom.code_bytes + sub * S::kSubBytes;
    // ---- S = K q for the two 16-token m-blocks --------------------------
    float s[2][4];
    {
      uint32_t wa[2][S::kWords], wb[2][S::kWords];
#pragma unroll
      for (int mb = 0; mb < 2; ++mb) {
        const int r0 = r_base + 4 * mb;
        lds_words<S::kWords>(kc + r0 * S::kRowBytes + tig * (S::kRowBytes / 4), wa[mb]);
        lds_words<S::kWords>(kc + (r0 + 2) * S::kRowBytes + tig * (S::kRowBytes / 4), wb[mb]);
        s[mb][0] = s[mb][1] = s[mb][2] = s[mb][3] = 0.f;
      }
      if (BITS == 4) {
#pragma unroll
        for (int i = 0; i < S::kWords; ++i) {
#pragma unroll
          for (int mb = 0; mb < 2; ++mb) {
            uint32_t ra[4], rb[4];
            nibbles_to_f16(wa[mb][i], ra);
            nibbles_to_f16(wb[mb][i], rb);
            mma16816(s[mb], ra[0], rb[0], ra[1], rb[1], bq[2 * i][0], bq[2 * i][1]);
            mma16816(s[mb], ra[0], rb[0], ra[1], rb[1], bl[2 * i][0], bl[2 * i][1]);
            mma16816(s[mb], ra[2], rb[2], ra[3], rb[3], bq[2 * i + 1][0], bq[2 * i + 1][1]);
            mma16816(s[mb], ra[2], rb[2], ra[3], rb[3], bl[2 * i + 1][0], bl[2 * i + 1][1]);
          }
        }
      } else {
#pragma unroll
        for (int kk = 0; kk < S::kWords; ++kk) {
#pragma unroll
          for (int mb = 0; mb < 2; ++mb) {
            uint32_t ra[2], rb[2];
            bytes_to_f16(wa[mb][kk], ra);
            bytes_to_f16(wb[mb][kk], rb);
            mma16816(s[mb], ra[0], rb[0], ra[1], rb[1], bq[kk][0], bq[kk][1]);
            mma16816(s[mb], ra[0], rb[0], ra[1], rb[1], bl[kk][0], bl[kk][1]);
          }
        }
      }
    }
    // ---- online softmax (base 2) over the 32 tokens -----------------------
    float mx0 = fmaxf(fmaxf(s[0][0], s[0][2]), fmaxf(s[1][0], s[1][2]));
    float mx1 = fmaxf(fmaxf(s[0][1], s[0][3]), fmaxf(s[1][1], s[1][3]));
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float mn0 = fmaxf(st.m0, mx0), mn1 = fmaxf(st.m1, mx1);
    const float a0 = fast_exp2(st.m0 - mn0), a1 = fast_exp2(st.m1 - mn1);
    st.m0 = mn0;
    st.m1 = mn1;
    float pr[2][4];
#pragma unroll
    for (int mb = 0; mb < 2; ++mb) {
      pr[mb][0] = fast_exp2(s[mb][0] - mn0);
      pr[mb][1] = fast_exp2(s[mb][1] - mn1);
      pr[mb][2] = fast_exp2(s[mb][2] - mn0);
      pr[mb][3] = fast_exp2(s[mb][3] - mn1);
    }
    st.l0 = fmaf(st.l0, a0, (pr[0][0] + pr[0][2]) + (pr[1][0] + pr[1][2]));
    st.l1 = fmaf(st.l1, a1, (pr[0][1] + pr[0][3]) + (pr[1][1] + pr[1][3]));
    if (__any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
      for (int mt = 0; mt < S::kSteps; ++mt) {
        st.O[mt][0] *= a0;
        st.O[mt][1] *= a1;
        st.O[mt][2] *= a0;
        st.O[mt][3] *= a1;
      }
    }
    // ---- B operand of O: p / sV per token, transposed to the B layout ------
    uint32_t bp[2][2];
#pragma unroll
    for (int mb = 0; mb < 2; ++mb) {
      const int r0 = sub * 32 + r_base + 4 * mb;
      const float v0 = vscale[r0], v1 = vscale[r0 + 2];
      bp[mb][0] = transpose8x8(pack_f16x2(__fdividef(pr[mb][0], v0), __fdividef(pr[mb][1], v0)));
      bp[mb][1] = transpose8x8(pack_f16x2(__fdividef(pr[mb][2], v1), __fdividef(pr[mb][3], v1)));
    }
    // ---- O^T += V^T P ------------------------------------------------------
#pragma unroll
    for (int mt = 0; mt < S::kSteps; ++mt) {
      const int c_lo = 16 * mt + gid, c_hi = c_lo + 8;
      if (BITS == 4) {
        const uint32_t wl = *reinterpret_cast<const uint32_t*>(vc + c_lo * 16 + 4 * tig);
        const uint32_t wh = *reinterpret_cast<const uint32_t*>(vc + c_hi * 16 + 4 * tig);
        uint32_t rl[4], rh[4];
        nibbles_to_f16(wl, rl);
        nibbles_to_f16(wh, rh);
        mma16816(st.O[mt], rl[0], rh[0], rl[1], rh[1], bp[0][0], bp[0][1]);
        mma16816(st.O[mt], rl[2], rh[2], rl[3], rh[3], bp[1][0], bp[1][1]);
      } else {
        const uint2 vl = *reinterpret_cast<const uint2*>(vc + c_lo * 32 + 8 * tig);
        const uint2 vh = *reinterpret_cast<const uint2*>(vc + c_hi * 32 + 8 * tig);
        uint32_t rl[2], rh[2];
        bytes_to_f16(vl.x, rl);
        bytes_to_f16(vh.x, rh);
        mma16816(st.O[mt], rl[0], rh[0], rl[1], rh[1], bp[0][0], bp[0][1]);
        bytes_to_f16(vl.y, rl);
        bytes_to_f16(vh.y, rh);
        mma16816(st.O[mt], rl[0], rh[0], rl[1], rh[1], bp[1][0], bp[1][1]);
      }
    }
  }
}

template <int D, int BITS>
__global__ void __launch_bounds__(kMmaThreads) decode_mma_kernel(const DecodeParams p, int slots) {
  using S = Shape<D, BITS>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int u = blockIdx.y;
  const int i = u / p.Hkv, h = u - i * p.Hkv;
  bool win;
  int pg0, pg1, slot;
  if (!split_item(p, blockIdx.x, i, &win, &pg0, &pg1, &slot)) return;
  if (win) {
    simt_item<__nv_bfloat16, BITS, D / 32>(p, i, h, true, 0, 0, slot, reinterpret_cast<float*>(smem));
    return;
  }

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gid = lane >> 2, tig = lane & 3;
  const int b = p.seq_begin + i;
  const int g = p.g;
  const PageGeom geom = p.geom;
  const uint32_t page_bytes = (uint32_t)geom.page_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint8_t* buf = smem + ((kMmaWarps * slots * 8 + 127) / 128) * 128;
  uint8_t* my_buf = buf + (size_t)warp * slots * page_bytes;
  const uint32_t my_bar = smem_addr(bars + warp * slots);

  // this thread's query slice (head gid, channels tig*D/4 ...), pre-scaled
  const bool qlive = gid < g;
  float qreg[S::kChan];
  {
    const __nv_bfloat16* q = reinterpret_cast<const __nv_bfloat16*>(p.q) +
                             ((int64_t)b * p.Hq + (int64_t)h * g + (qlive ? gid : 0)) * D + tig * S::kChan;
#pragma unroll
    for (int c = 0; c < S::kChan; ++c) qreg[c] = qlive ? __bfloat162float(q[c]) * p.qk_scale : 0.f;
  }

  const uint8_t* unit_pages = p.pages + p.layout[b].page_base + h * p.layout[b].unit_stride;
  const int npg = pg1 - pg0;
  const int my_n = warp < npg ? (npg - warp + kMmaWarps - 1) / kMmaWarps : 0;
  if (lane == 0) {
    for (int s = 0; s < slots; ++s) mbar_init(my_bar + 8 * s, 1);
    fence_mbar_init();
    fence_proxy_async();
    for (int s = 0; s < slots && s < my_n; ++s) {
      mbar_expect_tx(my_bar + 8 * s, page_bytes);
      bulk_load(smem_addr(my_buf + (size_t)s * page_bytes),
                unit_pages + (int64_t)(pg0 + warp + s * kMmaWarps) * page_bytes, page_bytes, my_bar + 8 * s);
    }
  }
  __syncwarp();

  WarpState<D, BITS> st;
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) st.O[mt][0] = st.O[mt][1] = st.O[mt][2] = st.O[mt][3] = 0.f;
  st.m0 = st.m1 = -INFINITY;
  st.l0 = st.l1 = 0.f;

  int k = 0;
  bool ok = true;
  for (; k < my_n; ++k) {
    const int s = k % slots;
    if (!mbar_wait(my_bar + 8 * s, (uint32_t)((k / slots) & 1))) {
      ok = false;
      break;
    }
    mma_page<D, BITS>(my_buf + (size_t)s * page_bytes, geom, p.G, qlive, qreg, gid, tig, st);
    __syncwarp();
    if (lane == 0 && k + slots < my_n) {
      fence_proxy_async();
      mbar_expect_tx(my_bar + 8 * s, page_bytes);
      bulk_load(smem_addr(my_buf + (size_t)s * page_bytes),
                unit_pages + (int64_t)(pg0 + warp + (k + slots) * kMmaWarps) * page_bytes, page_bytes,
                my_bar + 8 * s);
    }
  }
  if (!ok) {
    // drain the copies still in flight (bounded), report, and contribute nothing
    const int issued = min(my_n, k + slots);
    for (int kk = k; kk < issued; ++kk) mbar_wait(my_bar + 8 * (kk % slots), (uint32_t)((kk / slots) & 1));
    if (lane == 0) atomicOr(p.status, kStatusWaitTimeout);
    st.m0 = st.m1 = -INFINITY;
    st.l0 = st.l1 = 0.f;
  }
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    st.l0 += __shfl_xor_sync(0xffffffffu, st.l0, off);
    st.l1 += __shfl_xor_sync(0xffffffffu, st.l1, off);
  }
  __syncthreads();  // every warp is done with its slots: reuse them for the merge

  float* mrg = reinterpret_cast<float*>(buf);  // [kMmaWarps][kMaxGqa][D + 2]
  const int hd0 = 2 * tig, hd1 = 2 * tig + 1;
  float* mw = mrg + (size_t)warp * kMaxGqa * (D + 2);
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) {
    const int c_lo = 16 * mt + gid;
    if (hd0 < g) {
      mw[hd0 * (D + 2) + c_lo] = ok ? st.O[mt][0] : 0.f;
      mw[hd0 * (D + 2) + c_lo + 8] = ok ? st.O[mt][2] : 0.f;
    }
    if (hd1 < g) {
      mw[hd1 * (D + 2) + c_lo] = ok ? st.O[mt][1] : 0.f;
      mw[hd1 * (D + 2) + c_lo + 8] = ok ? st.O[mt][3] : 0.f;
    }
  }
  if (gid == 0) {
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
  const int64_t unit = (int64_t)b * p.Hkv + h;
  float* part = p.partials + (unit * p.max_splits + slot) * (int64_t)g * (D + 2);
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
    part[(int64_t)j * (D + 2) + c] = O;
    if (c == 0) {
      part[(int64_t)j * (D + 2) + D] = M;
      part[(int64_t)j * (D + 2) + D + 1] = L;
    }
  }
}

int mma_slots(int64_t page_bytes) {
  int slots = (int)(80 * 1024 / (kMmaWarps * page_bytes));
  if (slots < 2) slots = 2;
  if (slots > 6) slots = 6;
  return slots;
}

template <int D>
size_t smem_for(const DecodeParams& p) {
  const int slots = mma_slots(p.geom.page_bytes);
  size_t pages = (size_t)kMmaWarps * slots * p.geom.page_bytes;
  const size_t merge = (size_t)kMmaWarps * kMaxGqa * (D + 2) * sizeof(float);
  const size_t simt = (size_t)simt_scratch_floats<D / 32>() * sizeof(float);
  if (pages < merge) pages = merge;
  if (pages < simt) pages = simt;
  return ((kMmaWarps * slots * 8 + 127) / 128) * 128 + pages;
}

template <int D, int BITS>
cudaError_t launch_t(const DecodeParams& p, cudaStream_t s) {
  const size_t smem = smem_for<D>(p);
  static size_t configured = 0;
  if (smem > configured) {
    const cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel<D, BITS>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  const dim3 grid(p.grid_splits + 1, p.n_seqs * p.Hkv);
  decode_mma_kernel<D, BITS><<<grid, kMmaThreads, smem, s>>>(p, mma_slots(p.geom.page_bytes));
  return cudaGetLastError();
}

}  // namespace

size_t decode_mma_smem_bytes(const DecodeParams& p) {
  return p.D == 64 ? smem_for<64>(p) : smem_for<128>(p);
}

cudaError_t launch_decode_mma(const DecodeParams& p, cudaStream_t s, int* supported) {
  *supported = (p.D == 64 || p.D == 128) && (p.G % 32 == 0) && p.g <= kMaxGqa;
  if (!*supported) return cudaSuccess;
  if (p.D == 64) return p.bits == 4 ? launch_t<64, 4>(p, s) : launch_t<64, 8>(p, s);
  return p.bits == 4 ? launch_t<128, 4>(p, s) : launch_t<128, 8>(p, s);
}

}  // namespace kvq
