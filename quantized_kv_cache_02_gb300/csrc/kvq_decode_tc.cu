// Fifth-generation tensor-core (tcgen05) split kernel of the decode attention
// for head_dim 128 and 4-bit codes.
//
// Same work items, inputs and partial format as decode_mma_kernel; the
// residual-window items still run window_rows.  A page item is taken in blocks
// of four 32-token units (128 tokens): one row of the 128 TMEM lanes per token
// for the scores, one per channel for the output.
//
//   S[t][n] = sum_k A_K[t][k] B_Q[k][n]      (M = 128 tokens, N = 4 units x (hi, lo) x GP heads)
//   O^T[c][h] += sum_t A_V[c][t] B_P[t][h]   (M = 128 channels, N = 16)
//
// A_K (Key codes, one token per lane) and A_V (Value codes, one channel per
// lane) are cut out of the stored words as f16 subnormals (code + 8) * 2^-24
// exactly as in decode_mma_kernel and written to tensor memory with
// tcgen05.st; B_Q = q / sK as f16 hi and lo rows and B_P = p / sV as f16 sit in
// shared memory (K-major, no swizzle: 8-row x 16-byte core matrices, LBO the
// step along K, SBO the step along N).  The offset bias is taken out on the CUDA
// cores: 8 * sum_c q / sK per unit and head for the scores, and for the output
// 8 times the sum of exactly the f16 values B_P held.  One thread issues every
// MMA; completion is signalled through tcgen05.commit on mbarriers.  Softmax
// (base 2, the same lazy running max as decode_mma_kernel, shared by the whole
// CTA) runs one token per thread on the scores read back with tcgen05.ld.
// ("KV Cache Quantization Strategies", restore; "KV Cache 与自回归视频生成"
// 3.1, attn_step and section 05, FlashDecoding.)

#include "kvq_decode_mma.cuh"

namespace kvq {
namespace {

// ---- tcgen05 PTX -----------------------------------------------------------
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
// D (tmem) (+)= A (tmem) * B (smem descriptor)
__device__ __forceinline__ void tc_mma(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tc_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
// N consecutive 32-bit columns of this thread's lane
template <int N>
__device__ __forceinline__ void tc_ld(uint32_t taddr, float (&v)[N]);
template <>
__device__ __forceinline__ void tc_ld<2>(uint32_t taddr, float (&v)[2]) {
  uint32_t r[2];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0,%1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(taddr) : "memory");
  v[0] = __uint_as_float(r[0]);
  v[1] = __uint_as_float(r[1]);
}
template <>
__device__ __forceinline__ void tc_ld<4>(uint32_t taddr, float (&v)[4]) {
  uint32_t r[4];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr)
               : "memory");
#pragma unroll
  for (int j = 0; j < 4; ++j) v[j] = __uint_as_float(r[j]);
}
template <>
__device__ __forceinline__ void tc_ld<8>(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = __uint_as_float(r[j]);
}
template <int N>
__device__ __forceinline__ void tc_st_f(uint32_t taddr, const float (&v)[N]) {
  if constexpr (N == 2) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1,%2};" ::"r"(taddr), "r"(__float_as_uint(v[0])),
                 "r"(__float_as_uint(v[1]))
                 : "memory");
  } else if constexpr (N == 4) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr),
                 "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
                 "r"(__float_as_uint(v[3]))
                 : "memory");
  } else {
    uint32_t r[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) r[j] = __float_as_uint(v[j]);
    tc_st8(taddr, r);
  }
}

// Shared-memory matrix descriptor: K-major, no swizzle (version 1 at bit 46).
__device__ __forceinline__ uint64_t tc_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46);
}
// Instruction descriptor of kind::f16: f32 D, f16 A and B, both K-major.
__host__ __device__ constexpr uint32_t tc_idesc(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ---- layout ---------------------------------------------------------------
constexpr int kTcD = 128;
constexpr int kTcGroup = 128;                        // threads of one worker group (4 warps)
constexpr int kTcThreads = 2 * kTcGroup + 64;        // Key warps 0-3, Value warps 4-7, MMA warp 8, copy warp 9
constexpr int kTcMmaWarp = 8, kTcCopyWarp = 9;
constexpr int kTcUnit = 32 * kTcD / 2 * 2 + 4 * kTcD + 4 * 32;  // a G = 32 page: 4736 bytes
constexpr int kTcUnitStride = kTcUnit + 16;  // units staggered by 16 bytes across the banks
constexpr int kTcKsc = 2 * 32 * kTcD / 2;    // Key scales within a unit
constexpr int kTcVsc = kTcKsc + 4 * kTcD;    // Value scales
constexpr int kTcVcode = 32 * kTcD / 2;      // Value codes
constexpr int kTcSlots = 4;                  // blocks of 4 units in flight
constexpr int kTcBlock = 4 * kTcUnitStride;
constexpr int kTcBRow = 2 * kTcD;            // bytes of one B row (K = 128 f16)
constexpr uint32_t kTcSbo = 16 * 128;        // next 8-row group: 16 core matrices along K

template <int GP>
struct TcShape {
  static constexpr int NS = 8 * GP;   // score columns: 4 units x (hi, lo) x GP heads
  static constexpr int CPG = GP / 2;  // heads of one unit per B_Q-building thread
  // tensor memory: A_K, A_V, scores (two buffers), output accumulator
  static constexpr uint32_t kColAK = 0, kColAV = 64, kColS0 = 128, kColS1 = kColS0 + NS, kColO = kColS1 + NS;
  static constexpr uint32_t kCols = kColO + 16 <= 256 ? 256 : 512;
  static constexpr size_t kBOff = ((size_t)kTcSlots * kTcBlock + 1023) / 1024 * 1024;  // B operands
  static constexpr size_t kBq = (size_t)NS * kTcBRow;                                  // one B_Q buffer
  static constexpr size_t smem =
      kBOff + 2 * kBq + 16 * kTcBRow + GP * kTcD * 4 + (96 + 3 * 4 * 8 + 8 + 3 * 4 + 2) * 4 + (2 * kTcSlots + 5) * 8 + 32;
};

template <uint32_t N>
__device__ __forceinline__ void tc_alloc_n(uint32_t dst_smem) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "n"(N) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
template <uint32_t N>
__device__ __forceinline__ void tc_dealloc_n(uint32_t taddr) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "n"(N) : "memory");
}

// Byte offset of element (n, k) of a K-major B matrix with K = 128.
__device__ __forceinline__ int b_off(int n, int k) {
  return (n >> 3) * kTcSbo + (k >> 3) * 128 + (n & 7) * 16 + (k & 7) * 2;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// barrier 1 over the four Key warps, with an OR of ``pred``
__device__ __forceinline__ bool kgroup_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, %2, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred), "n"(kTcGroup)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void kgroup_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kTcGroup) : "memory"); }

// Bounded wait; a warp that only issues copies or MMAs backs off with
// __nanosleep between tries (``sleep_ns``).  It also gives up as soon as
// ``*abort`` is set (another part of the CTA stopped and will not complete
// the phase).  About a second in all.
constexpr uint32_t kTcWaitTries = 1u << 22;
template <int sleep_ns = 0>
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, const volatile int* abort) {
  for (uint32_t it = 0; it < kTcWaitTries; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
    if (*abort) return false;
    if (sleep_ns > 0) __nanosleep(sleep_ns);
  }
  return false;
}
__device__ const int kNoAbort = 0;  // for waits that must not be cut short

// Range of the f16 operands (as in decode_mma_kernel, 4-bit codes).  The
// smallest Key scale for which a unit keeps biased codes and an unscaled
// B_Q: |q / sK| <= 2^9.  ``qred`` holds the largest |q * qk_scale| of each
// of the 8 warps that filled the queries.
__device__ __forceinline__ float tc_kthr(const float* qred, float eps, int* qexp) {
  float qa = qred[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) qa = fmaxf(qa, qred[w]);
  *qexp = float_exp2i(qa);
  const int e = *qexp + 1 - 9;
  return fmaxf(e < -126 ? 0.f : e > 127 ? INFINITY : __uint_as_float((uint32_t)(e + 127) << 23), eps);
}
// Whether block ``sb`` of up to four units has a token whose Value absmax
// (qmax / sV) exceeds kVWideAbs: its output terms are then summed in fp32
// (every Key warp decides alike).
__device__ __forceinline__ bool tc_value_wide(const uint8_t* sb, int nu, int lane, int vsc_off, int unit_stride,
                                              float vwide) {
  bool w = false;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (j < nu) w |= fast_rcp(reinterpret_cast<const float*>(sb + j * unit_stride + vsc_off)[lane]) > vwide;
  return __any_sync(0xffffffffu, w);
}

// Every mbarrier of the CTA completes once per block.  A thread arrives on a
// barrier for block b + 1 only after it has seen block b's phase complete, and
// it waits on a phase only while no later phase can complete without its own
// later arrival, so no phase is ever miscounted or mistaken for another.
template <int GP, int MODE>
__global__ void __launch_bounds__(kTcThreads, 2) decode_tc_kernel(const DecodeParams p) {
  constexpr int D = kTcD;
  using TS = TcShape<GP>;
  constexpr int NS = TS::NS, CPG = TS::CPG;
  extern __shared__ __align__(1024) uint8_t tc_smem[];
  pdl_wait();
  pdl_release();
  const int n_units = p.n_seqs * p.Hkv;
  const int col = blockIdx.x / n_units;
  const int u = blockIdx.x - col * n_units;
  const int i = u / p.Hkv, h = u - i * p.Hkv;
  bool win;
  int pg0, pg1, slot;
  if (!split_item(p, col, i, &win, &pg0, &pg1, &slot)) return;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int b = p.seq_begin + i;
  const int64_t unit = (int64_t)b * p.Hkv + h;

  if (win) {
    // the window runs on the four Key warps; the other warps only join the merge
    WarpState<D> st;
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) st.O[mt][0] = st.O[mt][1] = st.O[mt][2] = st.O[mt][3] = 0.f;
    st.C[0] = st.C[1] = st.C[2] = st.C[3] = 0.f;
    st.m0 = st.m1 = -INFINITY;
    st.l0 = st.l1 = 0.f;
    if (warp < 4) window_rows<D, GP>(p, i, h, lane, warp, lane >> 2, lane & 3, tc_smem, st);
    __syncthreads();
    write_partial<D, GP>(p, unit, slot, warp, lane >> 2, lane & 3, st, tc_smem);
    return;
  }

  // ---- shared memory ----------------------------------------------------------
  uint8_t* ring = tc_smem;
  uint8_t* bq = tc_smem + TS::kBOff;          // B_Q, two buffers of NS rows
  uint8_t* bpm = bq + 2 * TS::kBq;         // B_P: 16 rows
  float* qs = reinterpret_cast<float*>(bpm + 16 * kTcBRow);
  float* red = qs + GP * D;                // [0, 32): maxima; [32, 64): l; [64, 96): Value bias sums
  float* beta = red + 96;                  // [3][4 units][8 heads] Key bias sums
  float* qred = beta + 3 * 4 * 8;          // [8]: largest |q| seen by each filling warp
  float* kback = qred + 8;                 // [3][4 units]: 2^F taken out of the unit's B_Q
  int* vflag = reinterpret_cast<int*>(kback + 3 * 4);  // [2]: block (by parity) is wide (no output MMAs)
  uint64_t* bars = reinterpret_cast<uint64_t*>(vflag + 2);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2 * kTcSlots + 5);
  volatile int* abort = reinterpret_cast<volatile int*>(tslot + 1);  // set by whichever part stops
  // ring slots: ``full`` (copies landed) and ``empty`` (every worker is done with it)
  const uint32_t bar_ring = smem_addr(bars), bar_empty = bar_ring + 8 * kTcSlots;
  // A: A_K and B_Q of a block ready (both groups); P: A_V and B_P ready (both
  // groups); S[2]: the score MMAs of even / odd blocks done; O: the block's
  // output MMAs done
  const uint32_t bar_a = bar_empty + 8 * kTcSlots, bar_p = bar_a + 8, bar_s = bar_p + 8, bar_o = bar_s + 16;

  // ---- set-up -------------------------------------------------------------------
  if (warp == kTcMmaWarp) tc_alloc_n<TS::kCols>(smem_addr(tslot));
  if (t == 0) {
    *abort = 0;
    for (int s = 0; s < kTcSlots; ++s) {
      mbar_init(bar_ring + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_a, 2 * kTcGroup);
    mbar_init(bar_p, 2 * kTcGroup);
    mbar_init(bar_s, 1);
    mbar_init(bar_s + 8, 1);
    mbar_init(bar_o, 1);
    fence_mbar_init();
  }
  if (t < 2 * kTcGroup) {
    // queries (head n % g for the padding heads), pre-scaled
    float qa = 0.f;
    for (int idx = t; idx < GP * D; idx += 2 * kTcGroup) {
      const int n = idx / D, c = idx - n * D;
      qs[idx] = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(
                    p.q)[((int64_t)b * p.Hq + (int64_t)h * p.g + n % p.g) * D + c]) *
                p.qk_scale;
      qa = fmaxf(qa, fabsf(qs[idx]));
    }
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) qa = fmaxf(qa, __shfl_xor_sync(0xffffffffu, qa, off));
    if (lane == 0) qred[warp] = qa;
    // B operands start at zero (B_P rows GP..15 stay zero)
    for (int idx = t; idx < (int)((2 * TS::kBq + 16 * kTcBRow) / 16); idx += 2 * kTcGroup)
      reinterpret_cast<uint4*>(bq)[idx] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tslot;

  const PageGeom geom = p.geom;
  const int upp = MODE == kStaged ? p.G / 32 : 1;
  const int64_t stored = geom.page_bytes;
  const int nunits = (pg1 - pg0) * upp;
  const int nblk = (nunits + 3) / 4;
  constexpr float kTwo24 = 16777216.f, kSlack = 8.f;
  // TMEM lanes of this warp's quarter
  const uint32_t lane_base = tm + ((uint32_t)(32 * (warp & 3)) << 16);

  if (warp == kTcCopyWarp) {
    // ================= copy warp (lane 0): blocks of four units into the ring =======
    if (lane == 0) {
      const uint8_t* flat_base = MODE == kFlat32 ? p.pages + page_offset(p.map, stored, b, h, 0) : nullptr;
      auto page_ptr = [&](int pg) -> const uint8_t* {
        return MODE == kFlat32 ? flat_base + (int64_t)pg * stored : p.pages + page_offset(p.map, stored, b, h, pg);
      };
      auto issue = [&](int blk) {
        const int s = blk % kTcSlots;
        const int nu = min(4, nunits - 4 * blk);
        const uint32_t bar = bar_ring + 8 * s;
        mbar_expect_tx(bar, (uint32_t)(nu * kTcUnit));
        for (int j = 0; j < nu; ++j) {
          const uint32_t dst = smem_addr(ring + s * kTcBlock + j * kTcUnitStride);
          const int uu = pg0 * upp + 4 * blk + j;
          if constexpr (MODE != kStaged) {
            bulk_load(dst, page_ptr(uu), kTcUnit, bar);
          } else {
            constexpr int kRow = D / 2, kSub = 32 * D / 2;
            const int pg = uu / upp, sub = uu - pg * upp;
            const uint8_t* src = page_ptr(pg);
            bulk_load(dst, src + sub * 32 * kRow, 32 * kRow, bar);
            bulk_load(dst + kTcVcode, src + geom.code_bytes + sub * kSub, kSub, bar);
            bulk_load(dst + kTcKsc, src + geom.kscale_off, 4 * D, bar);
            bulk_load(dst + kTcVsc, src + geom.vscale_off + 128 * sub, 128, bar);
          }
        }
      };
      int issued = min(kTcSlots, nblk);
      fence_proxy_async();
      for (int k = 0; k < issued; ++k) issue(k);
      for (; issued < nblk; ++issued) {
        // the slot's previous block (issued - kTcSlots) has been read by every worker
        const int s = issued % kTcSlots;
        if (!wait_or_abort<256>(bar_empty + 8 * s, (uint32_t)(issued / kTcSlots - 1) & 1u, abort)) {
          *abort = 1;
          break;
        }
        fence_proxy_async();
        issue(issued);
      }
      // nothing in flight when the CTA ends
      for (int k = max(0, issued - kTcSlots); k < issued; ++k)
        wait_or_abort<256>(bar_ring + 8 * (k % kTcSlots), (uint32_t)(k / kTcSlots) & 1u, &kNoAbort);
    }
  } else if (warp == kTcMmaWarp) {
    // ================= MMA warp (lane 0) =====================================
    if (lane == 0) {
      const uint32_t idesc_s = tc_idesc(128, NS), idesc_o = tc_idesc(128, 16);
      const uint64_t dq0 = tc_desc(smem_addr(bq), 128, kTcSbo);
      const uint64_t dq1 = tc_desc(smem_addr(bq + TS::kBq), 128, kTcSbo);
      const uint64_t dp = tc_desc(smem_addr(bpm), 128, kTcSbo);
      int n_s = 0, n_o = 0;
      // the score MMAs of block k, into score buffer k & 1
      auto scores = [&](int k) -> bool {
        if (!wait_or_abort<32>(bar_a, (uint32_t)k & 1u, abort)) return false;
        tc_fence_after();
        const uint64_t dq = (k & 1) ? dq1 : dq0;
        const uint32_t d = tm + ((k & 1) ? TS::kColS1 : TS::kColS0);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)  // the B start advances by 256 bytes (two core matrices) per k-step
          tc_mma(d, tm + TS::kColAK + 8 * ks, dq + 16 * ks, idesc_s, ks > 0 ? 1u : 0u);
        tc_commit(bar_s + 8 * (k & 1));
        ++n_s;
        return true;
      };
      bool go = scores(0);
      for (int blk = 0; blk < nblk && go; ++blk) {
        // the next block's scores run while the workers finish this block's softmax
        if (blk + 1 < nblk && !scores(blk + 1)) {
          go = false;
          break;
        }
        if (!wait_or_abort<32>(bar_p, (uint32_t)blk & 1u, abort)) {
          *abort = 1;
          break;
        }
        mbar_arrive(bar_empty + 8 * (blk % kTcSlots));  // the copy warp may refill this block's slot
        tc_fence_after();
        // a wide block's output terms are added by the Key warps in fp32;
        // O starts at zero (the Key warps clear it before block 0)
        if (vflag[blk & 1] == 0) {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            tc_mma(tm + TS::kColO, tm + TS::kColAV + 8 * ks, dp + 16 * ks, idesc_o, 1u);
        }
        tc_commit(bar_o);
        ++n_o;
      }
      if (!go) *abort = 1;
      // nothing in flight when the CTA ends (the last score commit's completion
      // implies every earlier MMA's)
      if (n_s > 0)
        wait_or_abort<32>(bar_s + 8 * ((n_s - 1) & 1), (uint32_t)((n_s - 1) >> 1) & 1u, &kNoAbort);
      if (n_o > 0) wait_or_abort<32>(bar_o, (uint32_t)(n_o - 1) & 1u, &kNoAbort);
    }
  } else if (warp >= 4) {
    // ================= Value warps: A_V (one channel per thread), B_Q and the
    // Key bias sums of unit ``vw`` ============================================
    const int vw = warp - 4, c = t - kTcGroup;
    const int oct = lane >> 1, e0 = (lane & 1) * CPG;
    // range of q / sK (as in decode_mma_kernel): the plain path needs every
    // Key scale of the unit >= kthr; otherwise the unit's B_Q carries 2^-F
    int qexp;
    const float kthr = tc_kthr(qred, p.eps, &qexp);
    float qreg[CPG][8];
#pragma unroll
    for (int e = 0; e < CPG; ++e)
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        // k-slot kk of the octet holds channel 8 oct + kk/2 + 4 (kk % 2); the
        // slots whose codes carry x16 get 1/16 here
        const int ch = 8 * oct + (kk >> 1) + 4 * (kk & 1);
        qreg[e][kk] = qs[(e0 + e) * D + ch] * (((kk >> 1) & 1) ? 0.0625f : 1.f);
      }
    bool fail = false;
    // B_Q rows of unit vw for block blk (hi: vw * 2GP + e; lo: + GP) and the
    // unit's Key bias sums, then the arrival on A
    auto b_build = [&](int blk) {
      const int s = blk % kTcSlots;
      const int nu = min(4, nunits - 4 * blk);
      const uint8_t* sb = ring + s * kTcBlock;
      fail |= !wait_or_abort(bar_ring + 8 * s, (uint32_t)(blk / kTcSlots) & 1u, abort);
      uint8_t* bqb = bq + (blk & 1) * TS::kBq;
      if (vw < nu) {
        const float4* ks4 = reinterpret_cast<const float4*>(sb + vw * kTcUnitStride + kTcKsc) + 2 * oct;
        float4 s0 = ks4[0], s1 = ks4[1];
        const float smin = fminf(fminf(fminf(s0.x, s0.y), fminf(s0.z, s0.w)), fminf(fminf(s1.x, s1.y), fminf(s1.z, s1.w)));
        float fs = 1.f, fb = 1.f;
        const bool wide = __any_sync(0xffffffffu, smin < kthr);
        if (wide) {
          // scales below eps divide by eps; 2^-F keeps every B element below 2^14
          float m = fmaxf(smin, p.eps);
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) m = fminf(m, __shfl_xor_sync(0xffffffffu, m, off));
          const int F = min(kMaxRangeShift, max(0, qexp + 1 + 4 - float_exp2i(m) + 1 - 14));
          fs = pow2_neg(F);
          fb = __uint_as_float((uint32_t)(127 + F) << 23);
          s0 = make_float4(fmaxf(s0.x, p.eps), fmaxf(s0.y, p.eps), fmaxf(s0.z, p.eps), fmaxf(s0.w, p.eps));
          s1 = make_float4(fmaxf(s1.x, p.eps), fmaxf(s1.y, p.eps), fmaxf(s1.z, p.eps), fmaxf(s1.w, p.eps));
        }
        if (lane == 0) kback[(blk % 3) * 4 + vw] = fb;
        const float r[8] = {fast_rcp(s0.x) * fs, fast_rcp(s0.y) * fs, fast_rcp(s0.z) * fs, fast_rcp(s0.w) * fs,
                            fast_rcp(s1.x) * fs, fast_rcp(s1.y) * fs, fast_rcp(s1.z) * fs, fast_rcp(s1.w) * fs};
#pragma unroll
        for (int e = 0; e < CPG; ++e) {
          uint32_t hw[4], lw[4];
          float bsum = 0.f;
#pragma unroll
          for (int pr = 0; pr < 4; ++pr) {
            const int k0 = 2 * pr, k1 = 2 * pr + 1;
            const float x0 = qreg[e][k0] * r[(k0 >> 1) + 4 * (k0 & 1)];
            const float x1 = qreg[e][k1] * r[(k1 >> 1) + 4 * (k1 & 1)];
            bsum += (pr & 1) ? 16.f * (x0 + x1) : x0 + x1;  // q / sK with the x16 slots' 1/16 undone
            const __half2 hi = __floats2half2_rn(x0, x1);
            const float2 back = __half22float2(hi);
            const __half2 lo = __floats2half2_rn(x0 - back.x, x1 - back.y);
            hw[pr] = *reinterpret_cast<const uint32_t*>(&hi);
            lw[pr] = *reinterpret_cast<const uint32_t*>(&lo);
          }
          const int nh = vw * 2 * GP + e0 + e;
          *reinterpret_cast<uint4*>(bqb + b_off(nh, 8 * oct)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(bqb + b_off(nh + GP, 8 * oct)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          // sum over the 16 octets (lanes of the same parity)
#pragma unroll
          for (int off = 2; off < 32; off <<= 1) bsum += __shfl_xor_sync(0xffffffffu, bsum, off);
          // signed Key codes (a wide unit) take no bias out
          if (oct == 0) beta[((blk % 3) * 4 + vw) * 8 + e0 + e] = wide ? 0.f : bsum;
        }
      }
      fence_proxy_async();
      mbar_arrive(bar_a);
    };
    b_build(0);
    for (int blk = 0; blk < nblk && !fail; ++blk) {
      if (blk + 1 < nblk) {
        // B_Q buffer (blk + 1) & 1 was last read by the score MMAs of block blk - 1
        if (blk > 0) fail |= !wait_or_abort(bar_s + 8 * ((blk - 1) & 1), (uint32_t)((blk - 1) >> 1) & 1u, abort);
        fail |= !wait_or_abort(bar_a, (uint32_t)blk & 1u, abort);  // block blk's A phase is complete
        b_build(blk + 1);
      }
      const uint8_t* sb = ring + (blk % kTcSlots) * kTcBlock;  // landed: b_build(blk) waited for it
      uint32_t vr[4][16];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 w = *reinterpret_cast<const uint4*>(sb + j * kTcUnitStride + kTcVcode + c * 16);
        nibble_regs(w.x, *reinterpret_cast<uint32_t(*)[4]>(&vr[j][0]));
        nibble_regs(w.y, *reinterpret_cast<uint32_t(*)[4]>(&vr[j][4]));
        nibble_regs(w.z, *reinterpret_cast<uint32_t(*)[4]>(&vr[j][8]));
        nibble_regs(w.w, *reinterpret_cast<uint32_t(*)[4]>(&vr[j][12]));
      }
      // the previous block's O MMAs have read A_V
      if (blk > 0) fail |= !wait_or_abort(bar_o, (uint32_t)(blk - 1) & 1u, abort);
      tc_fence_after();
#pragma unroll
      for (int j = 0; j < 4; ++j) tc_st16(lane_base + TS::kColAV + 16 * j, vr[j]);
      tc_wait_st();
      tc_fence_before();
      mbar_arrive(bar_p);
    }
    if (fail) *abort = 1;
  } else {
    // ================= Key warps: A_K (one token per thread), scores, softmax,
    // B_P, and the unit's partial =============================================
    bool fail = false;
    int qexp;
    const float kthr = tc_kthr(qred, p.eps, &qexp);
    auto k_codes = [&](int blk) {
      const int s = blk % kTcSlots;
      const uint8_t* sb = ring + s * kTcBlock;
      fail |= !wait_or_abort(bar_ring + 8 * s, (uint32_t)(blk / kTcSlots) & 1u, abort);
      const uint4* kr = reinterpret_cast<const uint4*>(sb + warp * kTcUnitStride + lane * (D / 2));
      const uint32_t colk = TS::kColAK;
      // a wide unit (some Key scale below kthr, decided as its B_Q builder
      // decides) enters with signed codes
      bool wide = false;
      if (warp < min(4, nunits - 4 * blk)) {
        const float4 s4 = reinterpret_cast<const float4*>(sb + warp * kTcUnitStride + kTcKsc)[lane];
        wide = fminf(fminf(s4.x, s4.y), fminf(s4.z, s4.w)) < kthr;
      }
      wide = __any_sync(0xffffffffu, wide);
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        const uint4 w = kr[qq];
        uint32_t r[16];
        nibble_regs(w.x, *reinterpret_cast<uint32_t(*)[4]>(r + 0));
        nibble_regs(w.y, *reinterpret_cast<uint32_t(*)[4]>(r + 4));
        nibble_regs(w.z, *reinterpret_cast<uint32_t(*)[4]>(r + 8));
        nibble_regs(w.w, *reinterpret_cast<uint32_t(*)[4]>(r + 12));
        if (wide) {
#pragma unroll
          for (int q4i = 0; q4i < 4; ++q4i) unbias_nibbles(*reinterpret_cast<uint32_t(*)[4]>(r + 4 * q4i));
        }
        tc_st16(lane_base + colk + 16 * qq, r);
      }
      tc_wait_st();
      tc_fence_before();
      mbar_arrive(bar_a);
    };
    float m_run[GP], l_part[GP], c_part[GP];
#pragma unroll
    for (int e = 0; e < GP; ++e) {
      m_run[e] = -INFINITY;
      l_part[e] = 0.f;
      c_part[e] = 0.f;
    }
    {
      float z[GP];
#pragma unroll
      for (int e = 0; e < GP; ++e) z[e] = 0.f;
      tc_st_f<GP>(lane_base + TS::kColO, z);
      tc_wait_st();
    }
    k_codes(0);
    int n_o = 0;
    for (int blk = 0; blk < nblk; ++blk) {
      const int nu = min(4, nunits - 4 * blk);
      const uint8_t* sb = ring + (blk % kTcSlots) * kTcBlock;
      // block blk's A phase is complete (also: the Value warps' bias sums are
      // visible) and its score MMAs are done with A_K: the next block's Key
      // codes go in at once, so that its score MMAs overlap this softmax
      fail |= !wait_or_abort(bar_a, (uint32_t)blk & 1u, abort);
      fail |= !wait_or_abort(bar_s + 8 * (blk & 1), (uint32_t)(blk >> 1) & 1u, abort);
      tc_fence_after();
      if (blk + 1 < nblk) k_codes(blk + 1);
      // -- scores of this thread's token: hi and lo columns of its unit, minus the bias
      const uint32_t cols = (blk & 1) ? TS::kColS1 : TS::kColS0;
      const bool valid = warp < nu;
      float sc2[2 * GP];
      if constexpr (GP == 2) {
        tc_ld<4>(lane_base + cols + warp * 2 * GP, sc2);
      } else if constexpr (GP == 4) {
        tc_ld<8>(lane_base + cols + warp * 2 * GP, sc2);
      } else {
        tc_ld<8>(lane_base + cols + warp * 2 * GP, *reinterpret_cast<float(*)[8]>(sc2));
        tc_ld<8>(lane_base + cols + warp * 2 * GP + 8, *reinterpret_cast<float(*)[8]>(sc2 + 8));
      }
      tc_wait_ld();
      float sc[GP];
      // this thread's token: 1/sV (x1/16 on the x16 slots)
      const float* vs = reinterpret_cast<const float*>(sb + warp * kTcUnitStride + kTcVsc);
      const bool x16 = (lane >> 1) & 1;
      float iv = valid ? fast_rcp(vs[lane]) * (x16 ? 0.0625f : 1.f) : 0.f;
      bool up = fail;
      const float kb = kback[(blk % 3) * 4 + warp];
#pragma unroll
      for (int e = 0; e < GP; ++e) {
        const float bias = 8.f * beta[((blk % 3) * 4 + warp) * 8 + e];
        sc[e] = valid ? fmaf(sc2[e] + sc2[GP + e], kTwo24, -bias) * kb : -INFINITY;
        up |= sc[e] > m_run[e] + kSlack;
      }
      // the previous block's O MMAs are done: B_P and the O accumulator are free
      if (n_o > 0) fail |= !wait_or_abort(bar_o, (uint32_t)(n_o - 1) & 1u, abort);
      tc_fence_after();
      if (kgroup_or(up || fail)) {
        // move the running max (maxima over the four Key warps; rescale l, the
        // Value bias sum and the O accumulator), or stop after a failed wait
        float a[GP];
#pragma unroll
        for (int e = 0; e < GP; ++e) {
          float mx = sc[e];
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
          if (lane == 0) red[warp * 8 + e] = mx;
        }
        const bool stop = kgroup_or(fail);  // also publishes the maxima (a barrier)
        if (stop) {
          fail = true;
          *abort = 1;
          break;
        }
#pragma unroll
        for (int e = 0; e < GP; ++e) {
          const float mn = fmaxf(fmaxf(m_run[e], fmaxf(red[e], red[8 + e])), fmaxf(red[16 + e], red[24 + e]));
          a[e] = m_run[e] == -INFINITY ? 0.f : fast_exp2(m_run[e] - mn);
          m_run[e] = mn;
          l_part[e] *= a[e];
          c_part[e] *= a[e];
        }
        if (n_o > 0) {
          float o[GP];
          tc_ld<GP>(lane_base + TS::kColO, o);
          tc_wait_ld();
#pragma unroll
          for (int e = 0; e < GP; ++e) o[e] *= a[e];
          tc_st_f<GP>(lane_base + TS::kColO, o);
          tc_wait_st();
        }
        kgroup_sync();  // every warp has read the maxima before they are written again
      }
      // -- P / sV into B_P (row e, k-slot = block token), x1/16 on the x16 slots;
      // the Value bias is 8 times the sum of exactly these f16 values.  A wide
      // block (some Value absmax > kVWideAbs, or a Value scale below eps,
      // which divides by eps) has no output MMAs: each thread adds its
      // channel's terms code * p * min(1/sV, 1/eps) * 2^-24 over the block's
      // tokens to O in fp32 (signed codes, no bias; the weights pass through
      // the B_P area, which no MMA reads for this block).
      {
        const int k = 32 * warp + lane;
        const bool vwide = tc_value_wide(sb, nu, lane, kTcVsc, kTcUnitStride, kVWideAbs / (float)p.qmax);
        if (t == 0) vflag[blk & 1] = vwide ? 1 : 0;
        float pw[GP];
#pragma unroll
        for (int e = 0; e < GP; ++e) {
          pw[e] = valid ? fast_exp2(sc[e] - (m_run[e] == -INFINITY ? 0.f : m_run[e])) : 0.f;
          l_part[e] += pw[e];
        }
        if (!vwide) {
#pragma unroll
          for (int e = 0; e < GP; ++e) {
            const __half hv = __float2half_rn(pw[e] * iv);
            c_part[e] = fmaf(__half2float(hv), x16 ? 16.f : 1.f, c_part[e]);
            *reinterpret_cast<__half*>(bpm + b_off(e, k)) = hv;
          }
        } else {
          float* wts = reinterpret_cast<float*>(bpm);  // [128 tokens][GP]
          const float ivr = fminf(iv * (x16 ? 16.f : 1.f), fast_rcp(p.eps)) * 5.9604644775390625e-8f;
#pragma unroll
          for (int e = 0; e < GP; ++e) wts[k * GP + e] = pw[e] * ivr;
          kgroup_sync();
          // this thread's channel c = k: its 16-byte code row in each unit
          float acc[GP];
#pragma unroll
          for (int e = 0; e < GP; ++e) acc[e] = 0.f;
#pragma unroll 1
          for (int j = 0; j < nu; ++j) {
            const uint4 cw = *reinterpret_cast<const uint4*>(sb + j * kTcUnitStride + kTcVcode + k * 16);
            const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
            for (int wi = 0; wi < 4; ++wi) {
#pragma unroll
              for (int nb = 0; nb < 8; ++nb) {
                // nibble nb of word wi is token 8 wi + 2 nb (nb < 4), else 8 wi + 2 (nb - 4) + 1
                const int tok = 32 * j + 8 * wi + (nb < 4 ? 2 * nb : 2 * (nb - 4) + 1);
                const float code = (float)((int)((words[wi] >> (4 * nb)) & 0xFu) - 8);
#pragma unroll
                for (int e = 0; e < GP; ++e) acc[e] = fmaf(code, wts[tok * GP + e], acc[e]);
              }
            }
          }
          float o[GP];
          tc_ld<GP>(lane_base + TS::kColO, o);
          tc_wait_ld();
#pragma unroll
          for (int e = 0; e < GP; ++e) o[e] += acc[e];
          tc_st_f<GP>(lane_base + TS::kColO, o);
          tc_wait_st();
          kgroup_sync();  // every thread has read the weights before B_P is written again
        }
      }
      tc_fence_before();
      fence_proxy_async();
      mbar_arrive(bar_p);
      ++n_o;
    }
    // ---- the unit's partial -------------------------------------------------------
    if (!fail && n_o > 0) fail |= !wait_or_abort(bar_o, (uint32_t)(n_o - 1) & 1u, abort);
    tc_fence_after();
    float o[GP];
    if (!fail) {
      tc_ld<GP>(lane_base + TS::kColO, o);
      tc_wait_ld();
    }
    float* csum = red + 64;
#pragma unroll
    for (int e = 0; e < GP; ++e) {
      float ls = l_part[e], cs = c_part[e];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        ls += __shfl_xor_sync(0xffffffffu, ls, off);
        cs += __shfl_xor_sync(0xffffffffu, cs, off);
      }
      if (lane == 0) {
        red[32 + warp * 8 + e] = ls;
        csum[warp * 8 + e] = cs;
      }
    }
    const bool bad = kgroup_or(fail);
    if (bad) *abort = 1;
    if (bad && t == 0) atomicOr(p.status, kStatusWaitTimeout);
    float* part = p.partials + (unit * p.max_splits + slot) * (int64_t)p.g * part_row(D);
#pragma unroll
    for (int e = 0; e < GP; ++e) {
      if (e < p.g) {
        const float C = (csum[e] + csum[8 + e]) + (csum[16 + e] + csum[24 + e]);
        part[(int64_t)e * part_row(D) + t] = bad ? 0.f : fmaf(o[e], kTwo24, -8.f * C);
        if (t == 0) {
          part[(int64_t)e * part_row(D) + D] = bad ? -INFINITY : m_run[e];
          part[(int64_t)e * part_row(D) + D + 1] = bad ? 0.f : (red[32 + e] + red[40 + e]) + (red[48 + e] + red[56 + e]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kTcMmaWarp) {
    __syncwarp();
    tc_dealloc_n<TS::kCols>(tm);
  }
}

template <int GP, int MODE>
cudaError_t launch_tc_t(const DecodeParams& p, cudaStream_t s) {
  const size_t smem = TcShape<GP>::smem;
  int dev = 0;
  cudaGetDevice(&dev);
  static size_t configured[64] = {};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (smem > configured[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(decode_tc_kernel<GP, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // all of the unified L1 as shared memory: two CTAs per SM
    e = cudaFuncSetAttribute(decode_tc_kernel<GP, MODE>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    configured[dev] = smem;
  }
  const dim3 grid((p.grid_splits + 1) * p.n_seqs * p.Hkv);
  return launch_pdl(decode_tc_kernel<GP, MODE>, grid, dim3(kTcThreads), smem, s, p);
}

template <int GP>
cudaError_t launch_tc_m(const DecodeParams& p, cudaStream_t s) {
  if (p.G != 32) return launch_tc_t<GP, kStaged>(p, s);
  return p.map.table ? launch_tc_t<GP, kPaged32>(p, s) : launch_tc_t<GP, kFlat32>(p, s);
}

}  // namespace

bool decode_tc_supported(const DecodeParams& p) {
  return p.D == kTcD && p.bits == 4 && p.G % 32 == 0 && p.g >= 2 && p.g <= kMaxGqa && !p.seg.kcodes;
}

cudaError_t launch_decode_tc(const DecodeParams& p, cudaStream_t s, int* supported) {
  *supported = decode_tc_supported(p);
  if (!*supported) return cudaSuccess;
  switch (gqa_pad(p.g)) {
    case 2: return launch_tc_m<2>(p, s);
    case 4: return launch_tc_m<4>(p, s);
    default: return launch_tc_m<8>(p, s);
  }
}

}  // namespace kvq
