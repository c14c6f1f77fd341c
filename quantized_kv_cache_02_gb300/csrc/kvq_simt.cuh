// CUDA-core decode attention over one split item (a run of quantized group
// pages, or the residual window) of one (sequence, KV head) unit, for all g
// query heads that read that KV head ("KV Cache 与自回归视频生成" section 04,
// attn_step: head h reads KV head h / g).  Each warp keeps an online-softmax
// state (running max m, sum l, unnormalised o) per head over its tokens; the
// CTA merges its warps and writes one partial (o[D], m, l) per head, which the
// combine kernel merges across splits (section 05, FlashDecoding).
// Dequantization follows the page's restore: x = code / scale (fp32 division).
#pragma once

#include <cuda_bf16.h>

#include "kvq_internal.h"

namespace kvq {

constexpr int kSimtThreads = 128;
constexpr int kSimtWarps = kSimtThreads / 32;

__device__ __forceinline__ float ld_f32(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ld_f32(const __nv_bfloat16* p, int64_t i) { return __bfloat162float(p[i]); }

// Signed code of channel c of token tl (group-local) of a page (stored as
// offset binary: code + 8 per nibble, code + 128 per byte).
template <int BITS>
__device__ __forceinline__ int key_code(const uint8_t* page, int tl, int c, int D) {
  if (BITS == 2) {
    const uint8_t byte = page[(int64_t)tl * (D / 4) + (c >> 2)];
    return (int)((byte >> (2 * (c & 3))) & 0x3) - 2;
  } else if (BITS == 4) {
    const uint8_t byte = page[(int64_t)tl * (D / 2) + (c >> 1)];
    const int nib = (c & 1) ? (byte >> 4) : (byte & 0xF);
    return nib - 8;
  } else {
    return (int)page[(int64_t)tl * D + c] - 128;
  }
}

template <int BITS>
__device__ __forceinline__ int value_code(const uint8_t* vbase, int G, int tl, int c, int D) {
  const int st = tl >> 5, o = tl & 31;
  const int n_st = min(32, G - 32 * st);
  const uint8_t* sub = vbase + (int64_t)st * 32 * D * BITS / 8;
  if (BITS == 2) {
    // 16-bit pieces of 8 tokens: token 2f in bits 2f, token 2f + 1 in bits 8 + 2f
    const int k = o & 7;
    const uint32_t piece = reinterpret_cast<const uint16_t*>(sub)[c * (n_st / 8) + (o >> 3)];
    return (int)((piece >> (8 * (k & 1) + 2 * (k >> 1))) & 0x3) - 2;
  } else if (BITS == 4) {
    const int w = o >> 3, k = o & 7;
    const int jn = (k >> 1) + 4 * (k & 1);  // nibble that holds token offset k
    const uint32_t word = reinterpret_cast<const uint32_t*>(sub)[c * (n_st / 8) + w];
    const int nib = (word >> (4 * jn)) & 0xF;
    return nib - 8;
  } else {
    return (int)sub[c * n_st + o] - 128;
  }
}

template <int CPL>
struct SimtState {
  float m[kMaxGqa], l[kMaxGqa], o[kMaxGqa][CPL];
};

template <int CPL>
__device__ __forceinline__ void simt_token(SimtState<CPL>& s, const float (&qv)[kMaxGqa][CPL],
                                           const float (&kv)[CPL], const float (&vv)[CPL], int g) {
#pragma unroll
  for (int j = 0; j < kMaxGqa; ++j) {
    if (j >= g) break;
    float part = 0.f;
#pragma unroll
    for (int k = 0; k < CPL; ++k) part = fmaf(qv[j][k], kv[k], part);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    const float m_new = fmaxf(s.m[j], part);
    const float corr = exp2f(s.m[j] - m_new);
    const float pw = exp2f(part - m_new);
    s.l[j] = fmaf(s.l[j], corr, pw);
#pragma unroll
    for (int k = 0; k < CPL; ++k) s.o[j][k] = fmaf(s.o[j][k], corr, pw * vv[k]);
    s.m[j] = m_new;
  }
}

// Shared scratch of simt_item in floats (q, per-warp m and l, per-warp o).
template <int CPL>
__host__ __device__ constexpr int simt_scratch_floats() {
  return kMaxGqa * CPL * 32 + 2 * kSimtWarps * kMaxGqa + kSimtWarps * kMaxGqa * CPL * 32;
}

// Channel of register k of a lane: strided (lane + 32 k) in general; for a
// segmented cache contiguous (CPL lane + k), so that a token's codes for the
// lane are one load.
template <int CPL, bool SEG>
__device__ __forceinline__ constexpr int lane_chan(int lane, int k) {
  return SEG ? CPL * lane + k : lane + 32 * k;
}

// Sums over the 32 lanes of N values (N = 4 or 8), every lane ending with all
// N sums.  The first log2(N) exchange steps halve the set each time, a lane
// keeping the half its lane bit selects, so each exchange carries half as many
// values as the last; the remaining steps finish one sum per lane, and N
// shuffles hand the sums back: 17 shuffles for 8 values instead of 40.
template <int N>
__device__ __forceinline__ void warp_sum_n(float (&v)[N], int lane) {
  static_assert(N == 4 || N == 8, "4 or 8 values");
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
  float a[N / 2];
#pragma unroll
  for (int i = 0; i < N / 2; ++i) {
    const float mine = b4 ? v[N / 2 + i] : v[i], other = b4 ? v[i] : v[N / 2 + i];
    a[i] = mine + __shfl_xor_sync(0xffffffffu, other, 16);
  }
  float x;
  if constexpr (N == 8) {
    float c[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float mine = b3 ? a[2 + i] : a[i], other = b3 ? a[i] : a[2 + i];
      c[i] = mine + __shfl_xor_sync(0xffffffffu, other, 8);
    }
    x = (b2 ? c[1] : c[0]) + __shfl_xor_sync(0xffffffffu, b2 ? c[0] : c[1], 4);  // value 4 b4 + 2 b3 + b2
  } else {
    x = (b3 ? a[1] : a[0]) + __shfl_xor_sync(0xffffffffu, b3 ? a[0] : a[1], 8);  // value 2 b4 + b3
    x += __shfl_xor_sync(0xffffffffu, x, 4);
  }
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  x += __shfl_xor_sync(0xffffffffu, x, 1);
#pragma unroll
  for (int i = 0; i < N; ++i)
    v[i] = N == 8 ? __shfl_sync(0xffffffffu, x, ((i >> 2) & 1) * 16 + ((i >> 1) & 1) * 8 + (i & 1) * 4)
                  : __shfl_sync(0xffffffffu, x, ((i >> 1) & 1) * 16 + (i & 1) * 8);
}

// Codes of channels CPL lane .. CPL lane + CPL - 1 of a token row, as floats.
// A field u (code + bias) OR-ed into the mantissa of 2^23 is the float 2^23 + u
// exactly, and subtracting 2^23 + bias leaves the code: a logic op and an add
// instead of an integer-to-float conversion.
template <int BITS, int CPL>
__device__ __forceinline__ void row_codes_f(const uint8_t* row, int lane, int D, float (&code)[CPL]) {
  constexpr int kBits = CPL * BITS;
  const int c0 = CPL * lane;
  if (c0 >= D) {
#pragma unroll
    for (int k = 0; k < CPL; ++k) code[k] = 0.f;
    return;
  }
  uint64_t v;
  const uint8_t* src = row + c0 * BITS / 8;
  if constexpr (kBits < 8) v = (uint64_t)(*src >> ((c0 * BITS) & 7));
  else if constexpr (kBits == 8) v = *src;
  else if constexpr (kBits == 16) v = *reinterpret_cast<const uint16_t*>(src);
  else if constexpr (kBits == 32) v = *reinterpret_cast<const uint32_t*>(src);
  else v = *reinterpret_cast<const uint64_t*>(src);
  constexpr float kOff = 8388608.f + (BITS == 2 ? 2.f : BITS == 4 ? 8.f : 128.f);
#pragma unroll
  for (int k = 0; k < CPL; ++k)
    code[k] = __uint_as_float(0x4B000000u | (uint32_t)((v >> (BITS * k)) & ((1u << BITS) - 1u))) - kOff;
}

// Whole split item on CUDA cores; writes the partial of slot ``slot``.
// ``win`` selects the residual window (tokens [Q, T) from the ring) instead of
// pages [pg0, pg1) of the quantized prefix.

// SEG: a segmented cache (token-major rows, a Key scale row per segment).
template <typename T, int BITS, int CPL, bool SEG>
__device__ inline void simt_item(const DecodeParams& p, int i, int h, bool win, int pg0, int pg1, int slot,
                          float* scratch) {
  float (*qs)[CPL * 32] = reinterpret_cast<float (*)[CPL * 32]>(scratch);
  float (*wm)[kMaxGqa] = reinterpret_cast<float (*)[kMaxGqa]>(scratch + kMaxGqa * CPL * 32);
  float (*wl)[kMaxGqa] = wm + kSimtWarps;
  float (*wo)[kMaxGqa][CPL * 32] =
      reinterpret_cast<float (*)[kMaxGqa][CPL * 32]>(scratch + kMaxGqa * CPL * 32 + 2 * kSimtWarps * kMaxGqa);
  const int D = p.D, g = p.g, G = p.G;
  const int b = p.seq_begin + i;
  const int64_t unit = (int64_t)b * p.Hkv + h;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const T* q = reinterpret_cast<const T*>(p.q) + ((int64_t)b * p.Hq + (int64_t)h * g) * D;
  for (int idx = threadIdx.x; idx < kMaxGqa * CPL * 32; idx += blockDim.x) {
    const int j = idx / (CPL * 32), c = idx - j * (CPL * 32);
    qs[j][c] = (j < g && c < D) ? ld_f32(q, (int64_t)j * D + c) * p.qk_scale : 0.f;
  }
  __syncthreads();
  float qv[kMaxGqa][CPL];
#pragma unroll
  for (int j = 0; j < kMaxGqa; ++j)
#pragma unroll
    for (int k = 0; k < CPL; ++k) qv[j][k] = qs[j][lane_chan<CPL, SEG>(lane, k)];

  SimtState<CPL> s;
#pragma unroll
  for (int j = 0; j < kMaxGqa; ++j) {
    s.m[j] = -INFINITY;
    s.l[j] = 0.f;
#pragma unroll
    for (int k = 0; k < CPL; ++k) s.o[j][k] = 0.f;
  }

  float kv[CPL], vv[CPL];
  if (win) {
    const int64_t T0 = p.ctr[i].total, Q0 = p.ctr[i].quantized;
    const T* rk = reinterpret_cast<const T*>(p.ring_k) + unit * p.Rcap * D;
    const T* rv = reinterpret_cast<const T*>(p.ring_v) + unit * p.Rcap * D;
    for (int64_t t = Q0 + warp; t < T0; t += kSimtWarps) {
      const int64_t row = (t % p.Rcap) * D;
#pragma unroll
      for (int k = 0; k < CPL; ++k) {
        const int c = lane_chan<CPL, SEG>(lane, k);
        kv[k] = c < D ? ld_f32(rk, row + c) : 0.f;
        vv[k] = c < D ? ld_f32(rv, row + c) : 0.f;
      }
      simt_token<CPL>(s, qv, kv, vv, g);
    }
  } else if constexpr (SEG) {
    // segmented cache: a "page" is one token of the token-major code rows.
    // q.k = sum_c q_c code_c / sK_c: the 1/sK of the token's segment is folded
    // into q whenever the segment changes (a prefill segment spans thousands
    // of tokens); the Value scale 1/sV goes onto the token's codes.  Two
    // tokens per pass (head_dim <= 128): both tokens' codes and scales are
    // loaded before either is used, so their memory latencies overlap, and
    // the pass's (token, head) dot products are summed over the warp at once.
    // The running max moves only when a score exceeds it by more than 8 (in
    // base 2), as in the tensor-core kernel: l and o always share m, so o / l
    // is exact, and a token costs one exp2 per head.
    const int32_t* first = p.seg.first + (int64_t)b * p.seg.cap;
    int cur = -1;
    constexpr int kTok = CPL <= 4 ? 2 : 1;
    constexpr float kSlack = 8.f;
    for (int64_t t0 = pg0 + warp; t0 < pg1; t0 += kTok * kSimtWarps) {
      int fk[kTok];
      float kc[kTok][CPL], vc[kTok][CPL], vsr[kTok];
#pragma unroll
      for (int u = 0; u < kTok; ++u) {
        const int64_t t = t0 + u * kSimtWarps;
        const bool ok = t < pg1;  // the same for every lane of the warp
        const int64_t row = unit * p.seg.cap + (ok ? t : t0);
        const uint8_t* kr = p.seg.kcodes + row * p.seg.row_bytes;
        const uint8_t* vr = p.seg.vcodes + row * p.seg.row_bytes;
        fk[u] = ok ? first[t] : -1;
        vsr[u] = p.seg.vscales[row];
        row_codes_f<BITS, CPL>(kr, lane, D, kc[u]);
        row_codes_f<BITS, CPL>(vr, lane, D, vc[u]);
      }
      // this lane's share of every (token, head) dot product
      float part[kTok][kMaxGqa];
#pragma unroll
      for (int u = 0; u < kTok; ++u) {
        if (fk[u] >= 0 && fk[u] != cur) {
          const float* ks = p.seg.kscales + (unit * p.seg.cap + fk[u]) * D;
#pragma unroll
          for (int k = 0; k < CPL; ++k) {
            const int c = lane_chan<CPL, SEG>(lane, k);
            const float r = c < D ? __frcp_rn(fmaxf(ks[c], p.eps)) : 0.f;
#pragma unroll
            for (int j = 0; j < kMaxGqa; ++j) qv[j][k] = qs[j][c] * r;  // q / sK from here on
          }
          cur = fk[u];
        }
#pragma unroll
        for (int j = 0; j < kMaxGqa; ++j) {
          float a = 0.f;
#pragma unroll
          for (int k = 0; k < CPL; ++k) a = fmaf(qv[j][k], kc[u][k], a);
          part[u][j] = a;
        }
      }
      // sums over the warp, four heads of every token per exchange set
      // (eight heads: two sets)
#pragma unroll
      for (int j0 = 0; j0 < kMaxGqa; j0 += 4) {
        if (j0 >= g) break;
        float v[4 * kTok];
#pragma unroll
        for (int u = 0; u < kTok; ++u)
#pragma unroll
          for (int j = 0; j < 4; ++j) v[4 * u + j] = part[u][j0 + j];
        warp_sum_n<4 * kTok>(v, lane);
#pragma unroll
        for (int u = 0; u < kTok; ++u)
#pragma unroll
          for (int j = 0; j < 4; ++j) part[u][j0 + j] = v[4 * u + j];
      }
      // move the reference max only when some score passes it by kSlack (the
      // sums are the same in every lane, so the branch is the warp's)
      bool up = false;
#pragma unroll
      for (int u = 0; u < kTok; ++u)
#pragma unroll
        for (int j = 0; j < kMaxGqa; ++j)
          if (j < g && fk[u] >= 0) up |= part[u][j] > s.m[j] + kSlack;
      if (up) {
#pragma unroll
        for (int j = 0; j < kMaxGqa; ++j) {
          if (j >= g) break;
          float mx = s.m[j];
#pragma unroll
          for (int u = 0; u < kTok; ++u)
            if (fk[u] >= 0) mx = fmaxf(mx, part[u][j]);
          const float corr = s.m[j] == -INFINITY ? 0.f : exp2f(s.m[j] - mx);
          s.m[j] = mx;
          s.l[j] *= corr;
#pragma unroll
          for (int k = 0; k < CPL; ++k) s.o[j][k] *= corr;
        }
      }
#pragma unroll
      for (int u = 0; u < kTok; ++u) {
        if (fk[u] < 0) break;
        const float iv = __frcp_rn(fmaxf(vsr[u], p.eps));
#pragma unroll
        for (int k = 0; k < CPL; ++k) vv[k] = vc[u][k] * iv;
#pragma unroll
        for (int j = 0; j < kMaxGqa; ++j) {
          if (j >= g) break;
          const float pw = exp2f(part[u][j] - s.m[j]);
          s.l[j] += pw;
#pragma unroll
          for (int k = 0; k < CPL; ++k) s.o[j][k] = fmaf(pw, vv[k], s.o[j][k]);
        }
      }
    }
  } else {
    const int64_t ntok = (int64_t)(pg1 - pg0) * G;
    for (int64_t tt = warp; tt < ntok; tt += kSimtWarps) {
      const int pg = pg0 + (int)(tt / G), tl = (int)(tt % G);
      const uint8_t* page = p.pages + page_offset(p.map, p.geom.page_bytes, b, h, pg);
      const float* ks = reinterpret_cast<const float*>(page + p.geom.kscale_off);
      const float vs = reinterpret_cast<const float*>(page + p.geom.vscale_off)[tl];
#pragma unroll
      for (int k = 0; k < CPL; ++k) {
        const int c = lane + 32 * k;
        if (c < D) {
          kv[k] = __fdiv_rn((float)key_code<BITS>(page, tl, c, D), fmaxf(ks[c], p.eps));
          vv[k] = __fdiv_rn((float)value_code<BITS>(page + p.geom.code_bytes, G, tl, c, D), fmaxf(vs, p.eps));
        } else {
          kv[k] = 0.f;
          vv[k] = 0.f;
        }
      }
      simt_token<CPL>(s, qv, kv, vv, g);
    }
  }

  // merge the warps of this CTA
  if (lane == 0) {
#pragma unroll
    for (int j = 0; j < kMaxGqa; ++j) {
      wm[warp][j] = s.m[j];
      wl[warp][j] = s.l[j];
    }
  }
#pragma unroll
  for (int j = 0; j < kMaxGqa; ++j)
#pragma unroll
    for (int k = 0; k < CPL; ++k) wo[warp][j][lane_chan<CPL, SEG>(lane, k)] = s.o[j][k];
  __syncthreads();
  float* part = p.partials + (unit * p.max_splits + slot) * (int64_t)g * part_row(D);
  for (int idx = threadIdx.x; idx < g * D; idx += blockDim.x) {
    const int j = idx / D, c = idx - j * D;
    float M = -INFINITY;
    for (int w = 0; w < kSimtWarps; ++w) M = fmaxf(M, wm[w][j]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
      for (int w = 0; w < kSimtWarps; ++w) {
        if (wm[w][j] == -INFINITY) continue;
        const float f = exp2f(wm[w][j] - M);
        L = fmaf(wl[w][j], f, L);
        O = fmaf(wo[w][j][c], f, O);
      }
    }
    part[(int64_t)j * part_row(D) + c] = O;
    if (c == 0) {
      part[(int64_t)j * part_row(D) + D] = M;
      part[(int64_t)j * part_row(D) + D + 1] = L;
    }
  }
}

// Merge of one (sequence, query head)'s split partials by one warp:
// M = max m_s, L = sum l_s 2^(m_s - M), o = sum o_s 2^(m_s - M) / L
// ("KV Cache 与自回归视频生成" section 05, FlashDecoding).  base points at
// the head's row in slot 0; slot k < nsplit is split column k, a later one
// the window's (column max_splits - 1); rows are ``stride`` floats apart.
// The slots are taken eight at a time: lane s reads slot s's (m, l) while
// every lane reads its 16-byte pieces of the eight o rows, so one round trip
// serves the whole chunk; the chunk is then folded into the running
// (M, L, o) with the usual rescale.  VPL = 16-byte pieces of o per lane (1
// for head_dim <= 128, 2 up to 256).  FRESH: the partials were written by
// other CTAs of the running launch, so they are read from L2 (ld.global.cg),
// never through a possibly stale L1 line.  No slots: zeros.
template <int VPL, bool FRESH>
__device__ __forceinline__ void merge_head(const float* base, int nsplit, int nslots, int max_splits, int64_t stride,
                                           int D, float* out_row, int lane) {
  // slots whose loads are in flight together: a whole warp's worth of (m, l)
  // and as many o rows as registers allow, so a short decode's 17 or so
  // slots take one round trip
  constexpr int kCombineChunk = VPL == 1 ? (FRESH ? 24 : 32) : 16;
  constexpr int kReduce = kCombineChunk > 16 ? 16 : kCombineChunk > 8 ? 8 : 4;  // first butterfly offset
  const int nvec = D >> 2;
  auto row = [&](int k) { return base + (k < nsplit ? k : max_splits - 1) * stride; };
  auto ld2 = [](const float* q) {
    return FRESH ? __ldcg(reinterpret_cast<const float2*>(q)) : __ldg(reinterpret_cast<const float2*>(q));
  };
  auto ld4 = [](const float* q, int c4) {
    return FRESH ? __ldcg(reinterpret_cast<const float4*>(q) + c4) : __ldg(reinterpret_cast<const float4*>(q) + c4);
  };
  float M = -INFINITY, L = 0.f;
  float4 o[VPL];
#pragma unroll
  for (int e = 0; e < VPL; ++e) o[e] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k0 = 0; k0 < nslots; k0 += kCombineChunk) {
    const int n = min(kCombineChunk, nslots - k0);
    float2 ml = make_float2(-INFINITY, 0.f);
    if (lane < n) ml = ld2(row(k0 + lane) + D);
    float4 v[kCombineChunk][VPL];
#pragma unroll
    for (int s = 0; s < kCombineChunk; ++s)
#pragma unroll
      for (int e = 0; e < VPL; ++e) {
        const int c4 = lane + 32 * e;
        v[s][e] = (s < n && c4 < nvec) ? ld4(row(k0 + s), c4) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    float cm = ml.x;
#pragma unroll
    for (int off = kReduce; off > 0; off >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, off));
    cm = __shfl_sync(0xffffffffu, cm, 0);
    const float Mn = fmaxf(M, cm);
    const float Ms = Mn == -INFINITY ? 0.f : Mn;
    const float corr = exp2f(M - Ms);
    const float f = exp2f(ml.x - Ms);  // lanes >= n: 0
    float ls = ml.y * f;
#pragma unroll
    for (int off = kReduce; off > 0; off >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, off);
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
  float4* out = reinterpret_cast<float4*>(out_row);
#pragma unroll
  for (int e = 0; e < VPL; ++e) {
    const int c4 = lane + 32 * e;
    if (c4 < nvec) out[c4] = make_float4(o[e].x * inv, o[e].y * inv, o[e].z * inv, o[e].w * inv);
  }
}

// Which split item CTA (x, unit) of a decode launch handles.  Returns false if
// the CTA has nothing to do.
__device__ __forceinline__ bool split_item(const DecodeParams& p, int x, int i, bool* win, int* pg0,
                                           int* pg1, int* slot) {
  const int T0 = p.ctr[i].total, Q0 = p.ctr[i].quantized;
  const int P = Q0 / p.G;
  const int nsplit = (P + p.chunk_pages - 1) / p.chunk_pages;
  if (x == p.grid_splits) {
    *win = true;
    *slot = p.max_splits - 1;
    *pg0 = *pg1 = 0;
    return T0 > Q0;
  }
  if (x >= nsplit) return false;
  *win = false;
  *slot = x;
  *pg0 = x * p.chunk_pages;
  *pg1 = min(P, *pg0 + p.chunk_pages);
  return true;
}

}  // namespace kvq
