// Persistent-warp split kernel of the decode attention ("work line").
//
// The launch's work is laid out as one line: unit (sequence i, KV head h) in
// launch order contributes its quantized prefix as 32-token items (a G = 32
// page, or a 32-token slice of a larger group) and then its residual window
// as 16-row steps, each counted kWinWeight positions.  Every warp of a grid
// of exactly the resident CTAs takes an equal run of positions
// [w C / N, (w + 1) C / N) across unit boundaries, so all warps stay in their
// loops from the first copy to the last and none waits for a CTA's set-up,
// merge or the grid's tail.  A warp streams its items through its own ring of
// shared-memory slots with cp.async.bulk and one mbarrier per slot (a page
// item takes one slot, a window step two: its 16 Key rows and its 16 Value
// rows, each row copied to a padded stride so ldmatrix reads them without
// bank conflicts); the copies of the next unit's items go out while the
// current unit is being finished.  Per unit it keeps the online softmax state
// of decode_mma_kernel (pages through mma_group, window steps through the
// bf16 MMA path), and writes one partial (o, m, l) per (unit, warp) to slot
// w - (first warp of the unit); the combine merges a unit's slots.
//
// ("KV Cache 与自回归视频生成" 3.1, attn_step and section 05, FlashDecoding;
// "KV Cache Quantization Strategies", restore.)

#pragma once

#include "kvq_decode_mma.cuh"

namespace kvq {
namespace {

constexpr int kWinRows = 16;    // rows of a window step
constexpr int kWinWeight = 2;   // line positions of a window step (about its bytes against a page's)
constexpr int kLineWarps = kMmaWarps;

// Bytes between window rows in a slot: the row plus 16, so the 8 rows an
// ldmatrix reads fall on distinct 16-byte bank groups.
template <int D>
__host__ __device__ constexpr int win_row_stride() {
  return 2 * D + 16;
}

// Shape of one unit on the line: U 32-token items, then S window steps.
struct LineUnit {
  int U, S, cost;  // cost = U + kWinWeight * S positions
};

__device__ __forceinline__ LineUnit line_unit(const DecodeParams& p, int i) {
  const int Q = p.ctr[i].quantized, T = p.ctr[i].total;
  LineUnit u;
  u.U = Q / 32;
  u.S = (T - Q + kWinRows - 1) / kWinRows;
  u.cost = u.U + kWinWeight * u.S;
  return u;
}

// Warp that holds line position x: the largest w with floor(w C / N) <= x.
__device__ __forceinline__ int line_warp_of(int64_t x, int64_t C, int N) {
  return (int)(((x + 1) * (int64_t)N - 1) / C);
}

// The unit holding line position x < C: its sequence i (the largest with
// line_start[i] <= x, which holds tokens), head h and first position.
struct LineUnitAt {
  int i, h;
  int start;
  LineUnit u;
};
__device__ __forceinline__ LineUnitAt line_unit_at(const DecodeParams& p, int x) {
  int lo = 0, hi = p.n_seqs;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (p.line_start[mid] <= x) lo = mid;
    else hi = mid;
  }
  LineUnitAt a;
  a.i = lo;
  a.u = line_unit(p, lo);
  const int s0 = (int)p.line_start[lo];
  a.h = (x - s0) / a.u.cost;
  a.start = s0 + a.h * a.u.cost;
  return a;
}

// The warp's items of one unit on the CUDA cores, in fp32 (a unit whose
// flushed maxima put it outside the tensor-core path's range): 32-token
// items [u0, u1) and window rows [r0, r1); writes the partial to ``slot``.
// Restore divides by max(scale, eps), as the page's restore does.
template <int D, int BITS>
__device__ __noinline__ void line_unit_cuda_cores(const uint8_t* pages, PageMap map, PageGeom geom,
                                                  const __nv_bfloat16* ring_k, const __nv_bfloat16* ring_v,
                                                  const __nv_bfloat16* q, float* part, int g, int G, int Rcap,
                                                  int64_t Q0, float eps, float qk_scale, int b, int h, int u0,
                                                  int u1, int r0, int r1) {
  constexpr int CPL = D / 32;
  const int lane = threadIdx.x & 31;
  float qv[kMaxGqa][CPL];
#pragma unroll
  for (int j = 0; j < kMaxGqa; ++j)
#pragma unroll
    for (int k = 0; k < CPL; ++k)
      qv[j][k] = j < g ? __bfloat162float(q[(int64_t)j * D + lane + 32 * k]) * qk_scale : 0.f;
  SimtState<CPL> s;
#pragma unroll
  for (int j = 0; j < kMaxGqa; ++j) {
    s.m[j] = -INFINITY;
    s.l[j] = 0.f;
#pragma unroll
    for (int k = 0; k < CPL; ++k) s.o[j][k] = 0.f;
  }
  float kv[CPL], vv[CPL];
  for (int64_t t = (int64_t)u0 * 32; t < (int64_t)u1 * 32; ++t) {
    const int pg = (int)(t / G), tl = (int)(t - (int64_t)pg * G);
    const uint8_t* page = pages + page_offset(map, geom.page_bytes, b, h, pg);
    const float* ks = reinterpret_cast<const float*>(page + geom.kscale_off);
    const float vs = reinterpret_cast<const float*>(page + geom.vscale_off)[tl];
#pragma unroll
    for (int k = 0; k < CPL; ++k) {
      const int c = lane + 32 * k;
      kv[k] = __fdiv_rn((float)key_code<BITS>(page, tl, c, D), fmaxf(ks[c], eps));
      vv[k] = __fdiv_rn((float)value_code<BITS>(page + geom.code_bytes, G, tl, c, D), fmaxf(vs, eps));
    }
    simt_token<CPL>(s, qv, kv, vv, g);
  }
  for (int r = r0; r < r1; ++r) {
    const int64_t row = ((Q0 + r) % Rcap) * D;
#pragma unroll
    for (int k = 0; k < CPL; ++k) {
      kv[k] = __bfloat162float(ring_k[row + lane + 32 * k]);
      vv[k] = __bfloat162float(ring_v[row + lane + 32 * k]);
    }
    simt_token<CPL>(s, qv, kv, vv, g);
  }
#pragma unroll
  for (int j = 0; j < kMaxGqa; ++j) {
    if (j >= g) break;
#pragma unroll
    for (int k = 0; k < CPL; ++k) part[(int64_t)j * part_row(D) + lane + 32 * k] = s.o[j][k];
    if (lane == 0) {
      part[(int64_t)j * part_row(D) + D] = s.m[j];
      part[(int64_t)j * part_row(D) + D + 1] = s.l[j];
    }
  }
}

// One 16-row window step on the tensor cores: rows [0, n) of the Key slot
// ``kb`` and the Value slot ``vb`` (row r at r * RS); bq holds the unit's q
// as bf16 B fragments.  As rows_mma: S = K q with bf16 MMAs, the exact
// running max, O^T += V^T P with P as a bf16 hi + lo pair.
template <int D, int GP>
__device__ __forceinline__ void window_step(const DecodeParams& p, uint32_t kb, uint32_t vb, int n,
                                            const uint32_t (&bq)[D / 16][2], int lane, int gid, int tig,
                                            WarpState<D>& st) {
  constexpr int RS = win_row_stride<D>();
  float s[4] = {0.f, 0.f, 0.f, 0.f};
  {
    const int r = (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t a[4];
      ldmatrix_x4(a, kb + r * RS + (2 * kk + (lane >> 4)) * 16);
      mma16816_bf16(s, a[0], a[1], a[2], a[3], bq[kk][0], bq[kk][1]);
    }
  }
  const bool v0 = gid < n, v1 = gid + 8 < n;
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
  const float mn0 = fmaxf(st.m0, mx0), mn1 = fmaxf(st.m1, mx1);  // finite: row 0 is valid
  const float a0 = fast_exp2(st.m0 - mn0), a1 = fast_exp2(st.m1 - mn1);
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
      ldmatrix_x4_trans(a, vb + r * RS + (2 * mt + ((lane >> 3) & 1)) * 16);
      mma16816_bf16(st.O[mt], a[0], a[1], a[2], a[3], bh[0], bh[1]);
      mma16816_bf16(st.O[mt], a[0], a[1], a[2], a[3], bl[0], bl[1]);
    }
  }
}

// Bytes of one ring slot: a page item (a G = 32 page, or a staged 32-token
// unit) or 16 window rows at the padded stride, whichever is larger.
template <int D>
__host__ __device__ int64_t line_slot_bytes(const DecodeParams& p) {
  const int64_t page = make_geom(32, D, p.bits).page_bytes;
  const int64_t win = (int64_t)kWinRows * win_row_stride<D>();
  return (page > win ? page : win + 15) / 16 * 16;
}

// Shared memory of one warp: its mbarriers (rounded to 16 bytes), reciprocal
// Key scales (PB pages), queries (GP heads, fp32, the mma_group layout) and
// ring, rounded to 128 bytes; a CTA holds kLineWarps of them.
__host__ __device__ inline size_t line_warp_bytes(int slots, int pb, int gp, int D, int64_t slot_bytes) {
  const size_t b = ((size_t)slots * 8 + 15) / 16 * 16 + ((size_t)pb * D + (size_t)gp * D) * sizeof(float) +
                   (size_t)slots * slot_bytes;
  return (b + 127) / 128 * 128;
}
template <int D>
size_t line_smem(const DecodeParams& p, int slots) {
  const int gp = gqa_pad(p.g);
  return (size_t)kLineWarps * line_warp_bytes(slots, 8 / gp, gp, D, line_slot_bytes<D>(p));
}

template <int D, int BITS, int GP, int MODE>
__global__ void __launch_bounds__(kMmaThreads, 3) decode_line_kernel(const DecodeParams p, int slots) {
  using S = Shape<D, BITS, GP>;
  constexpr int RS = win_row_stride<D>();
  extern __shared__ __align__(128) uint8_t smem[];
  pdl_wait();
  pdl_release();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gid = lane >> 2, tig = lane & 3;
  const int gw = blockIdx.x * kLineWarps + warp;
  const int N = gridDim.x * kLineWarps;
  // positions fit in 32 bits (the host checks the line's length)
  const int64_t C = p.line_start[p.n_seqs];
  const int lo = (int)((int64_t)gw * C / N), hi = (int)((int64_t)(gw + 1) * C / N);
  if (lo >= hi) return;

  // this warp's shared memory
  const int64_t slot_bytes = line_slot_bytes<D>(p);
  uint8_t* wbase = smem + (size_t)warp * line_warp_bytes(slots, S::PB, GP, D, slot_bytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(wbase);
  float* rsc = reinterpret_cast<float*>(wbase + ((size_t)slots * 8 + 15) / 16 * 16);
  float4* q4 = reinterpret_cast<float4*>(rsc + S::PB * D);
  uint8_t* ring = reinterpret_cast<uint8_t*>(rsc + S::PB * D + GP * D);
  const uint32_t bar0 = smem_addr(bars);

  const PageGeom geom = p.geom;
  const int upp = MODE == kStaged ? p.G / 32 : 1;
  const PageGeom ug = MODE == kStaged ? make_geom(32, D, BITS) : geom;
  const int64_t stored = geom.page_bytes;

  if (lane == 0) {
    for (int s = 0; s < slots; ++s) mbar_init(bar0 + 8 * s, 1);
    fence_mbar_init();
  }
  __syncwarp();

  // ---- issue side: the warp's items in line order into the ring ------------------
  // Per unit: its pages [ipg, ipg + ipn) (32-token items) and window steps
  // [iws, iws + iwn); the next unit starts at line position ix.
  int ix = lo;
  int ib = 0, ih = 0, ipn = 0, iwn = 0, iws = 0, ipg = 0;
  const uint8_t* isrc = nullptr;  // contiguous G = 32: the next page
  auto next_unit = [&]() {
    while ((ipn | iwn) == 0 && ix < hi) {
      const LineUnitAt ua = line_unit_at(p, ix);
      const int e = min(ua.start + ua.u.cost, hi);
      const int a = ix - ua.start, z = e - ua.start;
      ib = p.seq_begin + ua.i;
      ih = ua.h;
      ipg = min(a, ua.u.U);
      ipn = min(z, ua.u.U) - ipg;
      iws = a <= ua.u.U ? 0 : (a - ua.u.U + kWinWeight - 1) / kWinWeight;
      iwn = (z <= ua.u.U ? 0 : (z - ua.u.U + kWinWeight - 1) / kWinWeight) - iws;
      if (MODE == kFlat32) isrc = p.pages + page_offset(p.map, stored, ib, ih, ipg);
      ix = e;
    }
  };
  int islot = 0, free_slots = slots;
  // Slots are refilled once the warp has read them (a __syncwarp before each
  // refill); each issuing lane orders its earlier shared-memory reads before
  // its copies with one proxy fence per refill.
  auto refill = [&]() {
    next_unit();
    bool fenced = false;
    while (true) {
      if (ipn > 0) {
        if (free_slots < 1) break;
        const uint32_t bar = bar0 + 8 * islot, dst = smem_addr(ring + (size_t)islot * slot_bytes);
        if (lane == 0) {
          if (!fenced) fence_proxy_async();
          fenced = true;
          mbar_expect_tx(bar, (uint32_t)ug.page_bytes);
          if constexpr (MODE == kFlat32) {
            bulk_load(dst, isrc, (uint32_t)stored, bar);
          } else if constexpr (MODE == kPaged32) {
            bulk_load(dst, p.pages + page_offset(p.map, stored, ib, ih, ipg), (uint32_t)stored, bar);
          } else {
            const int pg = ipg / upp, sub = ipg - pg * upp;
            const uint8_t* src = p.pages + page_offset(p.map, stored, ib, ih, pg);
            bulk_load(dst, src + sub * 32 * S::kRowBytes, 32 * S::kRowBytes, bar);
            bulk_load(dst + (uint32_t)ug.code_bytes, src + geom.code_bytes + sub * S::kSubBytes, S::kSubBytes,
                      bar);
            bulk_load(dst + (uint32_t)ug.kscale_off, src + geom.kscale_off, 4 * D, bar);
            bulk_load(dst + (uint32_t)ug.vscale_off, src + geom.vscale_off + 128 * sub, 128, bar);
          }
        }
        if (MODE == kFlat32) isrc += stored;
        else ++ipg;
        --ipn;
        islot = islot + 1 == slots ? 0 : islot + 1;
        free_slots -= 1;
      } else if (iwn > 0) {
        if (free_slots < 2) break;
        const int s1 = islot + 1 == slots ? 0 : islot + 1;
        const int i = ib - p.seq_begin;
        const int64_t Q0 = p.ctr[i].quantized, T0 = p.ctr[i].total;
        const int n = (int)min((int64_t)kWinRows, T0 - Q0 - (int64_t)kWinRows * iws);
        const uint32_t bk = bar0 + 8 * islot, bv = bar0 + 8 * s1;
        if (lane == 0) {
          mbar_expect_tx(bk, (uint32_t)(n * 2 * D));
          mbar_expect_tx(bv, (uint32_t)(n * 2 * D));
        }
        __syncwarp();
        const int r = lane & 15;
        if (r < n) {
          const int64_t unit = (int64_t)ib * p.Hkv + ih;
          const int64_t row = ((Q0 + (int64_t)kWinRows * iws + r) % p.Rcap) * D;
          const bool isv = lane >= 16;
          const __nv_bfloat16* src =
              reinterpret_cast<const __nv_bfloat16*>(isv ? p.ring_v : p.ring_k) + unit * p.Rcap * D + row;
          const uint32_t dst = smem_addr(ring + (size_t)(isv ? s1 : islot) * slot_bytes) + r * RS;
          if (!fenced) fence_proxy_async();
          bulk_load(dst, src, 2 * D, isv ? bv : bk);
        }
        fenced = true;
        ++iws;
        --iwn;
        islot = s1 + 1 == slots ? 0 : s1 + 1;
        free_slots -= 2;
      } else {
        break;
      }
      next_unit();
    }
  };
  refill();

  // ---- consume side --------------------------------------------------------------
  int cslot = 0;
  uint32_t phases = 0;
  bool ok = true;
  auto wait_slot = [&](int s) {
    if (ok) ok = mbar_wait(bar0 + 8 * s, (phases >> s) & 1u);
    phases ^= 1u << s;
  };
  auto release = [&](int k) {
    cslot += k;
    if (cslot >= slots) cslot -= slots;
    free_slots += k;
    __syncwarp();
    refill();
  };

  WarpState<D> st;
  // every unit whose positions meet [lo, hi) gets a partial from this warp (an
  // empty one if no item starts here), so a unit's slots are exactly the warps
  // from the one holding its first position to the one holding its last
  for (int x = lo; x < hi;) {
    const LineUnitAt ua = line_unit_at(p, x);
    const int i = ua.i, h = ua.h, b = p.seq_begin + i;
    const LineUnit U = ua.u;
    const int ustart = ua.start;
    const int uend = min(ustart + U.cost, hi);
    const int la = x - ustart, lz = uend - ustart;
    x = uend;
    // this warp's items of the unit: pages [pa, pz) and window steps [wa, wz)
    const int pa = min(la, U.U), pz = min(lz, U.U);
    const int wa = la <= U.U ? 0 : (la - U.U + kWinWeight - 1) / kWinWeight;
    const int wz = lz <= U.U ? 0 : (lz - U.U + kWinWeight - 1) / kWinWeight;
    const int64_t unit = (int64_t)b * p.Hkv + h;
    const int slot = gw - line_warp_of(ustart, C, N);
    float* part = p.partials + (unit * p.max_splits + slot) * (int64_t)p.g * part_row(D);
    const __nv_bfloat16* qrow = reinterpret_cast<const __nv_bfloat16*>(p.q) + ((int64_t)b * p.Hq + (int64_t)h * p.g) * D;
    // queries (head n % g for the padding heads), pre-scaled, in the layout of
    // mma_group; their largest magnitude for the range test
    float qa = 0.f;
    for (int idx = lane; idx < GP * D; idx += 32) {
      const int n = idx / D, c = idx - n * D;
      const float qv = __bfloat162float(qrow[(int64_t)(n % p.g) * D + c]) * p.qk_scale;
      qa = fmaxf(qa, fabsf(qv));
      const int tg = c / S::kChan, i4 = (c - tg * S::kChan) >> 2;
      reinterpret_cast<float*>(q4)[((i4 * GP + n) * 4 + tg) * 4 + (c & 3)] = qv;
    }
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) qa = fmaxf(qa, __shfl_xor_sync(0xffffffffu, qa, off));
    __syncwarp();
    bool plain;
    {
      const int qexp = float_exp2i(qa);
      const float kthr = fmaxf(pow2i(BITS == 2 ? qexp + 1 + 4 - 14 : qexp + 1 - 9), p.eps);
      const float kabs = p.range ? __uint_as_float(p.range[2 * unit]) : 0.f;
      const float vabs = p.range ? __uint_as_float(p.range[2 * unit + 1]) : 0.f;
      plain = fmaxf(kabs, p.eps) * kthr <= (float)p.qmax * 0.9999f && vabs <= kVWideAbs * 0.999f;
    }
    if (!plain) {
      // this warp's part of the unit on the CUDA cores; its ring items are
      // waited for and released unread
      const int64_t W = p.ctr[i].total - p.ctr[i].quantized;
      const int64_t Q0 = p.ctr[i].quantized;
      line_unit_cuda_cores<D, BITS>(p.pages, p.map, geom,
                                    reinterpret_cast<const __nv_bfloat16*>(p.ring_k) + unit * p.Rcap * D,
                                    reinterpret_cast<const __nv_bfloat16*>(p.ring_v) + unit * p.Rcap * D, qrow,
                                    part, p.g, p.G, p.Rcap, Q0, p.eps, p.qk_scale, b, h, pa, pz,
                                    (int)min((int64_t)kWinRows * wa, W), (int)min((int64_t)kWinRows * wz, W));
      for (int k = pa; k < pz; ++k) {
        wait_slot(cslot);
        __syncwarp();
        release(1);
      }
      for (int k = wa; k < wz; ++k) {
        wait_slot(cslot);
        wait_slot(cslot + 1 == slots ? 0 : cslot + 1);
        __syncwarp();
        release(2);
      }
      continue;
    }

#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) st.O[mt][0] = st.O[mt][1] = st.O[mt][2] = st.O[mt][3] = 0.f;
    st.C[0] = st.C[1] = st.C[2] = st.C[3] = 0.f;
    st.m0 = st.m1 = -INFINITY;
    st.l0 = st.l1 = 0.f;
    // ---- page items: groups of up to PB consecutive items
    for (int k = pa; k < pz; k += S::PB) {
      const int np = min(S::PB, pz - k);
      const uint8_t* pgs[S::PB];
#pragma unroll
      for (int j = 0; j < S::PB; ++j) {
        int t = cslot + (j < np ? j : np - 1);
        if (t >= slots) t -= slots;
        pgs[j] = ring + (size_t)t * slot_bytes;
        if (j < np) wait_slot(t);
      }
      if (!ok) break;
      if (np == S::PB)
        mma_group<D, BITS, GP, true>(pgs, np, ug, 32, q4, rsc, lane, gid, tig, st);
      else
        mma_group<D, BITS, GP, false>(pgs, np, ug, 32, q4, rsc, lane, gid, tig, st);
      __syncwarp();
      release(np);
    }
    const bool pages_open = pz > pa;
    // ---- close the page part: undo the code bias, fold the page streams
    auto close_pages = [&]() {
      constexpr float kTwo24 = 16777216.f;
      const float c0 = S::kBias * kTwo24 * st.C[0], c1 = S::kBias * kTwo24 * st.C[1];
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        st.O[mt][0] = fmaf(st.O[mt][0], kTwo24, -c0);
        st.O[mt][1] = fmaf(st.O[mt][1], kTwo24, -c1);
        st.O[mt][2] = fmaf(st.O[mt][2], kTwo24, -c0);
        st.O[mt][3] = fmaf(st.O[mt][3], kTwo24, -c1);
      }
#pragma unroll
      for (int off = GP / 2; off < 4; off <<= 1) merge_streams<D>(st, off);
    };
    if (pages_open) close_pages();
    // ---- window steps
    if (ok && wz > wa) {
      uint32_t bq[D / 16][2];
      {
        const __nv_bfloat16* qh = qrow + (int64_t)((gid % GP) % p.g) * D;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          bq[kk][0] = *reinterpret_cast<const uint32_t*>(qh + 16 * kk + 2 * tig);
          bq[kk][1] = *reinterpret_cast<const uint32_t*>(qh + 16 * kk + 2 * tig + 8);
        }
      }
      const int64_t W = p.ctr[i].total - p.ctr[i].quantized;
      for (int step = wa; step < wz; ++step) {
        const int n = (int)min((int64_t)kWinRows, W - (int64_t)kWinRows * step);
        const int s0 = cslot, s1 = cslot + 1 == slots ? 0 : cslot + 1;
        wait_slot(s0);
        wait_slot(s1);
        if (!ok) break;
        uint8_t* kb = ring + (size_t)s0 * slot_bytes;
        uint8_t* vb = ring + (size_t)s1 * slot_bytes;
        if (n < kWinRows) {
          // rows past the window: zero Values (their p is 0; stale bytes could be inf)
          for (int idx = lane; idx < (kWinRows - n) * (2 * D / 16); idx += 32) {
            const int r = n + idx / (2 * D / 16), c16 = idx % (2 * D / 16);
            *reinterpret_cast<uint4*>(vb + r * RS + c16 * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
          __syncwarp();
        }
        window_step<D, GP>(p, smem_addr(kb), smem_addr(vb), n, bq, lane, gid, tig, st);
        __syncwarp();
        release(2);
      }
    }
    if (!ok) break;
    // ---- the partial of (unit, this warp): l summed over the warp's rows
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      st.l0 += __shfl_xor_sync(0xffffffffu, st.l0, off);
      st.l1 += __shfl_xor_sync(0xffffffffu, st.l1, off);
    }
    const int hd0 = 2 * tig, hd1 = 2 * tig + 1;
    if (2 * tig < GP) {
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        const int c_lo = 16 * mt + gid;
        if (hd0 < p.g) {
          part[(int64_t)hd0 * part_row(D) + c_lo] = st.O[mt][0];
          part[(int64_t)hd0 * part_row(D) + c_lo + 8] = st.O[mt][2];
        }
        if (hd1 < p.g) {
          part[(int64_t)hd1 * part_row(D) + c_lo] = st.O[mt][1];
          part[(int64_t)hd1 * part_row(D) + c_lo + 8] = st.O[mt][3];
        }
      }
      if (gid == 0) {
        if (hd0 < p.g) {
          part[(int64_t)hd0 * part_row(D) + D] = st.m0;
          part[(int64_t)hd0 * part_row(D) + D + 1] = st.l0;
        }
        if (hd1 < p.g) {
          part[(int64_t)hd1 * part_row(D) + D] = st.m1;
          part[(int64_t)hd1 * part_row(D) + D + 1] = st.l1;
        }
      }
    }
  }
  if (!ok) {
    // a bounded wait gave up: report, and leave nothing in flight
    if (lane == 0) atomicOr(p.status, kStatusWaitTimeout);
    while (free_slots < slots) {
      mbar_wait(bar0 + 8 * cslot, (phases >> cslot) & 1u);
      phases ^= 1u << cslot;
      cslot = cslot + 1 == slots ? 0 : cslot + 1;
      ++free_slots;
    }
  }
}

// CTAs of the line kernel one SM holds (0 on error) and the launch.
template <int D, int BITS, int GP, int MODE>
int line_resident_t(const DecodeParams& p, int slots) {
  const size_t smem = line_smem<D>(p, slots);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  static size_t configured[64] = {};
  // (shared memory bytes << 8 | CTAs per SM), one word so that concurrent
  // callers never see one query's size with another's answer
  static std::atomic<uint64_t> known[64];
  const uint64_t k = known[dev].load(std::memory_order_relaxed);
  if ((k & 0xFFu) != 0 && (k >> 8) == (uint64_t)smem) return (int)(k & 0xFFu);
  if (smem > configured[dev]) {
    if (cudaFuncSetAttribute(decode_line_kernel<D, BITS, GP, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return 0;
    configured[dev] = smem;
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_line_kernel<D, BITS, GP, MODE>, kMmaThreads,
                                                    smem) != cudaSuccess)
    return 0;
  if (per_sm > 0 && per_sm < 256) known[dev].store((uint64_t)smem << 8 | (uint64_t)per_sm, std::memory_order_relaxed);
  return per_sm;
}

// Slots of each warp's ring: at least two page groups' worth and a window
// step's two, within about 57 KB of ring per CTA.
template <int D>
int line_slots(const DecodeParams& p) {
  const int pb = 8 / gqa_pad(p.g);
  int slots = (int)(57 * 1024 / (kLineWarps * line_slot_bytes<D>(p)));
  if (slots < pb + 1) slots = pb + 1;
  if (slots < 3) slots = 3;
  if (slots > 8) slots = 8;
  return slots;
}

// Query (launch = false: CTAs per SM into *per_sm) or launch the kernel with
// p.line_warps / kLineWarps CTAs.
template <int D, int BITS, int GP, int MODE>
cudaError_t line_t(const DecodeParams& p, bool launch, cudaStream_t s, int* per_sm) {
  const int slots = line_slots<D>(p);
  if (!launch) {
    *per_sm = line_resident_t<D, BITS, GP, MODE>(p, slots);
    return *per_sm > 0 ? cudaSuccess : cudaErrorInvalidConfiguration;
  }
  return launch_pdl(decode_line_kernel<D, BITS, GP, MODE>, dim3(p.line_warps / kLineWarps), dim3(kMmaThreads),
                    line_smem<D>(p, slots), s, p, slots);
}

template <int D, int BITS, int GP>
cudaError_t line_m(const DecodeParams& p, bool launch, cudaStream_t s, int* per_sm) {
  if (p.G != 32) return line_t<D, BITS, GP, kStaged>(p, launch, s, per_sm);
  return p.map.table ? line_t<D, BITS, GP, kPaged32>(p, launch, s, per_sm)
                     : line_t<D, BITS, GP, kFlat32>(p, launch, s, per_sm);
}

template <int D, int BITS>
cudaError_t line_g(const DecodeParams& p, bool launch, cudaStream_t s, int* per_sm) {
  switch (gqa_pad(p.g)) {
    case 2: return line_m<D, BITS, 2>(p, launch, s, per_sm);
    case 4: return line_m<D, BITS, 4>(p, launch, s, per_sm);
    default: return line_m<D, BITS, 8>(p, launch, s, per_sm);
  }
}

}  // namespace
}  // namespace kvq
