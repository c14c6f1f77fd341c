// Host side of libkvq: the C ABI of include/kvq.h.
//
// Bookkeeping follows "54. KV Cache Quantization Strategies" (append_and_partition:
// total / quantized / flushed counters, validation of the inputs) with the
// grouped flush rule; the byte ledger follows "KV Cache 量化与压缩" sections 01/05.
// Counters live on the host and travel to the kernels in the launch parameter
// block, so no call synchronizes with the device.

#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/kvq.h"
#include "kvq_internal.h"

using kvq::SeqCounters;

struct kvq_cache {
  kvq_config cfg;
  int bits;
  int esize;        // bytes per window / input element
  int rcap;         // ring rows per unit
  int g;            // query heads per KV head
  kvq::PageGeom geom;
  std::vector<int64_t> cap;         // per sequence
  std::vector<int64_t> pages_cap;   // group pages per unit, per sequence
  std::vector<int64_t> page_base;   // byte offset of (seq, head 0, page 0)
  std::vector<int32_t> total, quantized, last_flushed;
  // paged mode: a pool of blocks (one group of a sequence, every KV head) and
  // a block table per sequence; free_blocks is a stack of block ids
  bool paged;
  int64_t pool_blocks;
  int32_t table_stride;                      // table entries per sequence
  int32_t* table;                            // device [batch][table_stride]
  std::vector<int32_t> free_blocks;
  std::vector<std::vector<int32_t>> blocks;  // host copy of each sequence's table
  // segmented mode (the whole overflow of an append is one segment): token-major
  // codes and scales; cfg.group is 1 inside (a "page" is one token)
  bool segmented;
  kvq::SegArrays seg;
  uint32_t* kmax;                            // device [batch][Hkv][D]
  std::vector<std::vector<int32_t>> seg_starts;  // first token of each segment
  int max_splits;
  int min_chunk_pages;
  int n_sm;
  int device;
  // arena
  uint8_t* base;
  size_t arena_bytes;
  int32_t* status;
  uint32_t* range;  // [batch][Hkv][2]: largest flushed Key / Value absmax (null: segmented)
  uint32_t* done;   // [batch][Hkv]: finished split items of the running decode (null: segmented)
  kvq::SeqLayout* layout;
  uint8_t* pages;
  void* ring_k;
  void* ring_v;
  float* partials;
};

namespace {

thread_local std::string g_err;
std::atomic<uint64_t> g_launches{0};

kvq_status fail(kvq_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return st;
}

kvq_status cuda_fail(cudaError_t e, const char* what) {
  return fail(KVQ_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr int64_t kMinChunkTokens = 256;
constexpr size_t kAlign = 256;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

kvq_status check_config(const kvq_config* c) {
  if (!c) return fail(KVQ_EINVAL, "config is NULL");
  if (c->batch < 1) return fail(KVQ_EINVAL, "batch must be >= 1 (got %d)", c->batch);
  if (c->n_kv_heads < 1) return fail(KVQ_EINVAL, "n_kv_heads must be >= 1");
  if (c->n_q_heads < 1 || c->n_q_heads % c->n_kv_heads != 0)
    return fail(KVQ_EINVAL, "n_q_heads (%d) must be a positive multiple of n_kv_heads (%d)", c->n_q_heads,
                c->n_kv_heads);
  if (c->n_q_heads / c->n_kv_heads > kvq::kMaxGqa)
    return fail(KVQ_EUNSUPPORTED, "query heads per KV head must be <= %d", kvq::kMaxGqa);
  if (c->head_dim < 16 || c->head_dim > 256 || c->head_dim % 16 != 0)
    return fail(KVQ_EUNSUPPORTED, "head_dim must be a multiple of 16 in [16, 256] (got %d)", c->head_dim);
  if (c->residual_len <= 0) return fail(KVQ_EINVAL, "residual_length must be positive");
  if (c->group <= 0 || c->group % 8 != 0)
    return fail(KVQ_EUNSUPPORTED, "group must be a positive multiple of 8 (got %d)", c->group);
  if (c->qmax < 1 || c->qmax > 127) return fail(KVQ_EINVAL, "qmax must be in [1, 127] (got %d)", c->qmax);
  if (c->dtype != KVQ_BF16 && c->dtype != KVQ_FP32) return fail(KVQ_EINVAL, "unknown dtype %d", c->dtype);
  if (!(c->eps > 0.f) || !std::isfinite(c->eps)) return fail(KVQ_EINVAL, "eps must be positive and finite");
  const size_t flush_smem = kvq::flush_smem_bytes(c->group, c->head_dim, c->dtype == KVQ_BF16 ? 2 : 4);
  if (flush_smem > kvq::kFlushSmemMax)
    return fail(KVQ_EUNSUPPORTED, "group * head_dim too large for one flush tile (%zu bytes)", flush_smem);
  return KVQ_OK;
}

// Bits of one stored code: 2 (KIVI's 2-bit codes, qmax 1), 4 or 8.
int bits_of(const kvq_config* c) { return c->qmax <= 1 ? 2 : c->qmax <= 7 ? 4 : 8; }
int esize_of(const kvq_config* c) { return c->dtype == KVQ_BF16 ? 2 : 4; }
int rcap_of(const kvq_config* c) {
  return c->group * ((c->residual_len + c->group - 1) / c->group + 1);
}

struct ArenaPlan {
  size_t status, range, done, layout, table, pages, ring_k, ring_v, partials, total;
  std::vector<int64_t> pages_cap, page_base;
  int max_splits, min_chunk_pages;
  int32_t table_stride;
};

// Arena of a contiguous cache (pool_blocks = 0: each sequence's pages at a
// fixed place, sized by its capacity) or a paged one (pool_blocks > 0: a
// shared pool of blocks and a block table row per sequence, as long as its
// capacity in groups).
kvq_status plan_arena(const kvq_config* c, const int64_t* cap, ArenaPlan* a, int64_t pool_blocks = 0) {
  if (!cap) return fail(KVQ_EINVAL, "capacity_per_seq is NULL");
  const kvq::PageGeom geom = kvq::make_geom(c->group, c->head_dim, bits_of(c));
  a->pages_cap.assign(c->batch, 0);
  a->page_base.assign(c->batch, 0);
  int64_t pmax = 0, off = 0;
  for (int b = 0; b < c->batch; ++b) {
    if (cap[b] < 1 || cap[b] >= (int64_t(1) << 31))
      return fail(KVQ_EINVAL, "capacity of sequence %d must be in [1, 2^31) (got %lld)", b, (long long)cap[b]);
    a->pages_cap[b] = cap[b] / c->group;
    a->page_base[b] = pool_blocks > 0 ? 0 : off;
    off += (int64_t)c->n_kv_heads * a->pages_cap[b] * geom.page_bytes;
    pmax = std::max(pmax, a->pages_cap[b]);
  }
  a->table_stride = (int32_t)std::max<int64_t>(1, pmax);
  if (pool_blocks > 0) off = pool_blocks * c->n_kv_heads * geom.page_bytes;
  a->min_chunk_pages = (int)std::max<int64_t>(1, (kMinChunkTokens + c->group - 1) / c->group);
  a->max_splits = (int)((pmax + a->min_chunk_pages - 1) / a->min_chunk_pages) + 1;
  const int g = c->n_q_heads / c->n_kv_heads;
  const size_t units = (size_t)c->batch * c->n_kv_heads;
  size_t o = 0;
  a->status = o;
  o = align_up(o + sizeof(int32_t), kAlign);
  a->range = o;
  o = align_up(o + units * 2 * sizeof(uint32_t), kAlign);
  a->done = o;
  o = align_up(o + units * sizeof(uint32_t), kAlign);
  a->layout = o;
  o = align_up(o + (size_t)c->batch * sizeof(kvq::SeqLayout), kAlign);
  a->table = o;
  if (pool_blocks > 0) o = align_up(o + (size_t)c->batch * a->table_stride * sizeof(int32_t), kAlign);
  a->pages = o;
  o = align_up(o + (size_t)off, kAlign);
  const size_t ring = units * rcap_of(c) * c->head_dim * esize_of(c);
  a->ring_k = o;
  o = align_up(o + ring, kAlign);
  a->ring_v = o;
  o = align_up(o + ring, kAlign);
  a->partials = o;
  o = align_up(o + units * a->max_splits * g * kvq::part_row(c->head_dim) * sizeof(float), kAlign);
  a->total = o;
  return KVQ_OK;
}

// Arena of a segmented cache: token-major Key and Value code rows and scales
// for capacity_max tokens per unit, the segment maxima, rings of R rows and
// the split partials.
struct SegPlan {
  size_t status, range, layout, kcodes, vcodes, kscales, vscales, first, kmax, ring_k, ring_v, partials, total;
  int64_t cap;
  int max_splits;
};

kvq_status plan_arena_seg(const kvq_config* c, const int64_t* cap, SegPlan* a) {
  if (!cap) return fail(KVQ_EINVAL, "capacity_per_seq is NULL");
  int64_t cmax = 1;
  for (int b = 0; b < c->batch; ++b) {
    if (cap[b] < 1 || cap[b] >= (int64_t(1) << 31))
      return fail(KVQ_EINVAL, "capacity of sequence %d must be in [1, 2^31) (got %lld)", b, (long long)cap[b]);
    cmax = std::max(cmax, cap[b]);
  }
  // rows of 32 tokens start on 16-byte boundaries in every per-unit array
  // (the tensor-core kernel copies them whole)
  a->cap = (cmax + 31) / 32 * 32;
  a->max_splits = (int)((cmax + kMinChunkTokens - 1) / kMinChunkTokens) + 1;
  const size_t units = (size_t)c->batch * c->n_kv_heads, D = c->head_dim;
  const size_t rows = units * (size_t)a->cap;
  const int g = c->n_q_heads / c->n_kv_heads;
  size_t o = 0;
  a->status = o;
  o = align_up(o + sizeof(int32_t), kAlign);
  a->range = o;
  o = align_up(o + units * 2 * sizeof(uint32_t), kAlign);
  a->layout = o;
  o = align_up(o + (size_t)c->batch * sizeof(kvq::SeqLayout), kAlign);
  a->kcodes = o;
  o = align_up(o + rows * D * bits_of(c) / 8, kAlign);
  a->vcodes = o;
  o = align_up(o + rows * D * bits_of(c) / 8, kAlign);
  a->kscales = o;
  o = align_up(o + rows * D * sizeof(float), kAlign);
  a->vscales = o;
  o = align_up(o + rows * sizeof(float), kAlign);
  a->first = o;
  o = align_up(o + (size_t)c->batch * (size_t)a->cap * sizeof(int32_t), kAlign);
  a->kmax = o;
  o = align_up(o + units * D * sizeof(uint32_t), kAlign);
  const size_t ring = units * (size_t)c->residual_len * D * esize_of(c);
  a->ring_k = o;
  o = align_up(o + ring, kAlign);
  a->ring_v = o;
  o = align_up(o + ring, kAlign);
  a->partials = o;
  o = align_up(o + units * a->max_splits * g * kvq::part_row((int)D) * sizeof(float), kAlign);
  a->total = o;
  return KVQ_OK;
}

bool aligned16(const void* p) { return p && ((uintptr_t)p & 15u) == 0; }

kvq::PageMap page_map(const kvq_cache* c) {
  kvq::PageMap m;
  m.layout = c->layout;
  m.table = c->table;
  m.table_stride = c->table_stride;
  m.block_bytes = (int64_t)c->cfg.n_kv_heads * c->geom.page_bytes;
  return m;
}

void fill_counters(const kvq_cache* c, int seq_begin, int n, SeqCounters* out) {
  for (int i = 0; i < n; ++i) {
    out[i].total = c->total[seq_begin + i];
    out[i].quantized = c->quantized[seq_begin + i];
  }
}

// Split plan for the decode launch over sequences [s0, s0 + n).  ``slots``:
// the CTAs of the split kernel the GPU holds at once (0 if unknown).
void plan_splits(const kvq_cache* c, int s0, int n, int requested, int slots, int* chunk, int* grid_splits) {
  int64_t total_pages = 0, pmax = 0;
  for (int i = s0; i < s0 + n; ++i) {
    const int64_t P = c->quantized[i] / c->cfg.group;
    total_pages += P * c->cfg.n_kv_heads;
    pmax = std::max(pmax, P);
  }
  int64_t ch;
  if (requested > 0) {
    ch = requested;
  } else {
    // about 6 work items per SM for group pages, 8 for a segmented cache's
    // one-token pages (CUDA-core kernel).  Measured on the 32 x 8 x 8192
    // decode layer (CUDA events, split + combine): 6 per SM makes the chunk
    // 72 pages (three columns of 72 and a half column of 36, so the last wave
    // is short) and the split 78.1 -> 74.8 us; 8 per SM (chunk 56) and chunks
    // of 64 or 68 (a nearly full last column) are slower.  The segmented
    // decode is 2.8 % faster at 8 per SM.
    const int64_t target = (int64_t)c->n_sm * (c->segmented ? 8 : 6);
    ch = std::max<int64_t>(c->min_chunk_pages, (total_pages + target - 1) / target);
  }
  // Few units (at least 4 split columns per wave): choose the columns so that
  // the launch, its window items included, fills whole waves of the resident
  // CTAs -- half the waves the plan above would take, at least one, since
  // equal items need no later waves to even out.  A launch only a few CTAs
  // past a wave boundary takes about a whole CTA longer: on the long-video
  // decode (8 units of 3373 pages of G = 128, 456 resident CTAs) 59 columns
  // (472 CTAs) took 162 us, 113 columns (912, two waves) 116 us and 56 (456,
  // one wave) 114 us, against 121 us for the 106 columns above.
  const int64_t units = (int64_t)n * c->cfg.n_kv_heads;
  if (requested <= 0 && slots > 0 && units * 4 <= slots && pmax > 0) {
    const int64_t base_ctas = units * ((pmax + ch - 1) / ch + 1);
    const int64_t waves = std::max<int64_t>(1, base_ctas / (2 * (int64_t)slots));
    const int64_t cols = waves * slots / units - 1;
    if (cols >= 1) ch = std::max<int64_t>(c->min_chunk_pages, (pmax + cols - 1) / cols);
  }
  ch = std::max<int64_t>(ch, (pmax + c->max_splits - 2) / std::max(1, c->max_splits - 1));
  ch = std::max<int64_t>(ch, 1);
  // whole page groups for each of the tensor-core kernel's 4 warps (8 pages =
  // 4 warps x 2 pages at g = 4): every warp of a CTA gets the same work.  A
  // larger G is split into 32-token units, four warps' worth per page or more,
  // so any chunk keeps the warps even there.
  if (requested <= 0 && ch > 8 && c->cfg.group == 32) ch = (ch + 7) / 8 * 8;
  // a segmented cache's tokens go to the tensor-core kernel in 32-token
  // tiles, four warps' worth an item (the CUDA-core kernel takes any chunk)
  if (c->segmented) ch = (ch + 127) / 128 * 128;
  *chunk = (int)ch;
  *grid_splits = (int)((pmax + ch - 1) / ch);
}

// Kernels launch on the current device, and the cache's arena lives on
// c->device: a launch on another device would read or write the wrong GPU's
// memory, so every launching entry point refuses it first.
kvq_status check_device(const kvq_cache* c) {
  int cur = -1;
  const cudaError_t e = cudaGetDevice(&cur);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (cur != c->device)
    return fail(KVQ_EINVAL, "the current device is %d but the cache lives on device %d", cur, c->device);
  return KVQ_OK;
}

void base_decode_params(const kvq_cache* c, kvq::DecodeParams* p) {
  memset(p, 0, sizeof *p);
  p->D = c->cfg.head_dim;
  p->Hkv = c->cfg.n_kv_heads;
  p->Hq = c->cfg.n_q_heads;
  p->g = c->g;
  p->G = c->cfg.group;
  p->Rcap = c->rcap;
  p->bits = c->bits;
  p->qmax = c->cfg.qmax;
  p->eps = c->cfg.eps;
  p->qk_scale = (float)(1.4426950408889634 / std::sqrt((double)c->cfg.head_dim));
  p->geom = c->geom;
  p->pages = c->pages;
  p->map = page_map(c);
  p->seg = c->seg;
  p->ring_k = c->ring_k;
  p->ring_v = c->ring_v;
  p->partials = c->partials;
  p->max_splits = c->max_splits;
  p->status = c->status;
  p->range = c->range;
}

}  // namespace

extern "C" {

const char* kvq_last_error(void) { return g_err.c_str(); }

uint64_t kvq_kernel_launches(void) { return g_launches.load(); }

size_t kvq_page_bytes(const kvq_config* cfg) {
  if (check_config(cfg) != KVQ_OK) return 0;
  return (size_t)kvq::make_geom(cfg->group, cfg->head_dim, bits_of(cfg)).page_bytes;
}

}  // extern "C"

namespace {

kvq_status required_bytes(const kvq_config* cfg, const int64_t* capacity_per_seq, int64_t pool_blocks,
                          size_t* out_bytes) {
  if (!out_bytes) return fail(KVQ_EINVAL, "out_bytes is NULL");
  kvq_status st = check_config(cfg);
  if (st != KVQ_OK) return st;
  ArenaPlan a;
  st = plan_arena(cfg, capacity_per_seq, &a, pool_blocks);
  if (st != KVQ_OK) return st;
  *out_bytes = a.total;
  return KVQ_OK;
}

kvq_status create(const kvq_config* cfg, const int64_t* capacity_per_seq, int64_t pool_blocks, void* device_mem,
                  size_t device_bytes, kvq_cache** out, bool segmented = false) {
  if (!out) return fail(KVQ_EINVAL, "out is NULL");
  *out = nullptr;
  kvq_status st = check_config(cfg);
  if (st != KVQ_OK) return st;
  ArenaPlan a;
  st = plan_arena(cfg, capacity_per_seq, &a, pool_blocks);
  if (st != KVQ_OK) return st;
  SegPlan sp{};
  if (segmented && (st = plan_arena_seg(cfg, capacity_per_seq, &sp)) != KVQ_OK) return st;
  const size_t need = segmented ? sp.total : a.total;
  if (!device_mem || ((uintptr_t)device_mem & (kAlign - 1)))
    return fail(KVQ_EINVAL, "device_mem must be a 256-byte aligned device pointer");
  if (device_bytes < need)
    return fail(KVQ_ENOMEM, "arena of %zu bytes is smaller than the %zu bytes required", device_bytes, need);
  cudaPointerAttributes attr;
  cudaError_t e = cudaPointerGetAttributes(&attr, device_mem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaPointerGetAttributes");
  if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
    return fail(KVQ_EINVAL, "device_mem is not device memory");

  kvq_cache* c = new kvq_cache();
  c->cfg = *cfg;
  c->bits = bits_of(cfg);
  c->esize = esize_of(cfg);
  c->rcap = rcap_of(cfg);
  c->g = cfg->n_q_heads / cfg->n_kv_heads;
  c->geom = kvq::make_geom(cfg->group, cfg->head_dim, c->bits);
  c->cap.assign(capacity_per_seq, capacity_per_seq + cfg->batch);
  c->pages_cap = a.pages_cap;
  c->page_base = a.page_base;
  c->total.assign(cfg->batch, 0);
  c->quantized.assign(cfg->batch, 0);
  c->last_flushed.assign(cfg->batch, 0);
  c->max_splits = a.max_splits;
  c->min_chunk_pages = a.min_chunk_pages;
  c->paged = pool_blocks > 0;
  c->pool_blocks = pool_blocks;
  c->table_stride = a.table_stride;
  c->blocks.assign(cfg->batch, {});
  for (int64_t blk = pool_blocks - 1; blk >= 0; --blk) c->free_blocks.push_back((int32_t)blk);
  c->device = attr.device;
  int cur = 0;
  cudaGetDevice(&cur);
  if (cur != attr.device) cudaSetDevice(attr.device);
  e = cudaDeviceGetAttribute(&c->n_sm, cudaDevAttrMultiProcessorCount, attr.device);
  if (e != cudaSuccess) {
    delete c;
    return cuda_fail(e, "cudaDeviceGetAttribute");
  }
  c->base = static_cast<uint8_t*>(device_mem);
  c->arena_bytes = device_bytes;
  c->status = reinterpret_cast<int32_t*>(c->base + a.status);
  c->range = reinterpret_cast<uint32_t*>(c->base + a.range);
  c->done = reinterpret_cast<uint32_t*>(c->base + a.done);
  c->layout = reinterpret_cast<kvq::SeqLayout*>(c->base + a.layout);
  c->table = c->paged ? reinterpret_cast<int32_t*>(c->base + a.table) : nullptr;
  c->pages = c->base + a.pages;
  c->ring_k = c->base + a.ring_k;
  c->ring_v = c->base + a.ring_v;
  c->partials = reinterpret_cast<float*>(c->base + a.partials);
  if (segmented) {
    // a "page" is one token: group 1 inside, rings of R rows
    c->segmented = true;
    c->cfg.group = 1;
    c->rcap = cfg->residual_len;
    c->geom = kvq::make_geom(1, cfg->head_dim, c->bits);
    c->max_splits = sp.max_splits;
    c->min_chunk_pages = (int)kMinChunkTokens;
    c->seg.kcodes = c->base + sp.kcodes;
    c->seg.vcodes = c->base + sp.vcodes;
    c->seg.kscales = reinterpret_cast<float*>(c->base + sp.kscales);
    c->seg.vscales = reinterpret_cast<float*>(c->base + sp.vscales);
    c->seg.first = reinterpret_cast<int32_t*>(c->base + sp.first);
    c->seg.cap = sp.cap;
    c->seg.row_bytes = cfg->head_dim * c->bits / 8;
    c->kmax = reinterpret_cast<uint32_t*>(c->base + sp.kmax);
    c->status = reinterpret_cast<int32_t*>(c->base + sp.status);
    c->range = reinterpret_cast<uint32_t*>(c->base + sp.range);
    c->done = nullptr;
    c->layout = reinterpret_cast<kvq::SeqLayout*>(c->base + sp.layout);
    c->pages = nullptr;
    c->ring_k = c->base + sp.ring_k;
    c->ring_v = c->base + sp.ring_v;
    c->partials = reinterpret_cast<float*>(c->base + sp.partials);
    c->seg_starts.assign(cfg->batch, {});
  }

  std::vector<kvq::SeqLayout> table(cfg->batch);
  for (int b = 0; b < cfg->batch; ++b) {
    table[b].page_base = a.page_base[b];
    table[b].unit_stride = a.pages_cap[b] * c->geom.page_bytes;
  }
  e = cudaMemcpy(c->layout, table.data(), table.size() * sizeof(kvq::SeqLayout), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemset(c->status, 0, sizeof(int32_t));
  if (e == cudaSuccess && c->range)
    e = cudaMemset(c->range, 0, (size_t)cfg->batch * cfg->n_kv_heads * 2 * sizeof(uint32_t));
  if (e == cudaSuccess && c->done) e = cudaMemset(c->done, 0, (size_t)cfg->batch * cfg->n_kv_heads * sizeof(uint32_t));
  if (e == cudaSuccess) {
    const size_t smem = kvq::flush_launch_smem(cfg->group, cfg->head_dim, esize_of(cfg));
    e = kvq::configure_append(cfg->dtype, c->bits, smem);
  }
  if (cur != attr.device) cudaSetDevice(cur);
  if (e != cudaSuccess) {
    delete c;
    return cuda_fail(e, "kvq_create set-up");
  }
  *out = c;
  return KVQ_OK;
}

// Append to a segmented cache: zero the segment maxima of the sequences, run
// the two flush passes over the overflow of each sequence, then copy the new
// tokens that stay into the rings.
kvq_status append_segmented(kvq_cache* c, const void* new_k, const void* new_v, int64_t n_tokens, int32_t seq_begin,
                            int32_t n_seqs, cudaStream_t s) {
  const int64_t R = c->cfg.residual_len, H = c->cfg.n_kv_heads, D = c->cfg.head_dim;
  const int64_t per_seq_elems = H * n_tokens * D;
  for (int s0 = seq_begin; s0 < seq_begin + n_seqs; s0 += kvq::kMaxSeqsPerLaunch) {
    const int n = std::min(kvq::kMaxSeqsPerLaunch, seq_begin + n_seqs - s0);
    kvq::SegFlushParams p;
    memset(&p, 0, sizeof p);
    p.D = (int)D;
    p.Hkv = (int)H;
    p.R = (int)R;
    p.qmax = c->cfg.qmax;
    p.bits = c->bits;
    p.eps = c->cfg.eps;
    p.seg = c->seg;
    p.kmax = c->kmax;
    p.range = c->range;
    p.ring_k = p.ring_k_out = c->ring_k;
    p.ring_v = p.ring_v_out = c->ring_v;
    const int64_t in_off = (int64_t)(s0 - seq_begin) * per_seq_elems * c->esize;
    p.new_k = static_cast<const uint8_t*>(new_k) + in_off;
    p.new_v = static_cast<const uint8_t*>(new_v) + in_off;
    p.n = n_tokens;
    p.seq_begin = s0;
    p.n_seqs = n;
    fill_counters(c, s0, n, p.old);
    int64_t fmax = 0;
    for (int i = 0; i < n; ++i) fmax = std::max<int64_t>(fmax, p.old[i].total - p.old[i].quantized + n_tokens - R);
    cudaError_t e = cudaSuccess;
    if (fmax > 0) {
      e = cudaMemsetAsync(c->kmax + (int64_t)s0 * H * D, 0, (size_t)n * H * D * sizeof(uint32_t), s);
      if (e == cudaSuccess) e = kvq::launch_seg_flush(p, c->cfg.dtype == KVQ_BF16 ? 0 : 1, fmax, s);
      if (e == cudaSuccess) g_launches += 2;
    }
    if (e == cudaSuccess) e = kvq::launch_seg_window(p, c->cfg.dtype == KVQ_BF16 ? 0 : 1, s);
    if (e != cudaSuccess) return cuda_fail(e, "segmented append launch");
    g_launches += 1;
  }
  for (int b = seq_begin; b < seq_begin + n_seqs; ++b) {
    const int64_t F = std::max<int64_t>(0, c->total[b] - c->quantized[b] + n_tokens - R);
    if (F > 0) c->seg_starts[b].push_back(c->quantized[b]);
    c->quantized[b] += (int32_t)F;
    c->total[b] += (int32_t)n_tokens;
    c->last_flushed[b] = (int32_t)F;
  }
  return KVQ_OK;
}

}  // namespace

extern "C" {

kvq_status kvq_required_bytes(const kvq_config* cfg, const int64_t* capacity_per_seq, size_t* out_bytes) {
  return required_bytes(cfg, capacity_per_seq, 0, out_bytes);
}

kvq_status kvq_create(const kvq_config* cfg, const int64_t* capacity_per_seq, void* device_mem,
                      size_t device_bytes, kvq_cache** out) {
  return create(cfg, capacity_per_seq, 0, device_mem, device_bytes, out);
}

kvq_status kvq_required_bytes_paged(const kvq_config* cfg, const int64_t* capacity_per_seq, int64_t pool_blocks,
                                    size_t* out_bytes) {
  if (pool_blocks < 1 || pool_blocks >= (int64_t(1) << 31))
    return fail(KVQ_EINVAL, "pool_blocks must be in [1, 2^31) (got %lld)", (long long)pool_blocks);
  return required_bytes(cfg, capacity_per_seq, pool_blocks, out_bytes);
}

kvq_status kvq_create_paged(const kvq_config* cfg, const int64_t* capacity_per_seq, int64_t pool_blocks,
                            void* device_mem, size_t device_bytes, kvq_cache** out) {
  if (pool_blocks < 1 || pool_blocks >= (int64_t(1) << 31))
    return fail(KVQ_EINVAL, "pool_blocks must be in [1, 2^31) (got %lld)", (long long)pool_blocks);
  return create(cfg, capacity_per_seq, pool_blocks, device_mem, device_bytes, out);
}

kvq_status kvq_required_bytes_segmented(const kvq_config* cfg, const int64_t* capacity_per_seq, size_t* out_bytes) {
  if (!out_bytes) return fail(KVQ_EINVAL, "out_bytes is NULL");
  kvq_status st = check_config(cfg);
  if (st != KVQ_OK) return st;
  SegPlan sp{};
  st = plan_arena_seg(cfg, capacity_per_seq, &sp);
  if (st != KVQ_OK) return st;
  *out_bytes = sp.total;
  return KVQ_OK;
}

kvq_status kvq_create_segmented(const kvq_config* cfg, const int64_t* capacity_per_seq, void* device_mem,
                                size_t device_bytes, kvq_cache** out) {
  return create(cfg, capacity_per_seq, 0, device_mem, device_bytes, out, true);
}

void kvq_destroy(kvq_cache* cache) { delete cache; }

// The append; window_copy = false leaves the new tokens out of the rings
// (kvq_decode_step's split kernel stores them) and launches the flushes only.
static kvq_status append_impl(kvq_cache* c, const void* new_k, const void* new_v, int64_t n_tokens,
                              int32_t seq_begin, int32_t n_seqs, void* stream, bool window_copy) {
  if (!c) return fail(KVQ_EINVAL, "cache is NULL");
  if (kvq_status st = check_device(c)) return st;
  if (n_tokens <= 0) return fail(KVQ_EINVAL, "n_tokens must be positive (got %lld)", (long long)n_tokens);
  if (n_seqs <= 0 || seq_begin < 0 || seq_begin + (int64_t)n_seqs > c->cfg.batch)
    return fail(KVQ_EINVAL, "sequence range [%d, %d) is outside [0, %d)", seq_begin, seq_begin + n_seqs,
                c->cfg.batch);
  if (!aligned16(new_k) || !aligned16(new_v))
    return fail(KVQ_EINVAL, "new_k / new_v must be non-NULL 16-byte aligned device pointers");
  for (int b = seq_begin; b < seq_begin + n_seqs; ++b) {
    if (c->total[b] + n_tokens > c->cap[b])
      return fail(KVQ_ECAPACITY, "sequence %d: %lld + %lld tokens exceed its capacity %lld", b,
                  (long long)c->total[b], (long long)n_tokens, (long long)c->cap[b]);
  }
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  // a sequence that starts from empty (new, or released) starts its range
  // maxima afresh: one memset per run of such sequences, before any launch
  for (int b = seq_begin; b < seq_begin + n_seqs;) {
    if (c->total[b] != 0) {
      ++b;
      continue;
    }
    int e = b;
    while (e < seq_begin + n_seqs && c->total[e] == 0) ++e;
    const size_t per = (size_t)c->cfg.n_kv_heads * 2;
    const cudaError_t err = cudaMemsetAsync(c->range + b * per, 0, (size_t)(e - b) * per * sizeof(uint32_t), s);
    if (err != cudaSuccess) return cuda_fail(err, "range reset");
    b = e;
  }
  if (c->segmented) return append_segmented(c, new_k, new_v, n_tokens, seq_begin, n_seqs, s);
  const int64_t R = c->cfg.residual_len, G = c->cfg.group;
  const int64_t per_seq_elems = (int64_t)c->cfg.n_kv_heads * n_tokens * c->cfg.head_dim;
  // groups each sequence flushes in this call
  std::vector<int64_t> flushes(n_seqs);
  int64_t new_blocks = 0;
  for (int i = 0; i < n_seqs; ++i) {
    const int b = seq_begin + i;
    flushes[i] = kvq::flush_groups(c->total[b] - c->quantized[b], n_tokens, R, G);
    new_blocks += flushes[i];
  }
  // launches: at most kMaxSeqsPerLaunch sequences and, for a paged cache, at
  // most kMaxNewBlocks new blocks each
  std::vector<std::pair<int, int>> launches;  // (first sequence, count)
  for (int i = 0; i < n_seqs;) {
    int n = 0;
    int64_t blocks = 0;
    while (i + n < n_seqs && n < kvq::kMaxSeqsPerLaunch &&
           (!c->paged || blocks + flushes[i + n] <= kvq::kMaxNewBlocks)) {
      blocks += flushes[i + n];
      ++n;
    }
    if (n == 0)
      return fail(KVQ_EUNSUPPORTED, "sequence %d would flush %lld groups in one append; a paged cache takes at most %d "
                  "per call: split the append", seq_begin + i, (long long)flushes[i], kvq::kMaxNewBlocks);
    launches.emplace_back(seq_begin + i, n);
    i += n;
  }
  if (c->paged && new_blocks > (int64_t)c->free_blocks.size())
    return fail(KVQ_ECAPACITY, "the append needs %lld new blocks; the pool has %zu free", (long long)new_blocks,
                c->free_blocks.size());
  // take the blocks now (no launch has happened, nothing else can fail before them)
  std::vector<int32_t> taken;
  if (c->paged) {
    for (int64_t k = 0; k < new_blocks; ++k) {
      taken.push_back(c->free_blocks.back());
      c->free_blocks.pop_back();
    }
  }
  size_t next_taken = 0;
  for (const auto& ln : launches) {
    const int s0 = ln.first, n = ln.second;
    kvq::AppendParams p;
    memset(&p, 0, sizeof p);
    p.D = c->cfg.head_dim;
    p.Hkv = c->cfg.n_kv_heads;
    p.G = (int)G;
    p.R = (int)R;
    p.Rcap = c->rcap;
    p.qmax = c->cfg.qmax;
    p.bits = c->bits;
    p.eps = c->cfg.eps;
    p.v_prefetch = kvq::flush_v_prefetch((int)G, p.D, (int)c->esize);
    p.range = c->range;
    p.geom = c->geom;
    p.pages = c->pages;
    p.map = page_map(c);
    p.ring_k = c->ring_k;
    p.ring_v = c->ring_v;
    const int64_t in_off = (int64_t)(s0 - seq_begin) * per_seq_elems * c->esize;
    p.new_k = static_cast<const uint8_t*>(new_k) + in_off;
    p.new_v = static_cast<const uint8_t*>(new_v) + in_off;
    p.n = n_tokens;
    p.seq_begin = s0;
    p.n_seqs = n;
    fill_counters(c, s0, n, p.old);
    if (c->paged) {
      int32_t k = 0;
      for (int i = 0; i < n; ++i) {
        p.blk_first[i] = k;
        for (int64_t j = 0; j < flushes[s0 - seq_begin + i]; ++j) {
          const int32_t blk = taken[next_taken++];
          p.blk_ids[k++] = blk;
          c->blocks[s0 + i].push_back(blk);
        }
      }
    }
    int64_t fmax = 0;
    bool overlap = false;
    for (int i = 0; i < n; ++i) {
      const int64_t w = p.old[i].total - p.old[i].quantized;
      const int64_t F = kvq::flush_groups(w, n_tokens, R, G);
      fmax = std::max(fmax, F);
      // ring rows read by the flush and written by the window copy coincide only
      // when the old window plus the new tokens exceed the ring
      if (F > 0 && w + n_tokens > c->rcap) overlap = true;
    }
    cudaError_t e = cudaSuccess;
    if (!window_copy) {
      p.flush_blocks = (int)fmax;
      p.window_blocks = 0;
      if (fmax > 0) {
        e = kvq::launch_append(p, c->cfg.dtype, s);
        g_launches += 1;
      }
    } else if (!overlap) {
      p.flush_blocks = (int)fmax;
      p.window_blocks = 1;
      e = kvq::launch_append(p, c->cfg.dtype, s);
      g_launches += 1;
    } else {
      p.flush_blocks = (int)fmax;
      p.window_blocks = 0;
      e = kvq::launch_append(p, c->cfg.dtype, s);
      g_launches += 1;
      if (e == cudaSuccess) {
        p.flush_blocks = 0;
        p.window_blocks = 1;
        e = kvq::launch_append(p, c->cfg.dtype, s);
        g_launches += 1;
      }
    }
    if (e != cudaSuccess) return cuda_fail(e, "append launch");
  }
  for (int b = seq_begin; b < seq_begin + n_seqs; ++b) {
    const int64_t w = c->total[b] - c->quantized[b];
    const int64_t F = kvq::flush_groups(w, n_tokens, R, G);
    c->quantized[b] += (int32_t)(F * G);
    c->total[b] += (int32_t)n_tokens;
    c->last_flushed[b] = (int32_t)(F * G);
  }
  return KVQ_OK;
}

kvq_status kvq_append(kvq_cache* c, const void* new_k, const void* new_v, int64_t n_tokens, int32_t seq_begin,
                      int32_t n_seqs, void* stream) {
  return append_impl(c, new_k, new_v, n_tokens, seq_begin, n_seqs, stream, true);
}

// The decode; step_k / step_v (kvq_decode_step) hand the split kernel's window
// items this step's tokens, which are then not in the rings yet.
static kvq_status decode_impl(kvq_cache* c, const void* q, float* out, void* stream, const kvq_decode_opts* opts,
                              const void* step_k, const void* step_v) {
  if (!c) return fail(KVQ_EINVAL, "cache is NULL");
  if (kvq_status st = check_device(c)) return st;
  if (!aligned16(q) || !aligned16(out)) return fail(KVQ_EINVAL, "q / out must be 16-byte aligned device pointers");
  const int kernel = opts ? opts->kernel : 0;
  if (kernel < 0 || kernel > 4) return fail(KVQ_EINVAL, "unknown kernel choice %d", kernel);
  // (a segmented cache: 4-bit codes, in 32-token tiles)
  const bool mma_ok = c->cfg.dtype == KVQ_BF16 && (c->cfg.head_dim == 64 || c->cfg.head_dim == 128) &&
                      (c->segmented ? c->bits == 4 : c->cfg.group % 32 == 0) && c->g >= 2;
  if (kernel == 2 && !mma_ok)
    return fail(KVQ_EUNSUPPORTED,
                "tensor-core kernel needs bf16, head_dim 64/128, group %% 32 == 0 (segmented: 4-bit codes) and >= 2 "
                "query heads per KV head");
  const bool tc_ok = mma_ok && c->cfg.head_dim == 128 && c->bits == 4 && !c->segmented;
  if (kernel == 3 && !tc_ok)
    return fail(KVQ_EUNSUPPORTED,
                "tcgen05 kernel needs bf16, head_dim 128, 4-bit codes, group %% 32 == 0 and >= 2 query heads per KV head");
  if (kernel == 4 && !mma_ok)
    return fail(KVQ_EUNSUPPORTED,
                "persistent-warp kernel needs bf16, head_dim 64/128, group %% 32 == 0 and >= 2 query heads per KV head");
  const bool use_tc = kernel == 3;
  const bool use_line = kernel == 4 && !step_k && !c->segmented;
  const bool use_mma = kernel == 2 || kernel == 4 || (kernel == 0 && mma_ok);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (opts && opts->split_start) {
    const cudaError_t e = cudaEventRecord(static_cast<cudaEvent_t>(opts->split_start), s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  }
  // resident CTAs of the tensor-core split kernel, for the planner
  int mma_slots = 0;
  if (use_mma && !use_tc) {
    kvq::DecodeParams qp;
    base_decode_params(c, &qp);
    mma_slots = kvq::decode_mma_resident_per_sm(qp) * c->n_sm;
  }
  struct Batch {
    int s0, n, chunk, grid, line_warps;
    bool merged;  // the split launch merged its partials itself
    std::vector<int64_t> line_start;
  };
  std::vector<Batch> batches;
  for (int s0 = 0; s0 < c->cfg.batch; s0 += kvq::kMaxSeqsPerLaunch) {
    Batch bt;
    bt.s0 = s0;
    bt.n = std::min(kvq::kMaxSeqsPerLaunch, c->cfg.batch - s0);
    plan_splits(c, bt.s0, bt.n, opts ? opts->chunk_pages : 0, mma_slots, &bt.chunk, &bt.grid);
    kvq::DecodeParams p;
    base_decode_params(c, &p);
    p.q = q;
    p.chunk_pages = bt.chunk;
    p.grid_splits = bt.grid;
    p.seq_begin = bt.s0;
    p.n_seqs = bt.n;
    if (step_k) {
      const int64_t off = (int64_t)bt.s0 * c->cfg.n_kv_heads * c->cfg.head_dim * c->esize;
      p.step_k = static_cast<const uint8_t*>(step_k) + off;
      p.step_v = static_cast<const uint8_t*>(step_v) + off;
    }
    fill_counters(c, bt.s0, bt.n, p.ctr);
    cudaError_t e = cudaSuccess;
    int supported = 0;
    bt.line_warps = 0;
    if (use_line) {
      // the line: each sequence's units in order, Q/32 + 2 ceil(W/16)
      // positions a unit; warps = the resident CTAs x 4
      int per_sm = 0;
      e = kvq::decode_line(p, false, s, &per_sm);
      if (e != cudaSuccess) return cuda_fail(e, "persistent-warp kernel set-up");
      const int64_t N = (int64_t)per_sm * c->n_sm * 4;
      bt.line_start.assign(bt.n + 1, 0);
      for (int k = 0; k < bt.n; ++k) {
        const int64_t Q = c->quantized[bt.s0 + k], T = c->total[bt.s0 + k];
        bt.line_start[k + 1] = bt.line_start[k] + (int64_t)c->cfg.n_kv_heads * (Q / 32 + 2 * ((T - Q + 15) / 16));
      }
      const int64_t C = bt.line_start[bt.n];
      // a unit's partials: one per warp that meets it, within the arena's slots
      int64_t most = 0;
      for (int k = 0; k < bt.n && N > 0 && C > 0; ++k) {
        const int64_t cost = (bt.line_start[k + 1] - bt.line_start[k]) / c->cfg.n_kv_heads;
        if (cost == 0) continue;
        for (int h = 0; h < c->cfg.n_kv_heads; ++h) {
          const int64_t s0 = bt.line_start[k] + h * cost;
          most = std::max(most, ((s0 + cost) * N - 1) / C - ((s0 + 1) * N - 1) / C + 1);
        }
      }
      if (per_sm > 0 && C > 0 && C < (int64_t(1) << 31) && most <= c->max_splits) {
        bt.line_warps = (int)N;
        p.line_warps = (int)N;
        for (int k = 0; k <= bt.n; ++k) p.line_start[k] = bt.line_start[k];
        e = kvq::decode_line(p, true, s, &per_sm);
        supported = 1;
      }
    }
    bt.merged = false;
    if (supported) {
    } else if (use_tc) {
      e = kvq::launch_decode_tc(p, s, &supported);
      if (e == cudaSuccess && !supported) return fail(KVQ_EUNSUPPORTED, "tcgen05 kernel does not fit this configuration");
    } else if (use_mma) {
      // A short decode (one wave of resident CTAs, items of at most 16
      // 32-token units, as at batch 1) merges each unit's partials itself
      // (its last finishing CTA), so no combine launch follows it: 10.7 us
      // against 11.5 us a decode of a batch-1 4096-token layer.  Longer
      // launches keep the combine kernel: there the arrival count holds every
      // CTA's slot a little longer and the merges of many slots end the
      // launch (measured slower on the 32 x 8 x 8192 layer and on the
      // 432000-token layer).
      const int64_t ctas = (int64_t)(bt.grid + 1) * bt.n * c->cfg.n_kv_heads;
      const int64_t item_units = (int64_t)bt.chunk * (c->cfg.group / 32);
      if (kvq::decode_mma_supported(p) && mma_slots > 0 && ctas <= mma_slots && item_units <= 16) {
        p.done = c->done;
        p.out = out;
        bt.merged = c->done != nullptr;
      }
      e = kvq::launch_decode_mma(p, s, &supported);
      if (e == cudaSuccess && !supported && kernel == 2)
        return fail(KVQ_EUNSUPPORTED, "tensor-core kernel does not fit this configuration (shared memory)");
    }
    if (e == cudaSuccess && !supported) e = kvq::launch_decode_simt(p, c->cfg.dtype, s);
    if (e != cudaSuccess) return cuda_fail(e, "decode split launch");
    g_launches += 1;
    batches.push_back(bt);
  }
  if (opts && opts->split_stop) {
    const cudaError_t e = cudaEventRecord(static_cast<cudaEvent_t>(opts->split_stop), s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  }
  for (const Batch& bt : batches) {
    if (bt.merged) continue;
    kvq::CombineParams cp;
    memset(&cp, 0, sizeof cp);
    cp.D = c->cfg.head_dim;
    cp.Hkv = c->cfg.n_kv_heads;
    cp.Hq = c->cfg.n_q_heads;
    cp.g = c->g;
    cp.G = c->cfg.group;
    cp.max_splits = c->max_splits;
    cp.chunk_pages = bt.chunk;
    cp.partials = c->partials;
    cp.out = out;
    cp.seq_begin = bt.s0;
    cp.n_seqs = bt.n;
    cp.line_warps = bt.line_warps;
    for (int k = 0; k < (int)bt.line_start.size(); ++k) cp.line_start[k] = bt.line_start[k];
    fill_counters(c, bt.s0, bt.n, cp.ctr);
    const cudaError_t e = kvq::launch_combine(cp, s);
    if (e != cudaSuccess) return cuda_fail(e, "combine launch");
    g_launches += 1;
  }
  return KVQ_OK;
}

kvq_status kvq_decode_attention_ex(kvq_cache* c, const void* q, float* out, void* stream,
                                   const kvq_decode_opts* opts) {
  return decode_impl(c, q, out, stream, opts, nullptr, nullptr);
}

kvq_status kvq_decode_attention(kvq_cache* c, const void* q, float* out, void* stream) {
  return kvq_decode_attention_ex(c, q, out, stream, nullptr);
}

kvq_status kvq_decode_step(kvq_cache* c, const void* new_k, const void* new_v, const void* q, float* out,
                           void* stream, const kvq_decode_opts* opts) {
  if (!c) return fail(KVQ_EINVAL, "cache is NULL");
  if (!aligned16(new_k) || !aligned16(new_v) || !aligned16(q) || !aligned16(out))
    return fail(KVQ_EINVAL, "new_k / new_v / q / out must be non-NULL 16-byte aligned device pointers");
  const int kernel = opts ? opts->kernel : 0;
  // the tensor-core kernel takes the step's tokens from the input; any other
  // path runs the plain append and decode
  bool fuse = kernel != 1 && !c->segmented && c->cfg.dtype == KVQ_BF16 &&
              (c->cfg.head_dim == 64 || c->cfg.head_dim == 128) && c->cfg.group % 32 == 0 && c->g >= 2;
  if (fuse) {
    kvq::DecodeParams p;
    base_decode_params(c, &p);
    fuse = kvq::decode_mma_supported(p);
  }
  if (!fuse) {
    const kvq_status st = kvq_append(c, new_k, new_v, 1, 0, c->cfg.batch, stream);
    return st != KVQ_OK ? st : decode_impl(c, q, out, stream, opts, nullptr, nullptr);
  }
  const kvq_status st = append_impl(c, new_k, new_v, 1, 0, c->cfg.batch, stream, false);
  return st != KVQ_OK ? st : decode_impl(c, q, out, stream, opts, new_k, new_v);
}

}  // extern "C"

// ---- decode attention with library-owned scratch -------------------------------
//
// Some callers cannot allocate device memory when they run the decode: a plugin
// inside a host framework that owns every device allocation, or a deployment
// that reserves all its memory once at start-up, has no cudaMalloc to call and
// no spare buffer to hand over.  kvq_decode_attention_noalloc serves them: the
// split partials, the only scratch the decode needs, go to the fixed array
// below instead of the arena's scratch region.  The array is 8 MiB of device
// memory that every GPU which loads this library holds until the process exits.

constexpr size_t kNoAllocScratchFloats = size_t(2) << 20;  // 8 MiB of float
static __device__ __align__(256) float kvq_noalloc_scratch[kNoAllocScratchFloats];

namespace {

constexpr int kNoAllocMaxDevices = 64;
float* g_noalloc_ptr[kNoAllocMaxDevices];
std::mutex g_noalloc_mu;

// Device address of kvq_noalloc_scratch on ``device``, looked up once per
// device with that device current (host code only sees a stand-in symbol).
kvq_status noalloc_scratch(int device, float** out) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (device < 0 || device >= kNoAllocMaxDevices)
    return fail(KVQ_EUNSUPPORTED, "device %d is beyond the %d devices the scratch table covers", device,
                kNoAllocMaxDevices);
  if (!g_noalloc_ptr[device]) {
    int cur = 0;
    cudaError_t e = cudaGetDevice(&cur);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (cur != device && (e = cudaSetDevice(device)) != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, kvq_noalloc_scratch);
    if (cur != device) cudaSetDevice(cur);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(kvq_noalloc_scratch)");
    g_noalloc_ptr[device] = static_cast<float*>(p);
  }
  *out = g_noalloc_ptr[device];
  return KVQ_OK;
}

}  // namespace

extern "C" {

kvq_status kvq_decode_attention_noalloc(kvq_cache* c, const void* q, float* out, void* stream) {
  if (!c) return fail(KVQ_EINVAL, "cache is NULL");
  if (kvq_status st = check_device(c)) return st;
  if (!aligned16(q) || !aligned16(out)) return fail(KVQ_EINVAL, "q / out must be 16-byte aligned device pointers");
  const int B = c->cfg.batch, H = c->cfg.n_kv_heads, D = c->cfg.head_dim;
  // one split plan for every sequence, then as many split slots as the array holds
  int64_t pmax = 0;
  for (int b = 0; b < B; ++b) pmax = std::max<int64_t>(pmax, c->quantized[b] / c->cfg.group);
  const size_t per_slot = (size_t)B * H * c->g * kvq::part_row(D);  // floats of one split column
  const size_t min_slots = pmax > 0 ? 2 : 1;              // one quantized split plus the window
  if (per_slot * min_slots > kNoAllocScratchFloats)
    return fail(KVQ_ECAPACITY,
                "decode needs %zu floats of split scratch, more than the %zu floats (8 MiB) the library reserves",
                per_slot * min_slots, kNoAllocScratchFloats);
  int chunk = 1, grid = 0;
  plan_splits(c, 0, B, 0, 0, &chunk, &grid);
  const int64_t fit = (int64_t)(kNoAllocScratchFloats / per_slot);  // >= min_slots
  if (grid + 1 > fit) {
    chunk = (int)((pmax + (fit - 1) - 1) / (fit - 1));
    grid = (int)((pmax + chunk - 1) / chunk);
  }
  const int slots = grid + 1;
  float* scratch = nullptr;
  kvq_status st = noalloc_scratch(c->device, &scratch);
  if (st != KVQ_OK) return st;
  const bool use_mma = c->cfg.dtype == KVQ_BF16 && (D == 64 || D == 128) && c->cfg.group % 32 == 0 && c->g >= 2;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int s0 = 0; s0 < B; s0 += kvq::kMaxSeqsPerLaunch) {
    const int n = std::min(kvq::kMaxSeqsPerLaunch, B - s0);
    kvq::DecodeParams p;
    base_decode_params(c, &p);
    p.q = q;
    p.partials = scratch;
    p.max_splits = slots;
    p.chunk_pages = chunk;
    p.grid_splits = grid;
    p.seq_begin = s0;
    p.n_seqs = n;
    fill_counters(c, s0, n, p.ctr);
    cudaError_t e = cudaSuccess;
    int supported = 0;
    if (use_mma) e = kvq::launch_decode_mma(p, s, &supported);
    if (e == cudaSuccess && !supported) e = kvq::launch_decode_simt(p, c->cfg.dtype, s);
    if (e != cudaSuccess) return cuda_fail(e, "decode split launch");
    g_launches += 1;
  }
  for (int s0 = 0; s0 < B; s0 += kvq::kMaxSeqsPerLaunch) {
    kvq::CombineParams cp;
    memset(&cp, 0, sizeof cp);
    cp.D = D;
    cp.Hkv = H;
    cp.Hq = c->cfg.n_q_heads;
    cp.g = c->g;
    cp.G = c->cfg.group;
    cp.max_splits = slots;
    cp.chunk_pages = chunk;
    cp.partials = scratch;
    cp.out = out;
    cp.seq_begin = s0;
    cp.n_seqs = std::min(kvq::kMaxSeqsPerLaunch, B - s0);
    fill_counters(c, s0, cp.n_seqs, cp.ctr);
    const cudaError_t e = kvq::launch_combine(cp, s);
    if (e != cudaSuccess) return cuda_fail(e, "combine launch");
    g_launches += 1;
  }
  return KVQ_OK;
}

kvq_status kvq_ledger(const kvq_config* cfg, const int64_t* tokens_per_seq, kvq_bytes_t* out) {
  if (!out || !tokens_per_seq) return fail(KVQ_EINVAL, "NULL argument");
  const kvq_status st = check_config(cfg);
  if (st != KVQ_OK) return st;
  const int64_t R = cfg->residual_len, G = cfg->group, H = cfg->n_kv_heads, D = cfg->head_dim;
  const int bits = bits_of(cfg);
  kvq_bytes_t r;
  memset(&r, 0, sizeof r);
  for (int b = 0; b < cfg->batch; ++b) {
    const int64_t T = tokens_per_seq[b];
    if (T < 0) return fail(KVQ_EINVAL, "negative token count for sequence %d", b);
    const int64_t Q = T >= R + G ? (T - R) / G * G : 0;
    r.code_bytes += 2 * H * Q * D * bits / 8;
    r.n_scales += H * ((Q / G) * D + Q);
    r.window_elems += 2 * H * (T - Q) * D;
  }
  r.scale_bytes = 4 * r.n_scales;
  r.window_bytes = r.window_elems * esize_of(cfg);
  r.total = r.code_bytes + r.scale_bytes + r.window_bytes;
  *out = r;
  return KVQ_OK;
}

kvq_status kvq_bytes(const kvq_cache* c, kvq_bytes_t* out) {
  if (!c || !out) return fail(KVQ_EINVAL, "NULL argument");
  if (c->segmented) {
    // one Key scale per channel per segment, one Value scale per token
    const int64_t H = c->cfg.n_kv_heads, D = c->cfg.head_dim;
    int64_t code = 0, n_scales = 0, window = 0;
    for (int b = 0; b < c->cfg.batch; ++b) {
      code += 2 * H * (int64_t)c->quantized[b] * D * c->bits / 8;
      n_scales += H * ((int64_t)c->seg_starts[b].size() * D + c->quantized[b]);
      window += 2 * H * (int64_t)(c->total[b] - c->quantized[b]) * D;
    }
    out->code_bytes = code;
    out->n_scales = n_scales;
    out->scale_bytes = 4 * n_scales;
    out->window_elems = window;
    out->window_bytes = window * c->esize;
    out->total = code + 4 * n_scales + window * c->esize;
    out->allocated = (int64_t)c->arena_bytes;
    return KVQ_OK;
  }
  std::vector<int64_t> t(c->total.begin(), c->total.end());
  const kvq_status st = kvq_ledger(&c->cfg, t.data(), out);
  if (st == KVQ_OK) out->allocated = (int64_t)c->arena_bytes;
  return st;
}

kvq_status kvq_seq_state(const kvq_cache* c, int32_t seq, kvq_seq_info* out) {
  if (!c || !out) return fail(KVQ_EINVAL, "NULL argument");
  if (seq < 0 || seq >= c->cfg.batch) return fail(KVQ_EINVAL, "sequence %d out of range", seq);
  out->total = c->total[seq];
  out->quantized = c->quantized[seq];
  out->window = c->total[seq] - c->quantized[seq];
  out->last_flushed = c->last_flushed[seq];
  out->n_groups = c->segmented ? (int64_t)c->seg_starts[seq].size() : c->quantized[seq] / c->cfg.group;
  out->capacity = c->cap[seq];
  return KVQ_OK;
}

kvq_status kvq_export_pages(const kvq_cache* c, int32_t seq, int32_t kv_head, void* host_dst, size_t dst_bytes,
                            void* stream) {
  if (!c) return fail(KVQ_EINVAL, "NULL argument");
  if (seq < 0 || seq >= c->cfg.batch || kv_head < 0 || kv_head >= c->cfg.n_kv_heads)
    return fail(KVQ_EINVAL, "unit (%d, %d) out of range", seq, kv_head);
  if (c->segmented) return fail(KVQ_EUNSUPPORTED, "a segmented cache has no group pages (use kvq_export_unit)");
  const size_t bytes = (size_t)(c->quantized[seq] / c->cfg.group) * c->geom.page_bytes;
  if (bytes == 0) return KVQ_OK;
  if (!host_dst) return fail(KVQ_EINVAL, "host_dst is NULL");
  if (dst_bytes < bytes) return fail(KVQ_EINVAL, "host buffer of %zu bytes < %zu", dst_bytes, bytes);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (c->paged) {
    // one copy per block: the pages of a sequence lie wherever its blocks do
    const int64_t pb = c->geom.page_bytes;
    for (size_t j = 0; j < c->blocks[seq].size() && e == cudaSuccess; ++j) {
      const uint8_t* src = c->pages + (int64_t)c->blocks[seq][j] * c->cfg.n_kv_heads * pb + (int64_t)kv_head * pb;
      e = cudaMemcpyAsync(static_cast<uint8_t*>(host_dst) + j * pb, src, pb, cudaMemcpyDeviceToHost, s);
    }
  } else {
    const uint8_t* src = c->pages + c->page_base[seq] + (int64_t)kv_head * c->pages_cap[seq] * c->geom.page_bytes;
    e = cudaMemcpyAsync(host_dst, src, bytes, cudaMemcpyDeviceToHost, s);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e, "kvq_export_pages");
}

kvq_status kvq_release(kvq_cache* c, int32_t seq_begin, int32_t n_seqs) {
  if (!c) return fail(KVQ_EINVAL, "cache is NULL");
  if (n_seqs <= 0 || seq_begin < 0 || seq_begin + (int64_t)n_seqs > c->cfg.batch)
    return fail(KVQ_EINVAL, "sequence range [%d, %d) is outside [0, %d)", seq_begin, seq_begin + n_seqs,
                c->cfg.batch);
  for (int b = seq_begin; b < seq_begin + n_seqs; ++b) {
    // most recently taken first, so that a release followed by the same appends
    // hands the blocks out in the same order again
    for (auto it = c->blocks[b].rbegin(); it != c->blocks[b].rend(); ++it) c->free_blocks.push_back(*it);
    c->blocks[b].clear();
    if (c->segmented) c->seg_starts[b].clear();
    c->total[b] = c->quantized[b] = c->last_flushed[b] = 0;
  }
  return KVQ_OK;
}

kvq_status kvq_pool_state(const kvq_cache* c, int64_t* free_blocks, int64_t* pool_blocks) {
  if (!c || !free_blocks || !pool_blocks) return fail(KVQ_EINVAL, "NULL argument");
  *free_blocks = (int64_t)c->free_blocks.size();
  *pool_blocks = c->pool_blocks;
  return KVQ_OK;
}

kvq_status kvq_export_unit(const kvq_cache* c, int32_t seq, int32_t kv_head, const kvq_unit_view* view,
                           void* stream) {
  if (!c || !view) return fail(KVQ_EINVAL, "NULL argument");
  if (seq < 0 || seq >= c->cfg.batch || kv_head < 0 || kv_head >= c->cfg.n_kv_heads)
    return fail(KVQ_EINVAL, "unit (%d, %d) out of range", seq, kv_head);
  const int D = c->cfg.head_dim, G = c->cfg.group, bits = c->bits;
  const int64_t Q = c->quantized[seq], T = c->total[seq], P = c->segmented ? 0 : Q / G;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::vector<uint8_t> pages((size_t)P * c->geom.page_bytes);
  kvq_status st = c->segmented ? KVQ_OK : kvq_export_pages(c, seq, kv_head, pages.data(), pages.size(), stream);
  if (st != KVQ_OK) return st;
  if (c->segmented && Q > 0) {
    // token-major rows: codes, Value scales, and each segment's Key scale row in
    // the row of its first token
    const int64_t row0 = ((int64_t)seq * c->cfg.n_kv_heads + kv_head) * c->seg.cap;
    const int rb = c->seg.row_bytes;
    std::vector<uint8_t> kc((size_t)Q * rb), vc((size_t)Q * rb);
    std::vector<float> ks((size_t)Q * D), vs((size_t)Q);
    cudaError_t e = cudaMemcpyAsync(kc.data(), c->seg.kcodes + row0 * rb, kc.size(), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(vc.data(), c->seg.vcodes + row0 * rb, vc.size(), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(ks.data(), c->seg.kscales + row0 * D, ks.size() * 4, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(vs.data(), c->seg.vscales + row0, vs.size() * 4, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "kvq_export_unit");
    auto code_at = [&](const uint8_t* row, int ch) -> int8_t {
      if (bits == 2) return (int8_t)((int)((row[ch / 4] >> (2 * (ch % 4))) & 0x3) - 2);
      if (bits == 4) return (int8_t)((int)((row[ch / 2] >> (4 * (ch % 2))) & 0xF) - 8);
      return (int8_t)((int)row[ch] - 128);
    };
    for (int64_t t = 0; t < Q; ++t)
      for (int ch = 0; ch < D; ++ch) {
        if (view->k_codes) view->k_codes[t * D + ch] = code_at(kc.data() + t * rb, ch);
        if (view->v_codes) view->v_codes[t * D + ch] = code_at(vc.data() + t * rb, ch);
      }
    if (view->v_scales) memcpy(view->v_scales, vs.data(), vs.size() * 4);
    if (view->k_scales)
      for (size_t j = 0; j < c->seg_starts[seq].size(); ++j)
        memcpy(view->k_scales + j * D, ks.data() + (size_t)c->seg_starts[seq][j] * D, (size_t)D * 4);
  }
  // ring rows of the window, read whole and reordered on the host
  const size_t ring_bytes = (size_t)c->rcap * D * c->esize;
  std::vector<uint8_t> rk(ring_bytes), rv(ring_bytes);
  const int64_t unit = (int64_t)seq * c->cfg.n_kv_heads + kv_head;
  cudaError_t e = cudaMemcpyAsync(rk.data(), static_cast<const uint8_t*>(c->ring_k) + unit * ring_bytes, ring_bytes,
                                  cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(rv.data(), static_cast<const uint8_t*>(c->ring_v) + unit * ring_bytes, ring_bytes,
                        cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "kvq_export_unit");

  auto sext = [bits](uint32_t v) -> int8_t {  // offset binary -> signed code
    return bits == 2   ? (int8_t)((int)(v & 0x3) - 2)
           : bits == 4 ? (int8_t)((int)(v & 0xF) - 8)
                       : (int8_t)((int)(v & 0xFF) - 128);
  };
  for (int64_t pg = 0; pg < P; ++pg) {
    const uint8_t* page = pages.data() + pg * c->geom.page_bytes;
    const float* ks = reinterpret_cast<const float*>(page + c->geom.kscale_off);
    const float* vs = reinterpret_cast<const float*>(page + c->geom.vscale_off);
    for (int t = 0; t < G; ++t) {
      const int64_t tok = pg * G + t;
      for (int ch = 0; ch < D; ++ch) {
        if (view->k_codes) {
          const uint32_t byte = page[(size_t)t * (D * bits / 8) + ch * bits / 8];
          view->k_codes[tok * D + ch] = sext(bits == 8 ? byte : byte >> (bits * (ch % (8 / bits))));
        }
        if (view->v_codes) {
          const uint8_t* vb = page + c->geom.code_bytes;
          const int st_i = t / 32, o = t % 32, n_st = std::min(32, G - 32 * st_i);
          const uint8_t* sub = vb + (size_t)st_i * 32 * D * bits / 8;
          uint32_t code;
          if (bits == 2) {
            uint16_t piece;
            memcpy(&piece, sub + ((size_t)ch * (n_st / 8) + o / 8) * 2, 2);
            const int k = o % 8;
            code = (uint32_t)piece >> (8 * (k % 2) + 2 * (k / 2));
          } else if (bits == 4) {
            uint32_t word;
            memcpy(&word, sub + ((size_t)ch * (n_st / 8) + o / 8) * 4, 4);
            const int k = o % 8, jn = k / 2 + 4 * (k % 2);
            code = word >> (4 * jn);
          } else {
            code = sub[(size_t)ch * n_st + o];
          }
          view->v_codes[tok * D + ch] = sext(code);
        }
      }
      if (view->v_scales) view->v_scales[tok] = vs[t];
    }
    if (view->k_scales) memcpy(view->k_scales + pg * D, ks, (size_t)D * sizeof(float));
  }
  for (int64_t t = Q; t < T; ++t) {
    const size_t row = (size_t)(t % c->rcap) * D;
    for (int ch = 0; ch < D; ++ch) {
      float kf, vf;
      if (c->esize == 2) {
        uint16_t kb, vb;
        memcpy(&kb, rk.data() + (row + ch) * 2, 2);
        memcpy(&vb, rv.data() + (row + ch) * 2, 2);
        const uint32_t k32 = (uint32_t)kb << 16, v32 = (uint32_t)vb << 16;
        memcpy(&kf, &k32, 4);
        memcpy(&vf, &v32, 4);
      } else {
        memcpy(&kf, rk.data() + (row + ch) * 4, 4);
        memcpy(&vf, rv.data() + (row + ch) * 4, 4);
      }
      if (view->window_k) view->window_k[(t - Q) * D + ch] = kf;
      if (view->window_v) view->window_v[(t - Q) * D + ch] = vf;
    }
  }
  return KVQ_OK;
}

kvq_status kvq_device_status(const kvq_cache* c, int32_t* out_word, void* stream) {
  if (!c || !out_word) return fail(KVQ_EINVAL, "NULL argument");
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t w = 0;
  cudaError_t e = cudaMemcpyAsync(&w, c->status, sizeof w, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "kvq_device_status");
  *out_word = w;
  if (w != 0) return fail(KVQ_EDEVICE, "device status word is 0x%x", (unsigned)w);
  return KVQ_OK;
}

kvq_status kvq_restore(const kvq_cache* c, int32_t seq_begin, int32_t n_seqs, void* k_out, void* v_out,
                       int64_t t_stride, kvq_dtype out_dtype, void* stream) {
  if (!c) return fail(KVQ_EINVAL, "cache is NULL");
  if (kvq_status st = check_device(c)) return st;
  if (n_seqs <= 0 || seq_begin < 0 || seq_begin + (int64_t)n_seqs > c->cfg.batch)
    return fail(KVQ_EINVAL, "sequence range [%d, %d) is outside [0, %d)", seq_begin, seq_begin + n_seqs,
                c->cfg.batch);
  if (out_dtype != KVQ_BF16 && out_dtype != KVQ_FP32) return fail(KVQ_EINVAL, "unknown out_dtype %d", out_dtype);
  if (!aligned16(k_out) || !aligned16(v_out))
    return fail(KVQ_EINVAL, "k_out / v_out must be non-NULL 16-byte aligned device pointers");
  int64_t tmax = 0, pmax = 0;
  for (int b = seq_begin; b < seq_begin + n_seqs; ++b) {
    tmax = std::max<int64_t>(tmax, c->total[b]);
    pmax = std::max<int64_t>(pmax, c->quantized[b] / c->cfg.group);
  }
  if (t_stride < tmax || t_stride < 1)
    return fail(KVQ_EINVAL, "t_stride %lld is below the largest held length %lld", (long long)t_stride,
                (long long)tmax);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t unit_elems = t_stride * c->cfg.head_dim;
  const int osz = out_dtype == KVQ_BF16 ? 2 : 4;
  if (c->segmented) {
    for (int s0 = seq_begin; s0 < seq_begin + n_seqs; s0 += kvq::kMaxSeqsPerLaunch) {
      const int n = std::min(kvq::kMaxSeqsPerLaunch, seq_begin + n_seqs - s0);
      kvq::RestoreParams p;
      memset(&p, 0, sizeof p);
      p.D = c->cfg.head_dim;
      p.Hkv = c->cfg.n_kv_heads;
      p.G = 1;
      p.Rcap = c->rcap;
      p.bits = c->bits;
      p.eps = c->cfg.eps;
      p.seg = c->seg;
      p.ring_k = c->ring_k;
      p.ring_v = c->ring_v;
      p.in_dtype = c->cfg.dtype == KVQ_BF16 ? 0 : 1;
      p.out_dtype = out_dtype == KVQ_BF16 ? 0 : 1;
      const int64_t off = (int64_t)(s0 - seq_begin) * c->cfg.n_kv_heads * unit_elems * osz;
      p.k_out = static_cast<uint8_t*>(k_out) + off;
      p.v_out = static_cast<uint8_t*>(v_out) + off;
      p.t_stride = t_stride;
      p.seq_begin = s0;
      p.n_seqs = n;
      fill_counters(c, s0, n, p.ctr);
      const cudaError_t e = kvq::launch_seg_restore(p, tmax, s);
      if (e != cudaSuccess) return cuda_fail(e, "restore launch");
      g_launches += 1;
    }
    return KVQ_OK;
  }
  for (int s0 = seq_begin; s0 < seq_begin + n_seqs; s0 += kvq::kMaxSeqsPerLaunch) {
    const int n = std::min(kvq::kMaxSeqsPerLaunch, seq_begin + n_seqs - s0);
    kvq::RestoreParams p;
    memset(&p, 0, sizeof p);
    p.D = c->cfg.head_dim;
    p.Hkv = c->cfg.n_kv_heads;
    p.G = c->cfg.group;
    p.Rcap = c->rcap;
    p.bits = c->bits;
    p.eps = c->cfg.eps;
    p.geom = c->geom;
    p.pages = c->pages;
    p.map = page_map(c);
    p.ring_k = c->ring_k;
    p.ring_v = c->ring_v;
    p.in_dtype = c->cfg.dtype == KVQ_BF16 ? 0 : 1;
    p.out_dtype = out_dtype == KVQ_BF16 ? 0 : 1;
    const int64_t off = (int64_t)(s0 - seq_begin) * c->cfg.n_kv_heads * unit_elems * osz;
    p.k_out = static_cast<uint8_t*>(k_out) + off;
    p.v_out = static_cast<uint8_t*>(v_out) + off;
    p.t_stride = t_stride;
    p.page_cols = (int)pmax;
    p.seq_begin = s0;
    p.n_seqs = n;
    fill_counters(c, s0, n, p.ctr);
    const cudaError_t e = kvq::launch_restore(p, s);
    if (e != cudaSuccess) return cuda_fail(e, "restore launch");
    g_launches += 1;
  }
  return KVQ_OK;
}

kvq_status kvq_dense_decode_attention(kvq_cache* c, const void* k, const void* v, int64_t t_stride, const void* q,
                                      float* out, void* stream) {
  if (!c) return fail(KVQ_EINVAL, "cache is NULL");
  if (kvq_status st = check_device(c)) return st;
  if (!aligned16(k) || !aligned16(v) || !aligned16(q) || !aligned16(out))
    return fail(KVQ_EINVAL, "k / v / q / out must be non-NULL 16-byte aligned device pointers");
  if (c->cfg.dtype != KVQ_BF16 || (c->cfg.head_dim != 64 && c->cfg.head_dim != 128))
    return fail(KVQ_EUNSUPPORTED, "dense decode needs a bf16 cache with head_dim 64 or 128");
  int64_t tmax = 0, total = 0;
  for (int b = 0; b < c->cfg.batch; ++b) {
    tmax = std::max<int64_t>(tmax, c->total[b]);
    total += (int64_t)c->total[b] * c->cfg.n_kv_heads;
  }
  if (t_stride < tmax || t_stride < 1)
    return fail(KVQ_EINVAL, "t_stride %lld is below the largest held length %lld", (long long)t_stride,
                (long long)tmax);
  // chunks of whole 64-token rounds (16 tokens per warp step, 4 warps), about
  // 8 CTAs per SM over the batch, and never more chunks than split slots
  int64_t chunk = std::max<int64_t>(256, (total + (int64_t)c->n_sm * 8 - 1) / ((int64_t)c->n_sm * 8));
  chunk = std::max<int64_t>(chunk, (tmax + c->max_splits - 1) / c->max_splits);
  chunk = (chunk + 63) / 64 * 64;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int s0 = 0; s0 < c->cfg.batch; s0 += kvq::kMaxSeqsPerLaunch) {
    const int n = std::min(kvq::kMaxSeqsPerLaunch, c->cfg.batch - s0);
    kvq::DecodeParams p;
    base_decode_params(c, &p);
    p.q = q;
    p.dense_k = k;
    p.dense_v = v;
    p.t_stride = t_stride;
    p.dense_chunk = (int)chunk;
    p.seq_begin = s0;
    p.n_seqs = n;
    fill_counters(c, s0, n, p.ctr);
    int supported = 0;
    const cudaError_t e = kvq::launch_decode_dense(p, s, &supported);
    if (e != cudaSuccess) return cuda_fail(e, "dense decode launch");
    if (!supported) return fail(KVQ_EUNSUPPORTED, "dense decode does not support this configuration");
    g_launches += 1;
  }
  for (int s0 = 0; s0 < c->cfg.batch; s0 += kvq::kMaxSeqsPerLaunch) {
    kvq::CombineParams cp;
    memset(&cp, 0, sizeof cp);
    cp.D = c->cfg.head_dim;
    cp.Hkv = c->cfg.n_kv_heads;
    cp.Hq = c->cfg.n_q_heads;
    cp.g = c->g;
    cp.G = c->cfg.group;
    cp.max_splits = c->max_splits;
    cp.dense_chunk = (int)chunk;
    cp.partials = c->partials;
    cp.out = out;
    cp.seq_begin = s0;
    cp.n_seqs = std::min(kvq::kMaxSeqsPerLaunch, c->cfg.batch - s0);
    fill_counters(c, s0, cp.n_seqs, cp.ctr);
    const cudaError_t e = kvq::launch_combine(cp, s);
    if (e != cudaSuccess) return cuda_fail(e, "combine launch");
    g_launches += 1;
  }
  return KVQ_OK;
}

kvq_status kvq_compare(const void* key, const void* value, int64_t batch, int32_t heads, int64_t tokens,
                       int32_t head_dim, kvq_dtype dtype, int32_t qmax, float eps, int32_t group, void* workspace,
                       kvq_compare_t* out, void* stream) {
  if (!out) return fail(KVQ_EINVAL, "out is NULL");
  if (batch < 1 || heads < 1 || tokens < 1 || head_dim < 1)
    return fail(KVQ_EINVAL, "shape must be positive (batch %lld, heads %d, tokens %lld, head_dim %d)",
                (long long)batch, heads, (long long)tokens, head_dim);
  if (dtype != KVQ_BF16 && dtype != KVQ_FP32) return fail(KVQ_EINVAL, "unknown dtype %d", dtype);
  if (qmax < 1 || qmax > 127) return fail(KVQ_EINVAL, "qmax must be in [1, 127] (got %d)", qmax);
  if (!(eps > 0.f) || !std::isfinite(eps)) return fail(KVQ_EINVAL, "eps must be positive and finite");
  if (group < 0 || (group > 0 && tokens % group != 0))
    return fail(KVQ_EINVAL, "group %d must be 0 or divide tokens %lld", group, (long long)tokens);
  if (batch * heads > 65535) return fail(KVQ_EUNSUPPORTED, "batch * heads must be <= 65535");
  if (!key || !value || !workspace || ((uintptr_t)workspace & 7u) != 0)
    return fail(KVQ_EINVAL, "key / value / workspace must be non-NULL device pointers (workspace 8-byte aligned)");
  const int64_t group_len = group > 0 ? group : tokens;
  if (tokens / group_len > 0x7fffffff) return fail(KVQ_EUNSUPPORTED, "too many Key-scale groups");
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  kvq::CompareParams p;
  memset(&p, 0, sizeof p);
  p.key = key;
  p.value = value;
  p.tokens = tokens;
  p.D = head_dim;
  p.dtype = dtype == KVQ_BF16 ? 0 : 1;
  p.qmax = qmax;
  p.group_len = (int32_t)group_len;
  p.eps = eps;
  p.sums = static_cast<double*>(workspace);
  double sums[2] = {0.0, 0.0};
  cudaError_t e = cudaMemsetAsync(workspace, 0, 2 * sizeof(double), s);
  if (e == cudaSuccess) e = kvq::launch_compare(p, batch * heads, s);
  if (e == cudaSuccess) g_launches += 1;
  if (e == cudaSuccess) e = cudaMemcpyAsync(sums, workspace, sizeof sums, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "kvq_compare");
  const int64_t n = batch * heads * tokens * head_dim;
  const int64_t n_kscales = batch * heads * (tokens / group_len) * head_dim;
  const int64_t n_vscales = batch * heads * tokens;
  const int64_t scale_bytes = 4 * (n_kscales + n_vscales);
  out->key_mse = sums[0] / (double)n;
  out->value_mse = sums[1] / (double)n;
  out->n_key_scales = n_kscales;
  out->n_value_scales = n_vscales;
  out->raw_bytes = 2 * n * (dtype == KVQ_BF16 ? 2 : 4);
  out->container_quantized_bytes = 2 * n + scale_bytes;
  out->packed_quantized_bytes = (2 * n + 1) / 2 + scale_bytes;
  return KVQ_OK;
}

}  // extern "C"
