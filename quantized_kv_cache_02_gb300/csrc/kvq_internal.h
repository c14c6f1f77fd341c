// Internal definitions shared by the host side of libkvq and its kernels:
// launch parameter blocks, the group-page layout and small device helpers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace kvq {

// Sequences per kernel launch: their counters travel in the parameter block.
constexpr int kMaxSeqsPerLaunch = 256;
// Largest GQA group (query heads per KV head) the kernels handle.
constexpr int kMaxGqa = 8;
// New blocks one append launch of a paged cache may fill (their ids travel in
// the parameter block).
constexpr int kMaxNewBlocks = 4096;

// Floats of one split partial row (o[D], m, l): padded to a multiple of 16
// bytes so that the combine reads it with 16-byte loads.
__host__ __device__ constexpr int part_row(int D) { return D + 4; }

// Device status word codes (kvq_device_status).
constexpr int32_t kStatusWaitTimeout = 0x101;  // a bounded mbarrier wait gave up

// Counters of one sequence as they stand before a launch.
struct SeqCounters {
  int32_t total;      // tokens held
  int32_t quantized;  // tokens in the quantized prefix (multiple of G)
};

// Static placement of one sequence's pages (device table written at create).
struct SeqLayout {
  int64_t page_base;    // byte offset of (seq, kv head 0, page 0) from the page region
  int64_t unit_stride;  // bytes between consecutive kv heads of the sequence
};

// Where the group pages live.  Contiguous cache: the pages of unit (b, h) lie
// back to back from layout[b].page_base + h * layout[b].unit_stride.  Paged
// cache ("KV Cache 与自回归视频生成" section 05, a block table per request):
// a block holds one group of a sequence for every KV head (head h at
// h * page_bytes, codes and scales together), and table[b * table_stride + j]
// is the block of the sequence's group j.
struct PageMap {
  const SeqLayout* layout;
  int32_t* table;              // null: contiguous
  int32_t table_stride;        // table entries per sequence
  int64_t block_bytes;         // n_kv_heads * page_bytes
};

__host__ __device__ inline int64_t page_offset(const PageMap& m, int64_t page_bytes, int b, int h, int64_t pg) {
  if (m.table) return (int64_t)m.table[(int64_t)b * m.table_stride + pg] * m.block_bytes + (int64_t)h * page_bytes;
  return m.layout[b].page_base + h * m.layout[b].unit_stride + pg * page_bytes;
}

// Geometry of a group page (see the layout comment in kvq.h).
struct PageGeom {
  int32_t G, D, bits;
  int64_t code_bytes;   // bytes of one code block (Key or Value): G * D * bits / 8
  int64_t kscale_off;   // offset of the Key scales
  int64_t vscale_off;   // offset of the Value scales
  int64_t page_bytes;
};

__host__ __device__ inline PageGeom make_geom(int G, int D, int bits) {
  PageGeom g;
  g.G = G;
  g.D = D;
  g.bits = bits;
  g.code_bytes = (int64_t)G * D * bits / 8;
  g.kscale_off = 2 * g.code_bytes;
  g.vscale_off = g.kscale_off + 4 * (int64_t)D;
  g.page_bytes = g.vscale_off + 4 * (int64_t)G;
  return g;
}

// Number of groups flushed when an append of n tokens meets a window of w
// tokens (residual window R, group G).
__host__ __device__ inline int64_t flush_groups(int64_t w, int64_t n, int64_t R, int64_t G) {
  const int64_t tail = w + n;
  return tail < R + G ? 0 : (tail - R) / G;
}

// Segmented cache ("54. KV Cache Quantization Strategies", append_and_partition
// verbatim): every append flushes its whole overflow as one segment with one
// Key scale per channel over the segment's tokens.  Codes are token-major rows
// (the Key row packing of a group page, for Keys and Values alike); each
// token keeps its segment's Key scale row and its own Value scale.
struct SegArrays {
  uint8_t* kcodes;             // [batch][Hkv][cap][row_bytes]; null: not segmented
  uint8_t* vcodes;
  float* kscales;              // [batch][Hkv][cap][D]; a segment's row at its first token
  float* vscales;              // [batch][Hkv][cap]
  int32_t* first;              // [batch][cap]: first token of each token's segment
  int64_t cap;                 // token rows per unit (a multiple of 32)
  int32_t row_bytes;           // D * bits / 8
};

struct SegFlushParams {
  int32_t D, Hkv, R, qmax, bits;
  float eps;
  SegArrays seg;
  uint32_t* kmax;              // [batch][Hkv][D] bits of the segment's Key absmax (zeroed first)
  uint32_t* range;             // [batch][Hkv][2]: largest flushed Key / Value absmax (as AppendParams::range)
  const void* ring_k;          // [batch][Hkv][R][D] (the window before the append)
  const void* ring_v;
  void* ring_k_out;            // the same rings (written by the window pass only)
  void* ring_v_out;
  const void* new_k;           // [n_seqs][Hkv][n][D]
  const void* new_v;
  int64_t n;
  int32_t seq_begin, n_seqs;
  SeqCounters old[kMaxSeqsPerLaunch];
};

// Shared memory of a flush CTA: the G x D tile in the input dtype (esize
// bytes an element), the Key and Value scales, and the partial Key maxima of
// the threads' 16-byte columns (rows per pass x D floats; 16 / esize channels
// a column, kAppendThreads threads).
constexpr int kAppendThreads = 256;
__host__ __device__ inline size_t flush_smem_bytes(int G, int D, int esize) {
  const size_t partials = (size_t)kAppendThreads * (16 / esize) > (size_t)D ? (size_t)kAppendThreads * (16 / esize)
                                                                            : (size_t)D;
  return (size_t)G * D * esize + ((size_t)D + G + partials + G) * sizeof(float);
}
// Whether a flush CTA also holds a second tile, into which the Values are
// copied (cp.async) while the Keys are reduced and packed; and the shared
// memory of a flush launch with that choice.
constexpr size_t kFlushSmemMax = 200 * 1024;
inline bool flush_v_prefetch(int G, int D, int esize) {
  return flush_smem_bytes(G, D, esize) + (size_t)G * D * esize <= kFlushSmemMax;
}
inline size_t flush_launch_smem(int G, int D, int esize) {
  return flush_smem_bytes(G, D, esize) + (flush_v_prefetch(G, D, esize) ? (size_t)G * D * esize : 0);
}

struct AppendParams {
  int32_t D, Hkv, G, R, Rcap, qmax, bits;
  float eps;
  PageGeom geom;
  uint8_t* pages;              // page region (contiguous) or block pool (paged)
  PageMap map;
  void* ring_k;                // [batch][Hkv][Rcap][D] (dtype)
  void* ring_v;
  const void* new_k;           // [n_seqs][Hkv][n][D]
  const void* new_v;
  int64_t n;                   // new tokens per sequence
  int32_t seq_begin, n_seqs;
  int32_t flush_blocks;        // grid.x slots for flush groups (0 if none in this launch)
  int32_t window_blocks;       // grid.x slots for window writes (0 or 1)
  int32_t v_prefetch;          // flush_v_prefetch(G, D, esize)
  // [batch][Hkv][2]: bits of the largest Key and Value absmax each unit has
  // flushed (atomicMax; non-negative floats order as their bits)
  uint32_t* range;
  SeqCounters old[kMaxSeqsPerLaunch];
  // paged caches: the blocks of sequence i's new groups are
  // blk_ids[blk_first[i] ..]; the flush writes them into the block table
  int32_t blk_first[kMaxSeqsPerLaunch];
  int32_t blk_ids[kMaxNewBlocks];
};

struct DecodeParams {
  int32_t D, Hkv, Hq, g, G, Rcap, bits, qmax;
  float eps;
  float qk_scale;              // log2(e) / sqrt(D): scores are kept in base 2
  PageGeom geom;
  const uint8_t* pages;
  PageMap map;
  const void* ring_k;
  const void* ring_v;
  const void* q;               // [batch][Hq][D]
  const uint32_t* range;       // the flushed absmax maxima per unit (AppendParams::range)
  float* partials;             // [batch*Hkv][max_splits][g][part_row(D)]
  // non-null (tensor-core split kernel only): the combine runs inside the
  // split launch.  done[unit] counts the unit's finished items (0 between
  // launches); the CTA that finishes last merges the unit's partials into
  // out [batch][Hq][D] and sets the count back to 0
  uint32_t* done;
  float* out;
  int32_t max_splits;          // slots per unit; the window uses slot max_splits - 1
  int32_t chunk_pages;         // pages per quantized split
  int32_t grid_splits;         // quantized split columns in this launch (window column after)
  int32_t seq_begin, n_seqs;
  int32_t* status;
  SegArrays seg;                // segmented caches (pages are then single tokens, G = 1)
  // kvq_decode_step: this step's token per (sequence, KV head), [n_seqs][Hkv][D];
  // the window item reads it from here and writes it into its ring row
  const void* step_k;
  const void* step_v;
  // dense restored cache (decode_dense_kernel only): [batch][Hkv][t_stride][D]
  const void* dense_k;
  const void* dense_v;
  int64_t t_stride;
  int32_t dense_chunk;         // tokens per dense split
  // persistent-warp kernel: its warps (grid x 4) and the line position of
  // each sequence's first unit (line_start[n_seqs] = the line's length); a
  // sequence's units each take Q/32 + 2 ceil((T - Q) / 16) positions
  int32_t line_warps;
  int64_t line_start[kMaxSeqsPerLaunch + 1];
  SeqCounters ctr[kMaxSeqsPerLaunch];
};

struct CombineParams {
  int32_t D, Hkv, Hq, g, G, max_splits, chunk_pages;
  int32_t dense_chunk;         // > 0: slots are dense token chunks, no window slot
  // > 0: the partials of the persistent-warp kernel, which takes line_warps
  // warps over the line (as DecodeParams): a unit's slots are 0 .. n - 1 for
  // the n warps from the one holding its first position to its last
  int32_t line_warps;
  int64_t line_start[kMaxSeqsPerLaunch + 1];
  const float* partials;
  float* out;                  // [batch][Hq][D]
  int32_t seq_begin, n_seqs;
  SeqCounters ctr[kMaxSeqsPerLaunch];
};

// Programmatic dependent launch.  Every kernel of the library is launched
// with the programmatic stream serialization attribute and begins with
// pdl_wait(), which returns once the previous kernel in the stream has
// finished and its writes are visible: stream order is kept, but the launch
// and CTA start-up overlap the predecessor's last wave.  pdl_release() lets
// the next kernel be scheduled once every CTA of this grid has started.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_release() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... Args>
cudaError_t launch_pdl(void (*kernel)(Args...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Dequantize a cache into dense tensors (kvq_restore).  Grid: one CTA per
// (page column, unit) plus a window column.
struct RestoreParams {
  int32_t D, Hkv, G, Rcap, bits;
  float eps;
  PageGeom geom;
  const uint8_t* pages;
  PageMap map;
  const void* ring_k;          // cache dtype
  const void* ring_v;
  int32_t in_dtype, out_dtype; // 0 bf16, 1 fp32
  void* k_out;                 // [n_seqs][Hkv][t_stride][D] (out dtype)
  void* v_out;
  int64_t t_stride;
  SegArrays seg;               // segmented caches
  int32_t page_cols;           // pages of the longest unit (the launcher turns it into
                               // columns of page runs; the window column follows)
  int32_t seq_begin, n_seqs;
  SeqCounters ctr[kMaxSeqsPerLaunch];
};

// The datawhale page's compare: quantize a Key/Value pair, restore, sum the
// squared errors (kvq_compare).
struct CompareParams {
  const void* key;             // [rows][tokens][D] (dtype)
  const void* value;
  int64_t tokens;
  int32_t D, dtype, qmax;
  int32_t group_len;           // tokens per Key scale (a divisor of tokens)
  float eps;
  double* sums;                // [2]: Key, Value squared-error sums (accumulated)
};

// Launchers (defined in the kernel translation units). Return the launch's error code.
cudaError_t launch_append(const AppendParams& p, int dtype, cudaStream_t s);
cudaError_t configure_append(int dtype, int bits, size_t smem_bytes);
cudaError_t launch_decode_simt(const DecodeParams& p, int dtype, cudaStream_t s);
cudaError_t launch_decode_mma(const DecodeParams& p, cudaStream_t s, int* supported);
// the persistent-warp split kernel: launch = false returns its resident CTAs
// per SM in *per_sm (0: not supported); launch = true launches it with
// p.line_warps warps
cudaError_t decode_line(const DecodeParams& p, bool launch, cudaStream_t s, int* per_sm);
cudaError_t line_bits2(const DecodeParams& p, bool launch, cudaStream_t s, int* per_sm);
cudaError_t line_bits4(const DecodeParams& p, bool launch, cudaStream_t s, int* per_sm);
cudaError_t line_bits8(const DecodeParams& p, bool launch, cudaStream_t s, int* per_sm);
// the split kernel for one code width (one translation unit each)
// CTAs of the tensor-core split kernel one SM holds at once for p (0: not
// supported or unknown).
int decode_mma_resident_per_sm(const DecodeParams& p);
int resident_mma_bits2(const DecodeParams& p);
int resident_mma_bits4(const DecodeParams& p);
int resident_mma_bits8(const DecodeParams& p);
cudaError_t launch_mma_bits2(const DecodeParams& p, cudaStream_t s);
cudaError_t launch_mma_bits4(const DecodeParams& p, cudaStream_t s);
cudaError_t launch_mma_bits8(const DecodeParams& p, cudaStream_t s);
size_t decode_mma_smem_bytes(const DecodeParams& p);
bool decode_mma_supported(const DecodeParams& p);
// the fifth-generation tensor-core split kernel (head_dim 128, 4-bit codes)
cudaError_t launch_decode_tc(const DecodeParams& p, cudaStream_t s, int* supported);
bool decode_tc_supported(const DecodeParams& p);
cudaError_t launch_combine(const CombineParams& p, cudaStream_t s);
cudaError_t launch_decode_dense(const DecodeParams& p, cudaStream_t s, int* supported);
cudaError_t launch_restore(const RestoreParams& p, cudaStream_t s);
// segmented caches: pass 1 (Key absmax, Value codes), pass 2 (Key codes), window copy
cudaError_t launch_seg_flush(const SegFlushParams& p, int dtype, int64_t max_tokens, cudaStream_t s);
cudaError_t launch_seg_window(const SegFlushParams& p, int dtype, cudaStream_t s);
cudaError_t launch_seg_restore(const RestoreParams& p, int64_t max_tokens, cudaStream_t s);
cudaError_t launch_compare(const CompareParams& p, int64_t rows, cudaStream_t s);

}  // namespace kvq
