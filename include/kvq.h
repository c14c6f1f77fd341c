/*
 * kvq.h -- C ABI of libkvq.so: a KIVI-style asymmetric quantized KV cache with a
 * single-query GQA decode attention over it, for NVIDIA GB300 (sm_103a).
 *
 * What the library computes (sources named by page title and section):
 *
 *  - Quantizer: "54. KV Cache Quantization Strategies" (datawhale llm-algo-leetcode),
 *    Step 2 and the Step 4 reference solution.  Key: per channel, absmax over the
 *    tokens of a flushed group; Value: per token, absmax over head_dim;
 *    scale = qmax / max(absmax, eps) (correctly rounded fp32 division);
 *    code = clamp(round_half_even(x * scale), -qmax, qmax) with x * scale one fp32
 *    multiply; restore = code / scale.
 *  - Residual window: same page, Step 3 and ``append_and_partition``.  The newest
 *    tokens stay in a high-precision window (the input dtype); only tokens that
 *    overflow it are quantized; the quantized prefix is never rewritten.  This
 *    library flushes whole groups: after an append leaves L tokens in the window,
 *    F = floor((L - R) / G) groups of the oldest G tokens are quantized when
 *    L >= R + G (F = 0 otherwise), each group with its own Key scales.  With G = 1
 *    this is the page's rule flush = max(L - R, 0).  The held partition depends
 *    only on a sequence's length T: quantized = G * floor((T - R) / G) when
 *    T >= R + G, else 0; window = T - quantized, so R <= window < R + G once
 *    anything is quantized.
 *  - Decode attention: "KV Cache 与自回归视频生成" (jefxiong), section 3.1
 *    (o_t = sum_j softmax_j(q_t . k_j / sqrt(d)) v_j over every held token, the
 *    token appended in the same step included) and section 04 ``attn_step``
 *    (query head h reads KV head h / g, g = n_q_heads / n_kv_heads).  The
 *    quantized prefix is dequantized in registers; the split over the sequence
 *    and the merge of partial softmax states follow section 05 (FlashDecoding).
 *  - Byte ledger: "KV Cache 量化与压缩" (xuujii M005) sections 01 and 05.
 *
 * Conventions for every entry point:
 *  - Status codes: KVQ_OK on success; any other value leaves the cache state
 *    unchanged and sets a thread-local message readable with kvq_last_error().
 *  - Memory: the caller owns all device memory (the cache arena, inputs and
 *    outputs); the library allocates no device memory and keeps no pointer to
 *    inputs or outputs after a call returns (the work is stream ordered).
 *  - Streams: ``stream`` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  kvq_append and kvq_decode_attention* only enqueue work and never
 *    synchronize; the caller orders calls on one cache (one stream, or events).
 *  - Device pointers must be 16-byte aligned and the tensors contiguous.
 *  - Device: kernels launch on the current CUDA device; every entry point
 *    that launches work returns KVQ_EINVAL, before any launch, when that is
 *    not the device that holds the cache's arena.
 *  - One cache holds one layer.  A multi-layer model creates one cache per layer.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kvq_status {
  KVQ_OK = 0,
  KVQ_EINVAL = 1,       /* bad argument: config, pointer, range, alignment */
  KVQ_ECAPACITY = 2,    /* an append would exceed a sequence's capacity */
  KVQ_ENOMEM = 3,       /* the caller's arena is smaller than kvq_required_bytes */
  KVQ_ECUDA = 4,        /* a CUDA call or kernel launch failed */
  KVQ_EUNSUPPORTED = 5, /* valid but not implemented (e.g. head_dim, group size) */
  KVQ_EDEVICE = 6       /* a kernel reported an error through the device status word */
} kvq_status;

typedef enum kvq_dtype {
  KVQ_BF16 = 0, /* K/V/q inputs and the residual window are bfloat16 */
  KVQ_FP32 = 1  /* ... float32 */
} kvq_dtype;

/* Cache configuration (one layer). */
typedef struct kvq_config {
  int32_t batch;        /* B: number of sequences, >= 1 */
  int32_t n_kv_heads;   /* Hkv >= 1 */
  int32_t n_q_heads;    /* Hq, a multiple of Hkv with g = Hq / Hkv <= 8 */
  int32_t head_dim;     /* d: a multiple of 16, 16 <= d <= 256 */
  int32_t residual_len; /* R > 0: tokens kept at input precision */
  int32_t group;        /* G > 0, a multiple of 8: tokens quantized together */
  int32_t qmax;         /* 1: signed 2-bit codes (-1, 0, 1), four per byte;
                           2..7: signed 4-bit codes, two per byte;
                           8..127: signed 8-bit codes */
  int32_t dtype;        /* kvq_dtype of inputs and window */
  float eps;            /* absmax floor for the scale, e.g. 1e-8f (> 0) */
} kvq_config;

/* Held-bytes ledger (whole cache, all sequences and KV heads). */
typedef struct kvq_bytes_t {
  int64_t code_bytes;   /* Key + Value codes: 4-bit packed or 8-bit */
  int64_t n_scales;     /* Key: head_dim per flushed group; Value: one per token */
  int64_t scale_bytes;  /* 4 * n_scales (scales are fp32) */
  int64_t window_elems; /* Key + Value elements in the residual windows */
  int64_t window_bytes; /* window_elems * sizeof(dtype) */
  int64_t total;        /* code_bytes + scale_bytes + window_bytes */
  int64_t allocated;    /* bytes of the arena the cache was created on (0 for kvq_ledger) */
} kvq_bytes_t;

/* Per-sequence bookkeeping, the counters of ``append_and_partition``. */
typedef struct kvq_seq_info {
  int64_t total;        /* tokens appended so far (T) */
  int64_t quantized;    /* tokens in the quantized prefix (multiple of G) */
  int64_t window;       /* tokens in the residual window (T - quantized) */
  int64_t last_flushed; /* tokens quantized by the most recent append to this sequence */
  int64_t n_groups;     /* quantized / G */
  int64_t capacity;     /* capacity given at creation */
} kvq_seq_info;

/* Host view of one (sequence, KV head) unit, filled by kvq_export_unit.  Every
 * pointer is a HOST buffer owned by the caller, sized from kvq_seq_info:
 *   k_codes, v_codes: int8 [quantized][head_dim], logical (unpacked) codes
 *   k_scales: float [quantized / G][head_dim];  v_scales: float [quantized]
 *   window_k, window_v: float [window][head_dim], token order (oldest first)
 * Any pointer may be NULL to skip that part. */
typedef struct kvq_unit_view {
  int8_t* k_codes;
  int8_t* v_codes;
  float* k_scales;
  float* v_scales;
  float* window_k;
  float* window_v;
} kvq_unit_view;

/* Options of kvq_decode_attention_ex (zero-initialise for defaults). */
typedef struct kvq_decode_opts {
  int32_t kernel;      /* 0 = automatic; 1 = CUDA-core kernel (any supported
                          shape); 2 = tensor-core kernel on mma.sync (bf16,
                          head_dim 64/128, G a multiple of 32, or a
                          segmented cache with 4-bit codes); 3 = tcgen05
                          tensor-core kernel (bf16, head_dim 128, 4-bit codes,
                          G a multiple of 32; it handles the input range per
                          block of 128 tokens: groups with a Key scale below
                          the bound of kvq_decode_attention enter with signed
                          codes and q / sK scaled by a power of two, blocks
                          with a Value absmax above 16 are summed in fp32);
                          4 = persistent-warp mma.sync kernel (same
                          operands and range handling as 2): every warp
                          of one resident wave takes an equal share of a
                          line of work items (32-token quantized pages
                          weigh 1, 16-token window steps 2), so split
                          boundaries need not fall on whole groups of
                          pages; chunk_pages is ignored.  On a segmented
                          cache, in kvq_decode_step, and where a unit
                          would need more partials than the cache's split
                          slots, it runs as 2.  KVQ_EUNSUPPORTED if not
                          applicable */
  int32_t chunk_pages; /* 0 = automatic: about 6 split items per SM (8 on a
                          segmented cache), rounded to whole 8-page groups at
                          G = 32; with few (sequence, KV head) units on the
                          tensor-core kernel, as many columns as fill whole
                          waves of its resident CTAs.  Else quantized groups
                          per split item.  Results agree for any choice within
                          the attention tolerance (the summation order of the
                          splits differs).  A segmented cache counts tokens
                          and rounds the chunk up to a multiple of 128. */
  void* split_start;   /* optional cudaEvent_t recorded just before the split kernel */
  void* split_stop;    /* optional cudaEvent_t recorded just after it */
} kvq_decode_opts;

/* Result of kvq_compare (the datawhale page's compare ledger). */
typedef struct kvq_compare_t {
  double key_mse, value_mse;        /* mean of (x - restore(quantize(x)))^2 */
  int64_t n_key_scales;             /* batch * heads * (tokens / group_len) * head_dim */
  int64_t n_value_scales;           /* batch * heads * tokens */
  int64_t raw_bytes;                /* Key + Value elements * dtype bytes */
  int64_t container_quantized_bytes;/* one byte per code + 4 bytes per scale */
  int64_t packed_quantized_bytes;   /* (codes + 1) / 2 + 4 bytes per scale (two codes a byte) */
} kvq_compare_t;

typedef struct kvq_cache kvq_cache; /* opaque host handle */

/*
 * Device-memory layout (documented so that pages can be inspected).
 *
 * Group page: one per (sequence, KV head, flushed group), written once by the
 * flush and never again.  With bits = 2 (qmax <= 1, KIVI's 2-bit codes), 4
 * (qmax <= 7) or 8, in order:
 *   Codes are stored offset binary: code + 2 in two bits (1..3 for qmax 1),
 *   code + 8 in a nibble (1..15 for qmax 7), code + 128 in a byte.
 *   1. Key codes: G rows (token order) of head_dim*bits/8 bytes.  2-bit: byte
 *      i holds channel 4i+k in bits 2k..2k+1; 4-bit: byte i holds channel 2i in
 *      bits 0-3 and channel 2i+1 in bits 4-7; 8-bit: byte c is channel c.
 *   2. Value codes in sub-tiles of 32 tokens (the last sub-tile holds G mod 32
 *      tokens if G is not a multiple of 32).  A sub-tile of n tokens is head_dim
 *      rows (channel order) of n*bits/8 bytes.  4-bit rows are little-endian
 *      32-bit words; word w covers tokens 8w..8w+7 of the sub-tile and its
 *      nibble j holds token 8w+2j for j < 4 and token 8w+2(j-4)+1 for j >= 4.
 *      2-bit rows are little-endian 16-bit pieces; piece p covers tokens
 *      8p..8p+7, its bits 2f..2f+1 hold token 8p+2f and bits 8+2f..9+2f token
 *      8p+2f+1 (f = 0..3).  8-bit rows hold token i in byte i.
 *   3. Key scales: head_dim fp32.   4. Value scales: G fp32.
 *   Page size = 2*G*head_dim*bits/8 + 4*head_dim + 4*G bytes.
 * Pages of one unit are contiguous and in token order.
 * Residual window: per unit a ring of Rcap = G * (ceil(R / G) + 1) rows of
 * head_dim elements (dtype) for Key and another for Value; token t of the
 * sequence lives in row t mod Rcap.
 */

/* Bytes of device memory a cache with this configuration and these per-sequence
 * capacities needs (capacity_per_seq: host array of ``batch`` token counts,
 * each >= 1 and < 2^31).  Pure host function. */
kvq_status kvq_required_bytes(const kvq_config* cfg, const int64_t* capacity_per_seq,
                              size_t* out_bytes);

/* Create a cache on caller-owned device memory of the current CUDA device
 * (``device_mem``: 256-byte aligned, ``device_bytes`` >= kvq_required_bytes).
 * All sequences start empty.  Writes a small layout table and clears the
 * device status word with synchronous copies (set-up only).  *out receives the
 * handle; destroy it with kvq_destroy.  The memory must outlive the handle. */
kvq_status kvq_create(const kvq_config* cfg, const int64_t* capacity_per_seq, void* device_mem,
                      size_t device_bytes, kvq_cache** out);

/* Paged cache ("KV Cache 与自回归视频生成" section 05: fixed-size blocks and a
 * block table per request; "KV Cache 量化与压缩" section 07: low-bit data and
 * their scales addressed together).  A block is one flushed group of one
 * sequence for every KV head: n_kv_heads group pages (the layout above) back
 * to back, so codes and scales travel together.  The arena holds a pool of
 * ``pool_blocks`` blocks shared by all sequences, a block table row per
 * sequence (capacity_per_seq[b] / group entries) and the per-sequence residual
 * windows.  Blocks are taken from the pool when groups flush and returned by
 * kvq_release; capacity_per_seq[b] only bounds the length of sequence b, the
 * pool bounds the sum.  Every other call works on a paged cache as on a
 * contiguous one, with the same results.  kvq_append fails with KVQ_ECAPACITY
 * (before any launch, state unchanged) when the pool lacks the blocks its
 * flushes need, and with KVQ_EUNSUPPORTED when one call would flush more than
 * 4096 groups of one sequence (split such a prefill into several calls).
 * pool_blocks must be in [1, 2^31); other arguments as kvq_required_bytes /
 * kvq_create. */
kvq_status kvq_required_bytes_paged(const kvq_config* cfg, const int64_t* capacity_per_seq, int64_t pool_blocks,
                                    size_t* out_bytes);
kvq_status kvq_create_paged(const kvq_config* cfg, const int64_t* capacity_per_seq, int64_t pool_blocks,
                            void* device_mem, size_t device_bytes, kvq_cache** out);

/* Segmented cache: the flush rule of "54. KV Cache Quantization Strategies"
 * (append_and_partition) verbatim.  An append of n tokens to a window of L
 * flushes its whole overflow, max(L + n - R, 0) tokens, as ONE segment: Key
 * codes with one scale per channel over the segment's tokens, Value codes
 * with one scale per token; the newest min(L + n, R) tokens stay at input
 * precision.  cfg->group is not used (any valid value).  Storage: per unit,
 * token-major code rows (each row packed like a group page's Key row, for
 * Keys and Values alike), each segment's Key scales (head_dim fp32) in the
 * row of its first token, each token's Value scale, per sequence the first
 * token of each token's segment (int32), and a window ring of R rows.  Decode
 * attention (bf16, head_dim 64/128, 4-bit codes, >= 2 query heads per KV
 * head; else the CUDA-core kernel) runs on the tensor-core kernel in 32-token
 * tiles: a tile inside one segment shares one Key scale row, as a group page
 * does; a tile that holds a segment boundary (as every tile of one-token
 * segments does) or the unit's last, partial tile is scored on the CUDA cores
 * inside the same launch.  kvq_export_unit returns one Key
 * scale row per segment; kvq_export_pages returns KVQ_EUNSUPPORTED; the other
 * calls work as on a grouped cache.  Arguments as kvq_required_bytes /
 * kvq_create. */
kvq_status kvq_required_bytes_segmented(const kvq_config* cfg, const int64_t* capacity_per_seq, size_t* out_bytes);
kvq_status kvq_create_segmented(const kvq_config* cfg, const int64_t* capacity_per_seq, void* device_mem,
                                size_t device_bytes, kvq_cache** out);

/* Empty sequences [seq_begin, seq_begin + n_seqs) (counters to zero); a paged
 * cache returns their blocks to the pool.  Host bookkeeping only: work already
 * queued on a stream still sees the old contents, and a later append may
 * reuse the blocks, so issue everything on one stream (or order the streams)
 * around a release.  KVQ_EINVAL for a bad range. */
kvq_status kvq_release(kvq_cache* cache, int32_t seq_begin, int32_t n_seqs);

/* Free and total blocks of a paged cache's pool (both 0 for a contiguous
 * cache).  Host counters, no device access. */
kvq_status kvq_pool_state(const kvq_cache* cache, int64_t* free_blocks, int64_t* pool_blocks);

/* Append ``n_tokens`` new tokens to each of the sequences
 * [seq_begin, seq_begin + n_seqs) ("append_and_partition": cat with the window,
 * then flush whole groups).  new_k, new_v: device [n_seqs][n_kv_heads]
 * [n_tokens][head_dim] of the cache dtype (post-RoPE Keys).  Errors:
 * KVQ_EINVAL (n_tokens <= 0, bad range, NULL or misaligned pointer),
 * KVQ_ECAPACITY (total would exceed a capacity) -- both before any launch.
 * For ragged prefills call once per sequence with n_seqs = 1. */
kvq_status kvq_append(kvq_cache* cache, const void* new_k, const void* new_v, int64_t n_tokens,
                      int32_t seq_begin, int32_t n_seqs, void* stream);

/* Decode attention for every sequence: q device [batch][n_q_heads][head_dim] of
 * the cache dtype; out device float [batch][n_q_heads][head_dim].  A sequence
 * with no tokens yields zeros.  Uses the arena's split scratch region.
 * Launches: a split kernel (one per 256 sequences) and a combine kernel after
 * it, except for a short decode on the tensor-core kernel (one wave of the
 * resident CTAs, split items of at most 16 32-token units, e.g. a single
 * sequence), whose last CTA per (sequence, KV head) merges the partials
 * itself (an arrival count in the arena, back to 0 when the launch ends).
 *
 * Input range.  Any finite Key, Value and query values are accepted; scales
 * below eps (absmax > qmax / eps) restore as code / eps, as the page's restore
 * does.  The tensor-core kernels carry q / sK and p / sV as f16 operands, so
 * the cache tracks, per (sequence, KV head), the largest Key and Value absmax
 * it has flushed (reset when a sequence starts from empty).  A split item
 * runs on the tensor cores only while those bound every group of its unit:
 * |q| * qk_scale * (Key absmax) / qmax <= 2^9 (2^14 at 2-bit codes, x 1/16
 * below the f16 limit) -- i.e. every Key scale >= 2^(e + 1 - 9) with e the
 * binary exponent of the largest |q| / sqrt(head_dim) * log2(e) -- and every
 * Value absmax <= 16.  Other items run the CUDA-core path inside the same
 * launch (fp32, IEEE division with the eps clamp), so results stay within the
 * attention tolerance for any range, at CUDA-core speed for those units.
 * The residual window is attended from its bf16 rows on either path. */
kvq_status kvq_decode_attention(kvq_cache* cache, const void* q, float* out, void* stream);

/* Same as kvq_decode_attention with explicit options (kernel choice, split
 * size, timing events); opts may be NULL. */
kvq_status kvq_decode_attention_ex(kvq_cache* cache, const void* q, float* out, void* stream,
                                   const kvq_decode_opts* opts);

/* One decode step: append one new token to every sequence, then the decode
 * attention -- kvq_append(n_tokens = 1, all sequences) followed by
 * kvq_decode_attention_ex, with the same results.  new_k, new_v: device
 * [batch][n_kv_heads][1][head_dim] of the cache dtype; q, out as in
 * kvq_decode_attention; opts may be NULL.  On the tensor-core path the
 * append's window copy is folded into the split kernel: each window item
 * attends the step's token straight from new_k / new_v and stores it in its
 * ring row, so a step without a flush is two launches instead of three.
 * Errors as kvq_append and kvq_decode_attention, before any launch. */
kvq_status kvq_decode_step(kvq_cache* cache, const void* new_k, const void* new_v, const void* q, float* out,
                           void* stream, const kvq_decode_opts* opts);

/* No counterpart in the source pages: an addition for callers that cannot
 * allocate device memory when they decode (a plugin whose host framework owns
 * every device allocation, a deployment that reserves all memory once at
 * start-up).  Computes the same attention as kvq_decode_attention, within the
 * decode tolerance (its split boundaries may differ, so the fp32 rounding of
 * the partials may), but keeps the split partials -- the decode's only
 * scratch -- in a fixed array inside the library instead of the arena's
 * scratch region, and allocates nothing: no cudaMalloc, cudaFree or
 * allocating library call.
 *  - The array holds 2^21 floats (8 MiB); every GPU that loads the library
 *    holds it until the process exits.  A cache whose batch * n_kv_heads *
 *    (n_q_heads / n_kv_heads) * (head_dim + 4) floats times 2 split columns
 *    (1 without any flushed group) exceed it is rejected with KVQ_ECAPACITY
 *    before any launch; otherwise the split count is lowered to fit.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.
 *  - All calls on a device share the array and it keeps the last call's
 *    contents; nothing in it needs to start at zero, since every partial a
 *    call reads is written earlier in the same call.  Calls that overlap on the
 *    GPU (other streams, other caches) race on it: serialize them.
 * Arguments, layout, ownership and errors are those of kvq_decode_attention
 * (KVQ_EINVAL as well when the current device is not the cache's). */
kvq_status kvq_decode_attention_noalloc(kvq_cache* cache, const void* q, float* out, void* stream);

/* Held-bytes ledger of a live cache (host counters, no device access). */
kvq_status kvq_bytes(const kvq_cache* cache, kvq_bytes_t* out);

/* Ledger of a cache of this configuration holding tokens_per_seq[b] tokens per
 * sequence (host array of ``batch`` counts); pure host function. */
kvq_status kvq_ledger(const kvq_config* cfg, const int64_t* tokens_per_seq, kvq_bytes_t* out);

/* Bookkeeping of sequence ``seq`` (host counters, no device access). */
kvq_status kvq_seq_state(const kvq_cache* cache, int32_t seq, kvq_seq_info* out);

/* Copy one unit's codes, scales and window to host buffers, decoded from the
 * layout above (synchronizes ``stream``): k_codes, v_codes [quantized][head_dim]
 * int8; k_scales [n_groups][head_dim] (one row per flushed group, or per
 * segment of a segmented cache); v_scales [quantized]; window_k, window_v
 * [window][head_dim] fp32.  Any pointer may be NULL to skip that part. */
kvq_status kvq_export_unit(const kvq_cache* cache, int32_t seq, int32_t kv_head,
                           const kvq_unit_view* view, void* stream);

/* Copy the raw bytes of one unit's group pages (n_groups * page size bytes,
 * token order) to the host buffer ``host_dst`` of ``dst_bytes`` bytes
 * (synchronizes ``stream``).  With no flushed group it copies nothing and
 * ``host_dst`` may be NULL. */
kvq_status kvq_export_pages(const kvq_cache* cache, int32_t seq, int32_t kv_head, void* host_dst,
                            size_t dst_bytes, void* stream);

/* Read the device status word (synchronizes ``stream``).  0 means no kernel has
 * reported an error; non-zero codes come from bounded waits that gave up.
 * Returns KVQ_EDEVICE when the word is non-zero. */
kvq_status kvq_device_status(const kvq_cache* cache, int32_t* out_word, void* stream);

/* Dequantize-to-HBM, step 1 ("KV Cache 量化与压缩" section 06, read path (a);
 * "54. KV Cache Quantization Strategies", restore).  Writes the held Keys and
 * Values of sequences [seq_begin, seq_begin + n_seqs) as dense device tensors
 * k_out, v_out [n_seqs][n_kv_heads][t_stride][head_dim] of out_dtype.
 * Row t < quantized is code / max(scale, eps) computed in fp32 (Key codes over
 * their group's per-channel scales, Value codes over their per-token scales),
 * rounded to nearest even for KVQ_BF16; rows quantized <= t < total are the
 * residual window as held, converted to out_dtype.  Rows >= total are left
 * untouched.  t_stride >= the largest total in the range.  The buffers are the
 * caller's (16-byte aligned).  Errors before any launch: KVQ_EINVAL (bad range,
 * NULL or misaligned pointer, t_stride too small, unknown dtype). */
kvq_status kvq_restore(const kvq_cache* cache, int32_t seq_begin, int32_t n_seqs, void* k_out, void* v_out,
                       int64_t t_stride, kvq_dtype out_dtype, void* stream);

/* Dequantize-to-HBM, step 2: the standard decode attention over dense bf16
 * Key/Value tensors k, v [batch][n_kv_heads][t_stride][head_dim] (all
 * sequences, as kvq_restore writes them), each sequence's length taken from
 * this cache's counters.  The read path the fused kvq_decode_attention
 * replaces, kept as its measured foil ("KV Cache 量化与压缩" section 06 compares
 * the two): q and out as in kvq_decode_attention.  Uses the arena's split
 * scratch region.  Needs a bf16 cache with head_dim 64 or 128, else
 * KVQ_EUNSUPPORTED; KVQ_EINVAL for NULL or misaligned pointers or a t_stride
 * below the largest held length. */
kvq_status kvq_dense_decode_attention(kvq_cache* cache, const void* k, const void* v, int64_t t_stride,
                                      const void* q, float* out, void* stream);

/* The datawhale page's compare ("54. KV Cache Quantization Strategies",
 * compare), on the GPU.  key, value: device [batch][heads][tokens][head_dim]
 * of dtype.  Key is quantized per channel over runs of ``group`` tokens
 * (group = 0: over all ``tokens``, the page's choice; otherwise group must
 * divide tokens), Value per token over head_dim, with the cache's quantizer
 * (scale = qmax / max(absmax, eps), code = clamp(rint(x * scale))); restored as
 * code / max(scale, eps).  The squared errors are rounded in fp32 and summed in
 * fp64 (the order of the sum is not fixed).  The byte counts follow the page
 * (packed bytes assume two codes a byte whatever qmax).  workspace: 16 bytes
 * of 8-byte aligned device memory.  Synchronizes ``stream``.  Errors:
 * KVQ_EINVAL for a bad shape, dtype, qmax, eps, group or pointer;
 * KVQ_EUNSUPPORTED when batch * heads > 65535. */
kvq_status kvq_compare(const void* key, const void* value, int64_t batch, int32_t heads, int64_t tokens,
                       int32_t head_dim, kvq_dtype dtype, int32_t qmax, float eps, int32_t group,
                       void* workspace, kvq_compare_t* out, void* stream);

/* Size in bytes of one group page for this configuration (0 if invalid). */
size_t kvq_page_bytes(const kvq_config* cfg);

/* Kernel launches this library has enqueued in this process so far (all
 * caches, all devices); a monotonically increasing counter for accounting. */
uint64_t kvq_kernel_launches(void);

/* Free the host handle (device memory stays the caller's).  NULL is ignored. */
void kvq_destroy(kvq_cache* cache);

/* Message of the last failed call on this thread ("" if none). */
const char* kvq_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
