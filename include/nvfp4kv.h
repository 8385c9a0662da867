/*
 * nvfp4kv.h -- C ABI of libnvfp4kv.so: an NVFP4 paged KV cache on one GB300
 * (sm_103a).
 *
 * Format ("nvfp4-kv-cache-memory-wall", section 2, two-level scaling; "NVFP4:
 * breaking the memory wall", technical breakdown): each value is a 4-bit E2M1
 * code (1 sign, 2 exponent, 1 mantissa bit: +-{0,0.5,1,1.5,2,3,4,6}); every 16
 * consecutive values of one token and one head (along head_dim) share one
 * FP8 E4M3 block scale; each tensor (one layer's K, or its V) has one FP32
 * global scale g.  A value dequantises to e2m1 * e4m3 * g.  Storage is 9/16
 * byte per value ("nvfp4-kv-cache-memory-wall", section 1).
 *
 * Quantisation of one block (the amax of the block lands on E2M1's 6):
 *     sb   = E4M3_rne_satfinite(amax / (6 * g))
 *     code = E2M1_rne_satfinite(x / (E4M3val(sb) * g))
 * each step one IEEE binary32 operation rounded to nearest; rounding ties go
 * to the even code; a block whose E4M3val(sb) * g is 0 stores signed zeros.
 * Inputs (K, V, q) must be finite; non-finite inputs give unspecified codes
 * and outputs (never an out-of-bounds access).
 *
 * Cache layout (one caller-owned device pool, byte-addressed):
 *     pages : uint8 [num_pages][num_kv_heads][NVFP4KV_PAGE_HEAD_BYTES]
 * One page-head (16 tokens of one KV head of one page) is 2304 contiguous
 * bytes, and the page-heads of a page follow one another, so a whole page
 * (every KV head) is one contiguous run of num_kv_heads * 2304 bytes:
 *     [   0, 1024)  K data    16 rows x 64 bytes; element 2i of a row in the
 *                             low nibble of byte i
 *     [1024, 1152)  K scales  16 rows x 8 E4M3 bytes; scale j covers elements
 *                             16j..16j+15 of the row
 *     [1152, 2176)  V data    by token pair: 8 rows x 128 bytes; byte d of
 *                             row p holds element d of token 2p in its low
 *                             nibble and element d of token 2p + 1 in its
 *                             high nibble (the decode's P.V product pairs
 *                             two tokens of one element)
 *     [2176, 2304)  V scales  block-major: 8 blocks x 16 tokens, the scale of
 *                             block j of row r at 2176 + 16 j + r
 * A slot s is row (s % page_size) of page (s / page_size).  Supported:
 * head_dim = 128, page_size = 16.  The pool must be 16-byte aligned (256-byte
 * alignment lets every page-head start on a 128-byte line).
 *
 * Conventions for every call:
 *   - All pointers named device are CUDA device pointers; the library never
 *     allocates, frees or synchronises, and never keeps a pointer past a call.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and is asynchronous with respect to the host.  Calls keep no
 *     state between them and may be made from several host threads.
 *   - The return value is a host-side status (NVFP4KV_OK or an NVFP4KV_ERR_*
 *     code).  Argument errors are detected on the host before anything is
 *     enqueued; nothing is written then.
 *   - Indices read on the device (slots, page ids, lengths) are range-checked
 *     by the kernels.  An out-of-range index skips the access it guards (see
 *     each call) and, if `device_status` is not NULL, ORs an NVFP4KV_DEVERR_*
 *     bit into that device int32 (the caller zeroes it and reads it back).
 */
#ifndef NVFP4KV_H
#define NVFP4KV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, declared without CUDA headers. */
typedef struct CUstream_st* nvfp4kv_stream_t;

/* Host-side status codes. */
enum {
  NVFP4KV_OK = 0,
  NVFP4KV_ERR_INVALID_ARGUMENT = -1, /* null pointer, bad size, misaligned pool, bad scale */
  NVFP4KV_ERR_UNSUPPORTED = -2,      /* head_dim != 128, page_size != 16, a GQA group the call
                                        does not take (decode: > 8; extend: not a power of two
                                        <= 128), or sizes whose indices would not fit */
  NVFP4KV_ERR_CUDA = -3,             /* a CUDA runtime call or launch failed */
  NVFP4KV_ERR_WORKSPACE = -4         /* workspace null, too small or misaligned */
};

/* Format variants of nvfp4kv_quantize_append_variant. */
enum {
  NVFP4KV_VARIANT_SR = 1,       /* NVFP4 with stochastically rounded E2M1 codes */
  NVFP4KV_VARIANT_HADAMARD = 2, /* NVFP4 of the Hadamard-rotated head vector */
  NVFP4KV_VARIANT_MXFP4 = 3     /* MXFP4: blocks of 32, E8M0 scales (4 per row) */
};

/* Device-side error bits (ORed into *device_status when it is given). */
enum {
  NVFP4KV_DEVERR_SLOT = 1,   /* a slot >= num_pages * page_size: that token was skipped */
  NVFP4KV_DEVERR_PAGE = 2,   /* a page id outside [0, num_pages): that page was skipped */
  NVFP4KV_DEVERR_LENGTH = 4, /* a length < 0 or > max_pages_per_seq * page_size: clamped */
  NVFP4KV_DEVERR_TIMEOUT = 8, /* a copy into shared memory (or a tensor-core step) did not
                                 complete within ~1 s: the call's outputs are not valid */
  NVFP4KV_DEVERR_ROW = 16     /* a workspace row outside [0, total_rows): that row was skipped
                                 (an attention key reads as zero) */
};

/* Bytes of one page-head: 16 rows of K data and scales, then of V (9/16 byte
 * per value). */
#define NVFP4KV_PAGE_HEAD_BYTES 2304
/* Bytes of one page-head of the MXFP4 variant's pool (4 E8M0 scale bytes per
 * row): K data [0, 1024), K scales [1024, 1088) token-major, V data
 * [1088, 2112) by token pair as in the NVFP4 page-head, V scales
 * [2112, 2176) block-major (block j of row r at 2112 + 16 j + r). */
#define NVFP4KV_MXFP4_PAGE_HEAD_BYTES 2176

/* One layer's paged NVFP4 cache.  The struct itself is read on the host only. */
typedef struct nvfp4kv_cache {
  uint8_t* pages;       /* device, [num_pages][num_kv_heads][NVFP4KV_PAGE_HEAD_BYTES] */
  int64_t num_pages;    /* > 0 */
  int32_t num_kv_heads; /* > 0 */
  int32_t head_dim;     /* 128 */
  int32_t page_size;    /* 16 */
  float k_global_scale; /* g of K: finite, > 0 (the public setting is 1.0) */
  float v_global_scale; /* g of V: finite, > 0 */
} nvfp4kv_cache;

/*
 * Bytes of the pool of a cache of this shape:
 * num_pages * num_kv_heads * page_size * 2 * (head_dim/2 + head_dim/16), i.e.
 * 9/16 byte per K or V value ("nvfp4-kv-cache-memory-wall", section 1).
 * Host only.  Returns NVFP4KV_OK, NVFP4KV_ERR_INVALID_ARGUMENT (null output,
 * non-positive sizes, head_dim not a multiple of 16) or NVFP4KV_ERR_UNSUPPORTED
 * (a size that overflows).
 */
int nvfp4kv_cache_bytes(int64_t num_pages, int32_t num_kv_heads, int32_t head_dim,
                        int32_t page_size, size_t* pool_bytes);

/*
 * Quantise new K and V tokens into the cache ("nvfp4-kv-cache-memory-wall",
 * section 3, flowchart and item 1: new K/V are written to the cache as NVFP4;
 * nmedialink repost of NVIDIA's blog, figure 3: new keys and values are
 * quantised before they are appended).
 *   k, v          device bf16 [num_tokens][num_kv_heads][head_dim], rows contiguous
 *   slot_mapping  device int64 [num_tokens]; token t goes to slot slot_mapping[t];
 *                 a negative slot skips the token (padding); a slot past the
 *                 pool skips the token and raises NVFP4KV_DEVERR_SLOT
 *   num_tokens    >= 0 (0 enqueues nothing)
 * K uses cache->k_global_scale and V uses cache->v_global_scale.  Two tokens
 * mapped to one slot race: that row's bytes are unspecified (they may mix
 * the two tokens).  Any other slot mapping is exact, including the two tokens
 * of a pair of rows (2m, 2m + 1) written by different calls or in any order
 * within one call.
 */
int nvfp4kv_quantize_append(const nvfp4kv_cache* cache, const void* k, const void* v,
                            const int64_t* slot_mapping, int64_t num_tokens,
                            int32_t* device_status, nvfp4kv_stream_t stream);

/*
 * Bytes of device workspace nvfp4kv_decode_attention needs for this batch
 * shape on the current CUDA device: split-K partial results, two per warp of
 * the launch (so they depend on the device's SM count, not on the batch), and
 * one 4-byte page prefix per sequence.  Host only; query it with the device
 * current that will run the decode.
 */
int nvfp4kv_decode_workspace_size(const nvfp4kv_cache* cache, int32_t batch, int32_t num_q_heads,
                                  size_t* bytes);

/*
 * The same size from the batch shape alone, for callers that size the
 * workspace before a cache exists: bytes enough for any cache with
 * num_q_heads / G KV heads, on a device with num_sms SMs (pass that device's
 * cudaDevAttrMultiProcessorCount).  num_q_heads and max_seq_len are checked
 * and otherwise unused: the split-K partition cuts the pages of all sequences
 * together into as many ranges as the device runs at once, so the scratch
 * depends on the SM count and the batch, not on any length or head count.
 * Host only; returns 0 for batch < 0, num_q_heads <= 0 or num_sms <= 0.
 */
size_t nvfp4kv_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t max_seq_len,
                                      int32_t num_sms);

/*
 * Paged decode attention with the NVFP4 dequantisation inside the kernel
 * ("nvfp4-kv-cache-memory-wall", section 3, item 3: decode dequantises in
 * registers, with no separate dequantisation pass, because decode is bound by
 * the KV read).  For every sequence b and query head h (KV head h / G,
 * G = num_q_heads / num_kv_heads):
 *     s_t = softmax_scale * sum_d q[b,h,d] * Khat[t,d]      t < seq_lens[b]
 *     out[b,h,:] = sum_t softmax(s)_t * Vhat[t,:]
 * over the dequantised cache (Khat = e2m1*e4m3*g_K, Vhat = e2m1*e4m3*g_V).
 *   q               device bf16 [batch][num_q_heads][head_dim]
 *   out             device fp32 [batch][num_q_heads][head_dim]; a sequence of
 *                   length 0 gets zeros
 *   page_table      device int32 [batch][max_pages_per_seq]; row b lists the
 *                   pages of sequence b in token order; entries past
 *                   ceil(seq_lens[b]/page_size) are not read
 *   seq_lens        device int32 [batch]
 *   softmax_scale   finite, > 0 (usually 1/sqrt(head_dim))
 *   workspace       device, >= nvfp4kv_decode_workspace_size() bytes, 256-byte
 *                   aligned; scratch that needs no initialisation (each call
 *                   writes every byte of it that it reads).  Calls that
 *                   overlap on the GPU must not share a workspace.
 * Requires 1 <= G <= 8.  A page id out of range is skipped (its tokens do
 * not take part) with NVFP4KV_DEVERR_PAGE; a length out of range is clamped
 * with NVFP4KV_DEVERR_LENGTH.
 * Enqueues two kernels on `stream`: the split-K decode, then (batch > 0) a
 * combine of the partial results of pairs the split cut, launched as a
 * programmatic dependent of the decode.
 */
int nvfp4kv_decode_attention(const nvfp4kv_cache* cache, const void* q, float* out,
                             const int32_t* page_table, int32_t max_pages_per_seq,
                             const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                             float softmax_scale, void* workspace, size_t workspace_bytes,
                             int32_t* device_status, nvfp4kv_stream_t stream);

/*
 * One decode step in one call: nvfp4kv_quantize_append of the step's new tokens
 * followed by nvfp4kv_decode_attention over the cache that now holds them
 * ("nvfp4-kv-cache-memory-wall", section 3: the new token's K/V are quantised
 * into the cache, then decode attends over it; nmedialink repost of NVIDIA's
 * blog, figure 3).  The results are exactly those of the two calls made one
 * after the other on `stream`.
 *
 * The decode is launched as a programmatic dependent of the append: its set-up
 * (reading seq_lens, page_table and q, splitting the work, zeroing the outputs
 * of empty sequences) overlaps the append, and it waits for the append to
 * finish before it reads any page of the cache.  So q, page_table and seq_lens
 * must be ready when the call is enqueued (as for any stream-ordered call),
 * and none of them may alias the new k, v or slot_mapping.
 *
 * Arguments are those of nvfp4kv_quantize_append (k .. num_tokens) and of
 * nvfp4kv_decode_attention (q .. workspace_bytes), with one device_status for
 * both.  All arguments are checked before anything is enqueued.
 */
int nvfp4kv_append_decode_attention(const nvfp4kv_cache* cache, const void* k, const void* v,
                                    const int64_t* slot_mapping, int64_t num_tokens, const void* q, float* out,
                                    const int32_t* page_table, int32_t max_pages_per_seq,
                                    const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                                    float softmax_scale, void* workspace, size_t workspace_bytes,
                                    int32_t* device_status, nvfp4kv_stream_t stream);

/* Bytes of the fixed device scratch used by nvfp4kv_decode_attention_static. */
#define NVFP4KV_STATIC_SCRATCH_BYTES ((size_t)32 << 20)

/*
 * nvfp4kv_decode_attention without a caller-provided workspace, for callers
 * that cannot allocate device memory (for example code running inside an
 * allocator hook, or a plug-in whose host runtime owns all device memory).
 * The source pages have no counterpart to this call; it only changes where
 * the decode's split-K scratch lives.
 *
 * The scratch is a fixed NVFP4KV_STATIC_SCRATCH_BYTES (32 MiB) array in the
 * library's device image: every GPU that loads the library holds it until the
 * process exits.  The first call on each device looks up the array's device
 * address (cudaGetSymbolAddress) with that device current; make that first
 * call before any stream capture.  Each call then runs exactly what
 * nvfp4kv_decode_attention runs, whose scratch needs no clearing between
 * calls.  Nothing is allocated or freed.
 *
 * All calls share the one array, which keeps the last call's contents: calls
 * that overlap on the GPU (different streams, or different host threads
 * without ordering) race and give wrong results; serialise them.
 *
 * Arguments, layout and errors are those of nvfp4kv_decode_attention without
 * `workspace` / `workspace_bytes`.  A batch whose workspace would exceed the
 * fixed scratch (see nvfp4kv_decode_workspace_size: about 4.59 million
 * sequences on 152 SMs) returns NVFP4KV_ERR_WORKSPACE before anything is
 * enqueued.
 */
int nvfp4kv_decode_attention_static(const nvfp4kv_cache* cache, const void* q, float* out,
                                    const int32_t* page_table, int32_t max_pages_per_seq,
                                    const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                                    float softmax_scale, int32_t* device_status,
                                    nvfp4kv_stream_t stream);

/*
 * Dequantise cached prefixes into an FP8 E4M3 workspace for chunked prefill /
 * extend ("nvfp4-kv-cache-memory-wall", section 3, item 2: the NVFP4 prefix is
 * dequantised into one FP8 workspace pair that every layer reuses, so the
 * workspace does not eat the memory NVFP4 saved).  For token t < prefix_lens[b]
 * of sequence b, head h, element d:
 *     ws[cu_prefix[b] + t][h][d] = E4M3_rne_satfinite(fp32(fp32(e2m1*e4m3) * g) / ws_scale)
 * (sign kept, so -0 is 0x80); a consumer multiplies by ws_scale to recover
 * e2m1*e4m3*g.
 *   page_table      device int32 [batch][max_pages_per_seq]
 *   prefix_lens     device int32 [batch]
 *   cu_prefix       device int64 [batch + 1], non-decreasing, with
 *                   cu_prefix[b] + prefix_lens[b] <= cu_prefix[b+1] and
 *                   cu_prefix[batch] <= total_rows; rows between a prefix's end
 *                   and the next sequence's start are left untouched
 *   total_rows      rows of each workspace (host value)
 *   k_ws_scale, v_ws_scale   finite, > 0
 *   ws_k, ws_v      device uint8 E4M3 [total_rows][num_kv_heads][head_dim],
 *                   16-byte aligned
 * A page id out of range writes zeros for its rows with NVFP4KV_DEVERR_PAGE.
 */
int nvfp4kv_dequant_to_fp8_workspace(const nvfp4kv_cache* cache, const int32_t* page_table,
                                     int32_t max_pages_per_seq, const int32_t* prefix_lens,
                                     const int64_t* cu_prefix, int32_t batch, int64_t total_rows,
                                     float k_ws_scale, float v_ws_scale, uint8_t* ws_k,
                                     uint8_t* ws_v, int32_t* device_status,
                                     nvfp4kv_stream_t stream);

/* Chunked prefill / extend over the FP8 workspace ("nvfp4-kv-cache-memory-
 * wall", section 3, item 2 and the data-flow figure: the chunk attends over its
 * cached prefix, dequantised into the FP8 workspace that every layer reuses,
 * and over itself; the current tokens' own K/V take part as FP8).
 *
 * nvfp4kv_bf16_to_fp8_workspace writes the chunk's own K/V rows into the
 * workspace: ws[ws_rows[t]][h][d] = E4M3(fp32(x) / s_ws), round to nearest
 * even, sign kept, saturating at +-448 (one correctly rounded binary32
 * division).  Usually ws_rows[t] = cu_prefix[b] + prefix_lens[b] + (t's
 * position in its chunk), right after the rows nvfp4kv_dequant_to_fp8_workspace
 * wrote.
 *   k_bf16, v_bf16  device bf16 [num_tokens][num_kv_heads][head_dim], 16-byte aligned
 *   ws_rows         device int64 [num_tokens]; < 0 skips the token; a row
 *                   >= total_rows is skipped with NVFP4KV_DEVERR_ROW
 *   head_dim        128 (else NVFP4KV_ERR_UNSUPPORTED)
 *   k_ws_scale, v_ws_scale   finite, > 0
 *   ws_k, ws_v      device uint8 E4M3 [total_rows][num_kv_heads][head_dim], 16-byte aligned
 *
 * nvfp4kv_extend_attention: for sequence b, chunk token t (query row
 * cu_q[b] + t) and query head h (KV head h / G, G = num_q_heads /
 * num_kv_heads), out = softmax(softmax_scale * q . K^T) V over keys
 * j = 0 .. prefix_lens[b] + t (causal after the prefix), key j being workspace
 * row cu_prefix[b] + j dequantised as E4M3val(w) * s_ws.  Computed on the
 * tensor cores with f16 operands (E4M3 -> f16 is exact; q is rounded to f16,
 * exact for 2^-14 <= |q| <= 65504) and f32 accumulation; the probabilities
 * are rounded to f16 for the P V product.
 *   q_bf16        device bf16 [total_q][num_q_heads][head_dim], 16-byte aligned
 *   cu_q          device int64 [batch + 1], non-decreasing
 *   max_q_len     host: >= every chunk length (a longer chunk is cut to it,
 *                 with NVFP4KV_DEVERR_LENGTH); 0 does nothing
 *   ws_k, ws_v    device uint8 E4M3 [total_rows][num_kv_heads][head_dim], 16-byte aligned
 *   cu_prefix     device int64 [batch]: first workspace row of each sequence
 *   prefix_lens   device int32 [batch]: cached keys of each sequence (>= 0)
 *   G             a power of two <= 128 (else NVFP4KV_ERR_UNSUPPORTED);
 *                 batch and num_kv_heads <= 65535
 *   out           device fp32 [total_q][num_q_heads][head_dim], 16-byte aligned
 * A key row outside [0, total_rows) reads as zero with NVFP4KV_DEVERR_ROW. */
/* nvfp4kv_quantize_append_fp8 is nvfp4kv_quantize_append and
 * nvfp4kv_bf16_to_fp8_workspace of the same tokens in one pass over k and v
 * (each bf16 value is read once): the initial-prefill write ("nvfp4-kv-cache-
 * memory-wall", section 3, item 1: the prompt's K/V enter attention as FP8 and
 * are quantised to NVFP4 for later use at the same time), and the extend
 * chunk's write.  Arguments and errors as in the two calls; both outputs are
 * bit-identical to theirs.  The attention of an initial prefill is
 * nvfp4kv_extend_attention with prefix_lens = 0. */
int nvfp4kv_quantize_append_fp8(const nvfp4kv_cache* cache, const void* k, const void* v,
                                const int64_t* slot_mapping, int64_t num_tokens, const int64_t* ws_rows,
                                int64_t total_rows, float k_ws_scale, float v_ws_scale, uint8_t* ws_k,
                                uint8_t* ws_v, int32_t* device_status, nvfp4kv_stream_t stream);
int nvfp4kv_bf16_to_fp8_workspace(const void* k_bf16, const void* v_bf16, const int64_t* ws_rows,
                                  int64_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                                  int64_t total_rows, float k_ws_scale, float v_ws_scale, uint8_t* ws_k,
                                  uint8_t* ws_v, int32_t* device_status, nvfp4kv_stream_t stream);
int nvfp4kv_extend_attention(const void* q_bf16, const int64_t* cu_q, int32_t max_q_len,
                             const uint8_t* ws_k, const uint8_t* ws_v, const int64_t* cu_prefix,
                             const int32_t* prefix_lens, int32_t batch, int64_t total_rows,
                             int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                             float k_ws_scale, float v_ws_scale, float softmax_scale, float* out,
                             int32_t* device_status, nvfp4kv_stream_t stream);

/* Quantize-on-append of the format variants the pages compare with NVFP4
 * ("NVFP4: breaking the memory wall" (cloud.tencent.com): stochastic rounding
 * and a Hadamard rotation before quantisation, MXFP4's 32-value blocks;
 * "NVIDIA NVFP4: LLM memory doubled, inference 3x" (nmedialink), figure 6).
 * Same rows, slots and errors as nvfp4kv_quantize_append.  The SR and Hadamard
 * variants write the NVFP4 pool layout; MXFP4 writes its own page-heads of
 * NVFP4KV_MXFP4_PAGE_HEAD_BYTES (cache->pages is then
 * [num_pages][num_kv_heads][NVFP4KV_MXFP4_PAGE_HEAD_BYTES]).
 *   NVFP4KV_VARIANT_SR        the block scale as in NVFP4; each element code
 *                             rounds to one of its two E2M1 neighbours, up iff
 *                             (r + 0.5) / 256 < (|y| - a) / (b - a) for the
 *                             input byte r of that value (rand_k / rand_v:
 *                             device uint8 [num_tokens][num_kv_heads][head_dim],
 *                             16-byte aligned)
 *   NVFP4KV_VARIANT_HADAMARD  NVFP4 of H x, H the orthonormal Walsh-Hadamard
 *                             transform of the 128-value head vector (Sylvester
 *                             order; binary32 butterfly passes h = 1 .. 64, then
 *                             one product with RN(1 / sqrt(128))); a reader
 *                             applies H again (or rotates q the same way)
 *   NVFP4KV_VARIANT_MXFP4     blocks of 32 with a power-of-two scale, the E8M0
 *                             byte e + 127, e = floor(log2 amax) - 2 (clamped to
 *                             [-127, 127]); elements E2M1(x * 2^-e); each row
 *                             has head_dim / 32 = 4 scale bytes and the global
 *                             scales are not used
 * Unknown variants return NVFP4KV_ERR_INVALID_ARGUMENT. */
int nvfp4kv_quantize_append_variant(int variant, const nvfp4kv_cache* cache, const void* k, const void* v,
                                    const int64_t* slot_mapping, int64_t num_tokens, const uint8_t* rand_k,
                                    const uint8_t* rand_v, int32_t* device_status, nvfp4kv_stream_t stream);

/* Decode attention over a format variant's cache, so that each variant's
 * accuracy and decode throughput can be set beside NVFP4's ("NVFP4: breaking
 * the memory wall" (cloud.tencent.com), quantisation techniques; "NVIDIA
 * NVFP4: LLM memory doubled, inference 3x" (nmedialink), figure 6).  The same
 * attention as nvfp4kv_decode_attention, over the rows the variant's append
 * wrote:
 *   NVFP4KV_VARIANT_SR        the pool is NVFP4 (stochastically rounded codes):
 *                             exactly nvfp4kv_decode_attention
 *   NVFP4KV_VARIANT_HADAMARD  the pool holds NVFP4 of H k and H v (H the
 *                             orthonormal 128-point Walsh-Hadamard transform,
 *                             its own inverse): the keys and values are
 *                             H Khat and H Vhat.  q is rotated once (q . H k =
 *                             H q . k) and the output rotated back, in fp32
 *   NVFP4KV_VARIANT_MXFP4     the pool holds MXFP4 page-heads
 *                             (NVFP4KV_MXFP4_PAGE_HEAD_BYTES): values
 *                             e2m1 * 2^(s - 127), global scales not used.
 *                             Within a page-head, blocks more than 24 binades
 *                             below the page's largest scale of K (or V)
 *                             read as zero (their weight is < 2^-21 of it)
 * Arguments, workspace (nvfp4kv_decode_workspace_size), layout and errors as
 * in nvfp4kv_decode_attention.  Unknown variants return
 * NVFP4KV_ERR_INVALID_ARGUMENT. */
int nvfp4kv_decode_attention_variant(int variant, const nvfp4kv_cache* cache, const void* q, float* out,
                                     const int32_t* page_table, int32_t max_pages_per_seq,
                                     const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                                     float softmax_scale, void* workspace, size_t workspace_bytes,
                                     int32_t* device_status, nvfp4kv_stream_t stream);

/* Global-scale calibration ("nvfp4-kv-cache-memory-wall", section 2: the
 * FP32 per-tensor scale is 1 in the uncalibrated public setting; a calibrated
 * scale maps the tensor's largest magnitude onto the largest NVFP4 magnitude,
 * E2M1 6 times E4M3 448).
 *
 * nvfp4kv_tensor_amax writes max |x| over n bf16 values into *amax, a device
 * float; the result is exact (a bf16 value) and is +0 when n == 0.  NaN inputs
 * count as magnitudes above every finite value and infinity (their bit
 * patterns are larger), so a NaN input gives a NaN amax.
 *   x_bf16      device bf16 [n], 16-byte aligned (may be NULL when n == 0)
 *   n           >= 0
 *   amax        device float, 4-byte aligned
 *   accumulate  0: *amax is zeroed on the stream first; else *amax must hold
 *               +0 or an earlier result and becomes max(*amax, max |x|), so one
 *               scale can be calibrated over many tensors (all of a layer's
 *               sequences) without a host round trip
 * Asynchronous on stream: read *amax after synchronising.
 *
 * nvfp4kv_calibrated_global_scale is host-only and synchronous:
 * *g = amax / 2688 in one binary32 division (round to nearest even), or 1 when
 * amax == 0 (an all-zero tensor keeps the uncalibrated scale).  amax must be
 * finite and >= 0, else NVFP4KV_ERR_INVALID_ARGUMENT and *g is untouched.
 * The result is the k_global_scale / v_global_scale of a cache whose K or V is
 * that tensor. */
int nvfp4kv_tensor_amax(const void* x_bf16, int64_t n, float* amax, int accumulate,
                        nvfp4kv_stream_t stream);
int nvfp4kv_calibrated_global_scale(float amax, float* g);

/* Streaming probe (a measurement aid, not part of the method): reads every
 * cached page-head of a decode batch once, with no attention math, so that the
 * decode's time can be set against the time its bytes take to stream alone
 * ("nvfp4-kv-cache-memory-wall", section 3, item 3: decode is bound by the KV
 * read).  Arguments as in nvfp4kv_decode_attention; sink is a device uint32
 * that receives an XOR of one word per page (keeps the reads alive).
 *   NVFP4KV_PROBE_DECODE_PATTERN  the decode's grid, split over warps, per-warp
 *                                 rings of 2304-byte page-heads copied by
 *                                 16-byte cp.async pieces, bounded waits
 *   NVFP4KV_PROBE_WHOLE_PAGES     every KV head of a page as one contiguous bulk
 *                                 copy (TMA), one warp per CTA, two CTAs per SM
 *                                 (num_kv_heads <= 16)
 * Both split the pages statically and evenly.  A page id or length out of
 * range is flagged as in the decode; a wait that gives up (~1 s) sets
 * NVFP4KV_DEVERR_TIMEOUT. */
enum { NVFP4KV_PROBE_DECODE_PATTERN = 0, NVFP4KV_PROBE_WHOLE_PAGES = 1 };
int nvfp4kv_stream_probe(const nvfp4kv_cache* cache, const int32_t* page_table, int32_t max_pages_per_seq,
                         const int32_t* seq_lens, int32_t batch, int mode, uint32_t* sink,
                         int32_t* device_status, nvfp4kv_stream_t stream);

/* Text of the CUDA error behind this thread's latest NVFP4KV_ERR_CUDA (the
 * runtime's own message; "no CUDA error" if there was none).  Never NULL. */
const char* nvfp4kv_last_cuda_error(void);

/* A static, human-readable string for a status code (never NULL). */
const char* nvfp4kv_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4KV_H */
