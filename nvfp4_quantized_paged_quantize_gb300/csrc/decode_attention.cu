// decode_attention.cu -- paged GQA decode attention over the NVFP4 cache with
// the dequantisation inside the kernel ("nvfp4-kv-cache-memory-wall", section
// 3, item 3: decode dequantises in registers with no separate pass, because
// decode is bound by the KV read; a round trip through memory would read and
// write the whole cache once more).
//
// Work partition (split-K, balanced): the flattened list of (sequence, KV
// head, page) items -- "page-heads" -- is cut into gridDim.x contiguous ranges
// whose sizes differ by at most one, one per CTA, and each CTA range into kNW
// such ranges, one per warp.
// A warp streams its pages through a private ring of kStages shared-memory
// stages.  A page-head is 2304 contiguous bytes of the pool (K data, K scales,
// V data, V scales); all 32 lanes copy it into a stage as it is, in 16-byte
// cp.async pieces, completion counted on one mbarrier per stage.  For each
// page it
//   1. converts K's E2M1 pairs to f16x2 with cvt.rn.f16x2.e2m1x2, multiplies
//      by the E4M3 block scale (exact in f16), and computes S^T = Khat q^T for
//      the 16 tokens x G query heads with mma.sync m16n8k16 (f16 in, f32 acc);
//      two pages of the same pair are taken per step (32 tokens);
//   2. runs the online softmax in base 2 (scores scaled by softmax_scale *
//      log2(e) * g_K, folded into one FMA per score); the running max is only
//      raised when a score exceeds it by more than 8, so the rescale of the
//      accumulators is rare;
//   3. transposes P (f16) with movmatrix and accumulates O^T += Vhat^T P^T,
//      Vhat^T converted straight from V's token-pair bytes (each byte one
//      dimension of two tokens) and scaled per token.
// A (sequence, KV head) pair that lies inside one warp range is finished by
// that warp.  A piece of a pair cut by a warp boundary is written to the
// workspace as a record (unnormalised O, running max m, sum l) and the warp
// is done: no CTA-wide barrier or merge sits at the end of the decode, where
// it would wait on the slowest warp and run cold code under full memory load.
// combine_kernel, launched right behind the decode as a programmatic
// dependent, merges each cut pair's records (the flash-decoding combine); it
// finds them from the split itself, which it rederives from the lengths while
// the decode still runs.
//
// Exactness: e2m1 * E4M3 has at most 6 significant bits in [2^-10, 2688], so
// Khat and Vhat are exact in f16.  q is bf16; it is multiplied by a power of
// two per head so its largest element sits in [2^14, 2^15) before rounding to
// f16, and the factor is folded back into the score scale.
#include <cstdint>

#include "nvfp4kv_device.cuh"
#include "nvfp4kv_launch.h"

namespace nvfp4kv {
namespace {

#ifndef NVFP4KV_DECODE_WARPS
#define NVFP4KV_DECODE_WARPS 4
#endif
#ifndef NVFP4KV_DECODE_STAGES
#define NVFP4KV_DECODE_STAGES 4
#endif
#ifndef NVFP4KV_DECODE_CTAS_PER_SM
#define NVFP4KV_DECODE_CTAS_PER_SM 3
#endif
#ifndef NVFP4KV_DECODE_QK_CHAINS
#define NVFP4KV_DECODE_QK_CHAINS 1  // independent QK accumulator chains per page (1 or 2)
#endif
constexpr int kNW = NVFP4KV_DECODE_WARPS;              // warps per CTA (each streams its own pages)
constexpr int kStages = NVFP4KV_DECODE_STAGES;         // ring stages per warp (2 pages in compute)
constexpr int kCtasPerSm = NVFP4KV_DECODE_CTAS_PER_SM; // resident CTAs per SM the launch is sized for
constexpr int kGMax = 8;        // query heads per KV head (one MMA n-tile)
constexpr float kLazy = 8.0f;   // running-max slack (log2 units): P <= 2^8 in f16

// Cache formats the decode reads: NVFP4; NVFP4 of Hadamard-rotated rows (q is
// rotated on the way in and the output rotated back, both exact orthonormal
// transforms); MXFP4 (blocks of 32 with E8M0 scales, 4 per row).
enum : int { kFmtNvfp4 = 0, kFmtHadamard = 1, kFmtMxfp4 = 2 };

// stage layout: the page-head as stored (K data | K scales | V data | V scales)
constexpr int kOffKD = kOffKData;
__host__ __device__ constexpr int ph_bytes(int F) { return F == kFmtMxfp4 ? kMxPageHeadBytes : kPageHeadBytes; }
__host__ __device__ constexpr int off_vd(int F) { return F == kFmtMxfp4 ? kMxOffVData : kOffVData; }
__host__ __device__ constexpr int off_ks(int F) { return F == kFmtMxfp4 ? kMxOffKScale : kOffKScale; }
__host__ __device__ constexpr int off_vs(int F) { return F == kFmtMxfp4 ? kMxOffVScale : kOffVScale; }
constexpr int kStageBytes = kPageHeadBytes;  // stage stride: the larger page-head (2304)

// a (partial) result record: O[kGMax][128] unnormalised, m[kGMax] (base 2), l[kGMax]
constexpr int kRecFloats = kGMax * kHeadDim + 2 * kGMax;
constexpr int kOffM = kGMax * kHeadDim;
constexpr int kOffL = kGMax * kHeadDim + kGMax;

constexpr int kRingBytes = kNW * kStages * kStageBytes;
constexpr int kBarBytes = kNW * kStages * 8;
constexpr int kSmemBytes = kRingBytes + kBarBytes;

struct DecodeParams {
  const uint8_t* pages;  // [num_pages][hkv][kPageHeadBytes]
  int32_t num_pages;
  int32_t hkv;
  const uint16_t* q;
  float* out;
  const int32_t* page_table;
  int32_t max_pages;
  const int32_t* seq_lens;
  int32_t batch;
  int32_t hq;
  int32_t group;
  float score_scale;  // softmax_scale * log2(e) * g_K
  float v_gscale;     // g_V
  float* part;        // [2 * num_ctas * kNW] records: warp w's first (2w) and last (2w + 1) cut piece
  int32_t* status;
  int32_t* cu_pages;  // [batch + 1], written by CTA 0: pages of the sequences before each, then of all
  int32_t ncta;       // CTAs of the decode grid (its split, rederived by the combine)
  int32_t comb_heads; // query heads per combine block
};

// ---------------------------------------------------------------------------
// small helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ int clamp_len(const DecodeParams& p, int b) {
  int L = __ldg(p.seq_lens + b);
  const int lmax = p.max_pages * kPage;
  if (L < 0 || L > lmax) {
    flag_error(p.status, NVFP4KV_DEVERR_LENGTH);
    L = L < 0 ? 0 : lmax;
  }
  return L;
}

__device__ __forceinline__ int pages_of(const DecodeParams& p, int b) {
  return (clamp_len(p, b) + kPage - 1) / kPage;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(a));
  return r;
}

__device__ __forceinline__ void mma16816(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The same with a zero accumulator: d = a * b (the first MMA of a chain).
__device__ __forceinline__ void mma16816_zero(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

__device__ __forceinline__ uint32_t dup_lo(uint32_t h2) { return __byte_perm(h2, 0, 0x1010); }

// a * (the low or the high half of s, in both halves): the broadcast is left to
// the multiply's operand selection
union H2U {
  uint32_t u;
  __half2 h;
};
template <bool kHi>
__device__ __forceinline__ uint32_t hmul2_bcast(uint32_t a, uint32_t s) {
  H2U x, y, r;
  x.u = a;
  y.u = s;
  r.h = __hmul2(x.h, kHi ? __high2half2(y.h) : __low2half2(y.h));
  return r.u;
}

template <int K>
__device__ __forceinline__ uint32_t cvt_sel(uint32_t w) { return e2m1x2_to_f16x2<K>(w); }

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Balanced partition of W page-heads over N CTAs: the first W % N CTAs take
// W / N + 1, the rest W / N.  (Weighting CTAs by their launch order on an SM,
// whose warp scheduler favours older CTAs by about 5%, balanced the CTAs'
// finish times but did not shorten the launch: the slowest warps are spread
// over all SMs.)
__device__ __forceinline__ long long cta_start(long long c, long long W, long long N) {
  // W < 2^31 (checked on the host): 32-bit division
  const int q = (int)W / (int)N, rem = (int)W - q * (int)N;
  return c * q + (c < rem ? c : rem);
}

// Where each item of a 32-item chunk of a warp's range lives (one per lane).
struct ItemMap {
  int row;     // the page id as loaded; after resolve_chunk the physical row pid * hkv + h, or -1
  int h;       // KV head
  int pair;    // b * hkv + h, -1 past the warp's range
  int page;    // page index within the sequence
  int np;      // pages of the pair
  int lastnv;  // valid tokens in the pair's last page (1..16)
  int nv;      // after resolve_chunk: valid tokens of the item's page (0 for an invalid id or past the range)
};

// The sequence a chunk walk starts from: its index, its first page (in units
// of pages of all earlier sequences) and its clamped length.
struct SeqCursor {
  int b;
  int cu;
  int L;
};

// Map items [i0, i0 + 32) of the warp range starting at wr0 (n items) to pages
// and start the page-table loads; resolve_chunk turns the loaded ids into rows
// later, so the load latency is hidden behind the pages already staged.
// `sc` is a sequence whose first page-head is <= the chunk's first item; on
// return it is the sequence of the chunk's last valid item.
__device__ __forceinline__ ItemMap map_chunk(const DecodeParams& p, long long wr0, int i0, int n, SeqCursor& sc,
                                             int lane) {
  ItemMap m;
  m.row = -1;
  m.h = 0;
  m.pair = -1;
  m.page = 0;
  m.np = 1;
  m.lastnv = kPage;
  m.nv = 0;
  const int i = i0 + lane;
  int b = sc.b, cu = sc.cu, L = sc.L;
  if (i < n) {
    const long long r = wr0 + i;
    int np = (L + kPage - 1) / kPage;
    while (r >= (long long)(cu + np) * p.hkv) {
      cu += np;
      ++b;
      L = clamp_len(p, b);
      np = (L + kPage - 1) / kPage;
    }
    const int local = (int)(r - (long long)cu * p.hkv);
    const int h = local / np;
    const int page = local - h * np;
    m.h = h;
    m.pair = b * p.hkv + h;
    m.page = page;
    m.np = np;
    m.lastnv = L - (np - 1) * kPage;
    m.row = __ldg(p.page_table + (long long)b * p.max_pages + page);
  }
  const int last = min(31, n - 1 - i0);
  sc.b = __shfl_sync(0xFFFFFFFFu, b, last);
  sc.cu = __shfl_sync(0xFFFFFFFFu, cu, last);
  sc.L = __shfl_sync(0xFFFFFFFFu, L, last);
  return m;
}

// Turn the loaded page ids of a chunk map into physical rows (-1 for an id out
// of range, which is flagged); returns the valid-page bits (bit l: lane l).
__device__ __forceinline__ uint32_t resolve_chunk(const DecodeParams& p, ItemMap& m) {
  const bool real = m.pair >= 0;
  const bool valid = real && m.row >= 0 && m.row < p.num_pages;
  if (real && !valid) flag_error(p.status, NVFP4KV_DEVERR_PAGE);
  m.row = valid ? m.row * p.hkv + m.h : -1;
  m.nv = valid ? (m.page == m.np - 1 ? m.lastnv : kPage) : 0;
  return __ballot_sync(0xFFFFFFFFu, valid);
}

// cp.async staging: lane l copies the 16-byte pieces l, l + 32, ... of the
// page-head (NVFP4: lanes 0-15 five of the 144, the others four; MXFP4: lanes
// 0-7 five of the 136), then arrives (no-increment) on the stage's mbarrier,
// which expects 32 arrivals.  The lane's source base and shared-memory offset
// are set up once.
struct LaneCopy {
  const uint8_t* src;  // pages + 16 * lane
  uint32_t off;        // 16 * lane
  bool fifth;          // a fifth piece at 16 * (lane + 128)
};

template <int F>
__device__ __forceinline__ LaneCopy lane_copy(const DecodeParams& p, int lane) {
  LaneCopy c;
  c.src = p.pages + 16 * lane;
  c.off = 16u * lane;
  c.fifth = lane + 128 < ph_bytes(F) / 16;
  return c;
}

// Wait, warp-wide, for a ring stage: one try_wait per lane and a vote when
// the data is there (the usual case); otherwise all lanes retry together
// until the phase completes or about a second has passed (returns false).
__device__ __forceinline__ bool stage_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
      : "=r"(done) : "r"(bar), "r"(parity), "r"(1000000u) : "memory");
  if (__all_sync(0xFFFFFFFFu, done)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
        : "=r"(done) : "r"(bar), "r"(parity), "r"(1000000u) : "memory");
    if (__all_sync(0xFFFFFFFFu, done)) return true;
    if (__shfl_sync(0xFFFFFFFFu, global_timer_ns() - t0 > 1000000000ull ? 1 : 0, 0)) return false;
  }
}

// An item of a warp's range as the loop uses it: the byte offset of its
// page-head in the pool and its valid tokens (0: nothing to copy or attend).
struct alignas(16) ItemEntry {
  long long off;
  int nv;
  int pad;
};

// cp.async staging of one page-head at byte offset `off` of the pool: lane l
// copies the 16-byte pieces l, l + 32, ... (NVFP4: lanes 0-15 five of the 144,
// the others four; MXFP4: lanes 0-7 five of the 136), predicated, none when nv
// is 0, then arrives (no-increment) on the stage's mbarrier, which expects 32
// arrivals; it fires once all of the lane's earlier copies have landed, so a
// stage's barrier covers every stage issued before it as well.
template <int F>
__device__ __forceinline__ void issue_page_off(const LaneCopy& c, long long off, int nv, uint32_t st, uint32_t bar) {
  const uint8_t* src = c.src + off;
  const uint32_t dst = st + c.off;
  const uint32_t v5 = (nv > 0 && c.fifth) ? 1u : 0u;
  asm volatile(
      "{\n .reg .pred p, q;\n"
      " setp.gt.s32 p, %2, 0;\n"
      " setp.ne.u32 q, %3, 0;\n"
      " @p cp.async.cg.shared.global [%0], [%1], 16;\n"
      " @p cp.async.cg.shared.global [%0+512], [%1+512], 16;\n"
      " @p cp.async.cg.shared.global [%0+1024], [%1+1024], 16;\n"
      " @p cp.async.cg.shared.global [%0+1536], [%1+1536], 16;\n"
      " @q cp.async.cg.shared.global [%0+2048], [%1+2048], 16;\n"
      " cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%4];\n"
      "}\n" ::"r"(dst), "l"(src), "r"(nv), "r"(v5), "r"(bar)
      : "memory");
}

// Two NVFP4 page-heads (288 pieces of 16 bytes: 9 per lane), into stages a and
// b: lane l copies pieces l + 32 k of the pair of page-heads, i.e. a's pieces
// l, l + 32, l + 64, l + 96, then a's l + 128 (l < 16) or b's l - 16 (l >= 16),
// then b's l + 16, l + 48, l + 80, l + 112; then arrives on both barriers.
// Nothing is copied for an entry with no valid tokens (a bad page id).
__device__ __forceinline__ void issue_two_off(const LaneCopy& c, const ItemEntry& a, const ItemEntry& b,
                                              uint32_t sta, uint32_t stb, uint32_t bara, uint32_t barb,
                                              bool lo) {
  const uint8_t* srca = c.src + a.off;
  const uint8_t* srcb = c.src + b.off;
  const uint32_t dsta = sta + c.off, dstb = stb + c.off;
  const uint32_t dst4 = lo ? dsta + 2048 : dstb - 256;
  const uint8_t* src4 = lo ? srca + 2048 : srcb - 256;
  const int n4 = lo ? a.nv : b.nv;
  asm volatile(
      "{\n .reg .pred pa, pb, p4;\n"
      " setp.gt.s32 pa, %4, 0;\n"
      " setp.gt.s32 pb, %5, 0;\n"
      " setp.gt.s32 p4, %6, 0;\n"
      " @pa cp.async.cg.shared.global [%0], [%2], 16;\n"
      " @pa cp.async.cg.shared.global [%0+512], [%2+512], 16;\n"
      " @pa cp.async.cg.shared.global [%0+1024], [%2+1024], 16;\n"
      " @pa cp.async.cg.shared.global [%0+1536], [%2+1536], 16;\n"
      " @p4 cp.async.cg.shared.global [%7], [%8], 16;\n"
      " @pb cp.async.cg.shared.global [%1+256], [%3+256], 16;\n"
      " @pb cp.async.cg.shared.global [%1+768], [%3+768], 16;\n"
      " @pb cp.async.cg.shared.global [%1+1280], [%3+1280], 16;\n"
      " @pb cp.async.cg.shared.global [%1+1792], [%3+1792], 16;\n"
      " cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%9];\n"
      " cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%10];\n"
      "}\n" ::"r"(dsta), "r"(dstb), "l"(srca), "l"(srcb), "r"(a.nv), "r"(b.nv), "r"(n4), "r"(dst4), "l"(src4),
      "r"(bara), "r"(barb)
      : "memory");
}

// Per-warp attention state of the current pair.
struct WarpState {
  float o[8][4];    // O^T tiles: tile i rows d = 16g+2i (c0,c1) and 16g+2i+1 (c2,c3), cols heads 2t,2t+1
  uint32_t qf[8][2];  // q B-fragments: tile i holds q[head g][32t+4i .. 32t+4i+3]
  float m0, m1;     // running max (base 2) of heads 2t, 2t+1
  float l0, l1;     // this lane's partial sums of P over its tokens
  float c0, c1;     // score multipliers of heads 2t, 2t+1
};

// Orthonormal Walsh-Hadamard transform (Sylvester order) of the 128 values of
// a row held by a group of lanes: each lane holds N consecutive values (index
// bits below log2 N); passes across lanes pair the lane with lane ^ x for
// each lane mask x in `xs` (index bits above, lowest first), the lower lane
// keeping a + b and the upper a - b.  Then one product with RN(1 / sqrt(128)).
template <int N, int NX>
__device__ __forceinline__ void hadamard_lanes(float (&v)[N], const int (&xs)[NX], int lane) {
#pragma unroll
  for (int h = 1; h < N; h *= 2)
#pragma unroll
    for (int i = 0; i < N; i += 2 * h)
#pragma unroll
      for (int j = i; j < i + h; ++j) {
        const float a = v[j], b = v[j + h];
        v[j] = a + b;
        v[j + h] = a - b;
      }
#pragma unroll
  for (int k = 0; k < NX; ++k) {
    const bool upper = (lane & xs[k]) != 0;
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const float o = __shfl_xor_sync(0xFFFFFFFFu, v[i], xs[k]);
      v[i] = upper ? o - v[i] : v[i] + o;
    }
  }
  const float c = 0x1.6a09e6p-4f;  // RN(1 / sqrt(128))
#pragma unroll
  for (int i = 0; i < N; ++i) v[i] *= c;
}

// 2^d as an f16 for an integer d <= 0 (0 below f16's range): the relative
// weight of an MXFP4 block whose E8M0 exponent is d below the page's largest.
__device__ __forceinline__ uint32_t exp2_f16_bits(int d) {
  if (d >= -14) return (uint32_t)(d + 15) << 10;   // normal
  if (d >= -24) return 1u << (d + 24);             // subnormal
  return 0u;
}

// 2^e as an fp32 for an E8M0 exponent e in [-127, 127].
__device__ __forceinline__ float exp2_f32(int e) {
  return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(0x00400000u);
}

// The bf16 q elements lane (g, t) needs for pair b * hkv + h: head h * G + g,
// elements 32t .. 32t + 31 (zeros for g >= G).  Query heads of pair P start at
// row P * G of q, since hq = hkv * G.
struct QRaw {
  uint4 w[4];
};

__device__ __forceinline__ QRaw fetch_q(const DecodeParams& p, int pair, int g, int t) {
  QRaw r;
  if (g < p.group) {
    const uint4* src = reinterpret_cast<const uint4*>(p.q + ((long long)pair * p.group + g) * kHeadDim + 32 * t);
#pragma unroll
    for (int j = 0; j < 4; ++j) r.w[j] = __ldg(src + j);
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) r.w[j] = make_uint4(0u, 0u, 0u, 0u);
  }
  return r;
}

// Turn fetched q into B-fragments with a per-head power-of-two prescale and
// reset the pair's softmax state.
template <int F>
__device__ __forceinline__ void load_q(const DecodeParams& p, const QRaw& raw, WarpState& s, int g, int t) {
  float qv[32];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint4 w = raw.w[j];
    qv[8 * j + 0] = bf16_to_f32(w.x & 0xFFFFu); qv[8 * j + 1] = bf16_to_f32(w.x >> 16);
    qv[8 * j + 2] = bf16_to_f32(w.y & 0xFFFFu); qv[8 * j + 3] = bf16_to_f32(w.y >> 16);
    qv[8 * j + 4] = bf16_to_f32(w.z & 0xFFFFu); qv[8 * j + 5] = bf16_to_f32(w.z >> 16);
    qv[8 * j + 6] = bf16_to_f32(w.w & 0xFFFFu); qv[8 * j + 7] = bf16_to_f32(w.w >> 16);
  }
  if constexpr (F == kFmtHadamard) {
    // the cache holds NVFP4 of H k for each key k: q . k = (H q) . (H k), so q
    // is rotated once here (lane t holds elements 32t .. 32t + 31: passes 1-16
    // inside the lane, 32 and 64 across lanes t ^ 1 and t ^ 2)
    const int xs[2] = {1, 2};
    hadamard_lanes<32, 2>(qv, xs, (g << 2) | t);
  }
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(qv[j]));
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
  // prescale 2^e so that amax * 2^e lies in [2^14, 2^15); e clamped to +-100
  int e = 0;
  if (amax > 0.0f) {
    const int ex = (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127;  // floor(log2 amax) for normals
    e = 14 - ex;
    e = e > 100 ? 100 : (e < -100 ? -100 : e);
  }
  const float pre = __uint_as_float((uint32_t)(e + 127) << 23);
  const float inv = __uint_as_float((uint32_t)(127 - e) << 23);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    s.qf[i][0] = pack_f16x2(qv[4 * i] * pre, qv[4 * i + 1] * pre);
    s.qf[i][1] = pack_f16x2(qv[4 * i + 2] * pre, qv[4 * i + 3] * pre);
  }
  const float c = p.score_scale * inv;  // score multiplier of head g
  s.c0 = __shfl_sync(0xFFFFFFFFu, c, (2 * t) * 4);
  s.c1 = __shfl_sync(0xFFFFFFFFu, c, (2 * t + 1) * 4);
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) s.o[i][j] = 0.0f;
  s.m0 = s.m1 = -INFINITY;
  s.l0 = s.l1 = 0.0f;
}

// Phase 1 of a step: S^T = Khat q^T for NP pages (16 tokens x G heads each),
// one accumulator chain per page (or two, tiles 0-3 and 4-7, with
// NVFP4KV_DECODE_QK_CHAINS 2: shorter chains, four more adds per page).
// MXFP4 pages carry their scales relative to the page's largest exponent (per
// K and per V, so every product stays inside f16): kx[k] = 2^(K's largest)
// multiplies the page's scores, ve[k] (V's largest) enters the softmax exponent.
struct PageExp {
  float kx;  // 2^ek
  int ve;    // ev
};

template <int NP, int F>
__device__ __forceinline__ void qk_phase(const uint8_t* const (&stage)[NP], const int (&nvalid)[NP],
                                         const WarpState& s, float (&sc)[NP][2][4], PageExp (&pe)[NP], int g,
                                         int t) {
#pragma unroll
  for (int k = 0; k < NP; ++k) {
    const uint8_t* kd = stage[k] + kOffKD;
    const uint8_t* ks = stage[k] + off_ks(F);
    const uint4 ka = *reinterpret_cast<const uint4*>(kd + g * kRowBytes + 16 * t);
    const uint4 kb = *reinterpret_cast<const uint4*>(kd + (g + 8) * kRowBytes + 16 * t);
    uint32_t sa, sb;  // f16x2: the scales of blocks 2t (low half) and 2t + 1 (high half) of rows g, g + 8
    if constexpr (F == kFmtMxfp4) {
      // the lane's 32 values of rows g and g + 8 are one block (t); the 64 K
      // scale bytes of the page are read once over the warp, as are V's
      // (rows at or past the page's valid tokens hold other data: they count as 0)
      const int nv = nvalid[k];
      const int ea = g < nv ? ks[g * kMxRowScales + t] : 0, eb = g + 8 < nv ? ks[(g + 8) * kMxRowScales + t] : 0;
      int ek = max(ea, eb);
      const uint8_t* vsc = stage[k] + off_vs(F) + (g >> 1) * kPage;
      int ev = max(max(2 * t < nv ? vsc[2 * t] : 0, 2 * t + 1 < nv ? vsc[2 * t + 1] : 0),
                   max(2 * t + 8 < nv ? vsc[2 * t + 8] : 0, 2 * t + 9 < nv ? vsc[2 * t + 9] : 0));
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        ek = max(ek, __shfl_xor_sync(0xFFFFFFFFu, ek, off));
        ev = max(ev, __shfl_xor_sync(0xFFFFFFFFu, ev, off));
      }
      pe[k].kx = exp2_f32(ek - 127);
      pe[k].ve = ev - 127;
      sa = dup_lo(exp2_f16_bits(ea - ek));
      sb = dup_lo(exp2_f16_bits(eb - ek));
    } else {
      sa = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(ks + g * kRowScales + 2 * t));
      sb = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(ks + (g + 8) * kRowScales + 2 * t));
      pe[k].kx = 1.0f;
      pe[k].ve = 0;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t wa = word_of(ka, i >> 1), wb = word_of(kb, i >> 1);
      uint32_t a0, a1, a2, a3;
      if (i & 1) {
        a0 = cvt_sel<2>(wa); a1 = cvt_sel<2>(wb); a2 = cvt_sel<3>(wa); a3 = cvt_sel<3>(wb);
      } else {
        a0 = cvt_sel<0>(wa); a1 = cvt_sel<0>(wb); a2 = cvt_sel<1>(wa); a3 = cvt_sel<1>(wb);
      }
      if (i < 4) {
        a0 = hmul2_bcast<false>(a0, sa); a2 = hmul2_bcast<false>(a2, sa);
        a1 = hmul2_bcast<false>(a1, sb); a3 = hmul2_bcast<false>(a3, sb);
      } else {
        a0 = hmul2_bcast<true>(a0, sa); a2 = hmul2_bcast<true>(a2, sa);
        a1 = hmul2_bcast<true>(a1, sb); a3 = hmul2_bcast<true>(a3, sb);
      }
      // chain c = i / 4 (two chains) or 0: its first MMA starts from zero
      const int c = NVFP4KV_DECODE_QK_CHAINS == 2 ? (i >> 2) : 0;
      if (i == 0 || (NVFP4KV_DECODE_QK_CHAINS == 2 && i == 4))
        mma16816_zero(sc[k][c], a0, a1, a2, a3, s.qf[i][0], s.qf[i][1]);
      else
        mma16816(sc[k][c], a0, a1, a2, a3, s.qf[i][0], s.qf[i][1]);
    }
  }

}

// Phase 2: online softmax (base 2) over the NP pages' scores, one running-max
// check for all of them; returns P^T as mma B fragments (k = tokens, n = heads).
template <int NP, bool kFull, int F>
__device__ __forceinline__ void softmax_phase(const float (&sc)[NP][2][4], const PageExp (&pe)[NP],
                                              const int (&nvalid)[NP], WarpState& s, uint32_t (&pb)[NP][2], int g) {
  // raw scores; the running max is kept in scaled (base-2) units: max(S c) = c max(S), c > 0.
  // MXFP4: page k's weights carry 2^ve[k] (its V exponent), folded into the
  // exponent so that P stays within f16; the sums l take it out again.
  float S[NP][4];
  float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
  for (int k = 0; k < NP; ++k) {
#pragma unroll
    for (int j = 0; j < 4; ++j) S[k][j] = NVFP4KV_DECODE_QK_CHAINS == 2 ? sc[k][0][j] + sc[k][1][j] : sc[k][0][j];
    if constexpr (F == kFmtMxfp4) {
#pragma unroll
      for (int j = 0; j < 4; ++j) S[k][j] *= pe[k].kx;
    }
    if (!kFull && nvalid[k] < kPage) {
      if (g >= nvalid[k]) S[k][0] = S[k][1] = -INFINITY;
      if (g + 8 >= nvalid[k]) S[k][2] = S[k][3] = -INFINITY;
    }
    float a0 = fmaxf(S[k][0], S[k][2]) * s.c0, a1 = fmaxf(S[k][1], S[k][3]) * s.c1;
    if constexpr (F == kFmtMxfp4) {
      a0 += (float)pe[k].ve;
      a1 += (float)pe[k].ve;
    }
    mx0 = fmaxf(mx0, a0);
    mx1 = fmaxf(mx1, a1);
  }
  const bool need = (mx0 > s.m0 + kLazy) || (mx1 > s.m1 + kLazy);
  if (__any_sync(0xFFFFFFFFu, need)) {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, off));
    }
    const float n0 = fmaxf(s.m0, mx0), n1 = fmaxf(s.m1, mx1);
    const float f0 = ex2(s.m0 - n0), f1 = ex2(s.m1 - n1);
    s.l0 *= f0;
    s.l1 *= f1;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      s.o[i][0] *= f0; s.o[i][1] *= f1; s.o[i][2] *= f0; s.o[i][3] *= f1;
    }
    s.m0 = n0;
    s.m1 = n1;
  }
  const float nm0 = -s.m0, nm1 = -s.m1;
#pragma unroll
  for (int k = 0; k < NP; ++k) {
    float o0 = nm0, o1 = nm1;
    if constexpr (F == kFmtMxfp4) {
      o0 += (float)pe[k].ve;
      o1 += (float)pe[k].ve;
    }
    const float p0 = ex2(fmaf(S[k][0], s.c0, o0)), p1 = ex2(fmaf(S[k][1], s.c1, o1));
    const float p2 = ex2(fmaf(S[k][2], s.c0, o0)), p3 = ex2(fmaf(S[k][3], s.c1, o1));
    if constexpr (F == kFmtMxfp4) {
      const float un = exp2_f32(-pe[k].ve);  // 2^-ve: the sum counts the plain weights
      s.l0 += (p0 + p2) * un;
      s.l1 += (p1 + p3) * un;
    } else {
      s.l0 += p0 + p2;
      s.l1 += p1 + p3;
    }
    // P^T (tokens x heads) in the accumulator layout -> B fragments (k = tokens, n = heads)
    pb[k][0] = movmatrix_trans(pack_f16x2(p0, p1));
    pb[k][1] = movmatrix_trans(pack_f16x2(p2, p3));
  }
}

// Phase 3: O^T += Vhat^T P^T for the NP pages.
template <int NP, bool kFull, int F>
__device__ __forceinline__ void pv_phase(const uint8_t* const (&stage)[NP], const int (&nvalid)[NP],
                                         const PageExp (&pe)[NP], const uint32_t (&pb)[NP][2], WarpState& s, int g,
                                         int t) {
#pragma unroll
  for (int k = 0; k < NP; ++k) {
    const uint8_t* vd = stage[k] + off_vd(F);
    const uint8_t* vs = stage[k] + off_vs(F);
    const int t0 = 2 * t, t1 = 2 * t + 1, t8 = 2 * t + 8, t9 = 2 * t + 9;
    uint32_t sv01, sv89;  // (token 2t, token 2t+1) and (2t+8, 2t+9) scales of the lane's block, f16x2
    if constexpr (F == kFmtMxfp4) {
      // the lane's 16 values are in block g / 2; its E8M0 exponents relative to the page's largest
      const uint8_t* b = vs + (g >> 1) * kPage;
      const bool full = kFull || nvalid[k] >= kPage;
      const int ve = pe[k].ve + 127;
      const uint32_t e0 = (full || t0 < nvalid[k]) ? exp2_f16_bits(b[t0] - ve) : 0u;
      const uint32_t e1 = (full || t1 < nvalid[k]) ? exp2_f16_bits(b[t1] - ve) : 0u;
      const uint32_t e8 = (full || t8 < nvalid[k]) ? exp2_f16_bits(b[t8] - ve) : 0u;
      const uint32_t e9 = (full || t9 < nvalid[k]) ? exp2_f16_bits(b[t9] - ve) : 0u;
      sv01 = e0 | (e1 << 16);
      sv89 = e8 | (e9 << 16);
    } else {
      // V scales are block-major: block g's scales of tokens (2t, 2t+1) and (2t+8, 2t+9) are adjacent pairs
      uint32_t p01 = *reinterpret_cast<const uint16_t*>(vs + g * kPage + t0);
      uint32_t p89 = *reinterpret_cast<const uint16_t*>(vs + g * kPage + t8);
      if (!kFull && nvalid[k] < kPage) {  // tokens past the end: scale 0 keeps unwritten bytes out of the sum
        if (t0 >= nvalid[k]) p01 &= 0xFF00u;
        if (t1 >= nvalid[k]) p01 &= 0x00FFu;
        if (t8 >= nvalid[k]) p89 &= 0xFF00u;
        if (t9 >= nvalid[k]) p89 &= 0x00FFu;
      }
      sv01 = e4m3x2_to_f16x2(p01);
      sv89 = e4m3x2_to_f16x2(p89);
    }
    // V data by token pair: pair t holds tokens (2t, 2t+1), pair t + 4 tokens
    // (2t+8, 2t+9); bytes 16g .. 16g + 15 of a pair row are dimensions 16g ..
    // 16g + 15, each byte the two tokens' codes of one dimension: one E2M1
    // conversion gives an A-operand register (k = the two tokens) as it is
    const uint4 w01 = *reinterpret_cast<const uint4*>(vd + t * kVPairBytes + 16 * g);
    const uint4 w89 = *reinterpret_cast<const uint4*>(vd + (t + 4) * kVPairBytes + 16 * g);
    const uint32_t pb0 = pb[k][0], pb1 = pb[k][1];
    // tile I: rows g and g + 8 are dimensions 16g + 2I and 16g + 2I + 1, bytes
    // 2I and 2I + 1 of the lane's 16
#define NVFP4KV_PV_TILE(I, W01, W89, K0, K1)                                    \
  {                                                                             \
    const uint32_t a0 = hmul2(cvt_sel<K0>(W01), sv01);                          \
    const uint32_t a1 = hmul2(cvt_sel<K1>(W01), sv01);                          \
    const uint32_t a2 = hmul2(cvt_sel<K0>(W89), sv89);                          \
    const uint32_t a3 = hmul2(cvt_sel<K1>(W89), sv89);                          \
    mma16816(s.o[I], a0, a1, a2, a3, pb0, pb1);                                 \
  }
    NVFP4KV_PV_TILE(0, w01.x, w89.x, 0, 1)
    NVFP4KV_PV_TILE(1, w01.x, w89.x, 2, 3)
    NVFP4KV_PV_TILE(2, w01.y, w89.y, 0, 1)
    NVFP4KV_PV_TILE(3, w01.y, w89.y, 2, 3)
    NVFP4KV_PV_TILE(4, w01.z, w89.z, 0, 1)
    NVFP4KV_PV_TILE(5, w01.z, w89.z, 2, 3)
    NVFP4KV_PV_TILE(6, w01.w, w89.w, 0, 1)
    NVFP4KV_PV_TILE(7, w01.w, w89.w, 2, 3)
#undef NVFP4KV_PV_TILE
  }
}

// NP pages of one KV head (16 tokens each, nvalid[k] of them valid) from ring
// stages, folded into the warp's running softmax state with one max update.
// kFull: every page has all 16 tokens (no masking code).
template <int NP, bool kFull, int F>
__device__ __forceinline__ void process_pages(const uint8_t* const (&stage)[NP], const int (&nvalid)[NP],
                                              WarpState& s, int g, int t) {
  float sc[NP][2][4];
  uint32_t pb[NP][2];
  PageExp pe[NP];
  qk_phase<NP, F>(stage, nvalid, s, sc, pe, g, t);
  softmax_phase<NP, kFull, F>(sc, pe, nvalid, s, pb, g);
  pv_phase<NP, kFull, F>(stage, nvalid, pe, pb, s, g, t);
}

// Finish a warp's piece of a pair: total l over the lanes, then either write
// the final output (complete pair) or store the piece's record at `slot`.
template <int F>
__device__ __forceinline__ void finish_piece(const DecodeParams& p, WarpState& s, int pair, bool complete,
                                             float* slot, int g, int t) {
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    s.l0 += __shfl_xor_sync(0xFFFFFFFFu, s.l0, off);
    s.l1 += __shfl_xor_sync(0xFFFFFFFFu, s.l1, off);
  }
  const int h0 = 2 * t, h1 = 2 * t + 1;
  if (complete) {
    const int b = pair / p.hkv, h = pair - (pair / p.hkv) * p.hkv;
    float* base = p.out + ((long long)b * p.hq + (long long)h * p.group) * kHeadDim;
    const float r0 = s.l0 > 0.0f ? p.v_gscale / s.l0 : 0.0f;
    const float r1 = s.l1 > 0.0f ? p.v_gscale / s.l1 : 0.0f;
    // the lane's values of heads 2t and 2t + 1: d = 16 g + k, k = 0 .. 15
    float v0[16], v1[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v0[2 * i] = s.o[i][0] * r0; v0[2 * i + 1] = s.o[i][2] * r0;
      v1[2 * i] = s.o[i][1] * r1; v1[2 * i + 1] = s.o[i][3] * r1;
    }
    if constexpr (F == kFmtHadamard) {
      // rotate the output back (d bits 0-3 in the lane, 4-6 across lanes g: lane ^ 4, 8, 16)
      const int xs[3] = {4, 8, 16};
      hadamard_lanes<16, 3>(v0, xs, (g << 2) | t);
      hadamard_lanes<16, 3>(v1, xs, (g << 2) | t);
    }
    if (h0 < p.group) {
      float4* dst = reinterpret_cast<float4*>(base + h0 * kHeadDim + 16 * g);
#pragma unroll
      for (int j = 0; j < 4; ++j) dst[j] = make_float4(v0[4 * j], v0[4 * j + 1], v0[4 * j + 2], v0[4 * j + 3]);
    }
    if (h1 < p.group) {
      float4* dst = reinterpret_cast<float4*>(base + h1 * kHeadDim + 16 * g);
#pragma unroll
      for (int j = 0; j < 4; ++j) dst[j] = make_float4(v1[4 * j], v1[4 * j + 1], v1[4 * j + 2], v1[4 * j + 3]);
    }
  } else {
    float4* d0 = reinterpret_cast<float4*>(slot + h0 * kHeadDim + 16 * g);
    float4* d1 = reinterpret_cast<float4*>(slot + h1 * kHeadDim + 16 * g);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      d0[j] = make_float4(s.o[2 * j][0], s.o[2 * j][2], s.o[2 * j + 1][0], s.o[2 * j + 1][2]);
      d1[j] = make_float4(s.o[2 * j][1], s.o[2 * j][3], s.o[2 * j + 1][1], s.o[2 * j + 1][3]);
    }
    if (g == 0) {
      slot[kOffM + h0] = s.m0;
      slot[kOffM + h1] = s.m1;
      slot[kOffL + h0] = s.l0;
      slot[kOffL + h1] = s.l1;
    }
  }
}

__device__ __forceinline__ long long block_sum_ll(long long v, long long* red, int warp, int lane) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  long long total = 0;
#pragma unroll
  for (int w = 0; w < kNW; ++w) total += red[w];
  __syncthreads();
  return total;
}

template <int F>
__global__ void __launch_bounds__(kNW * 32, kCtasPerSm) decode_kernel(const DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kRingBytes);
  __shared__ long long red[kNW];
  __shared__ int wstart_b[kNW], wstart_cu[kNW];
  // per warp: (page-head row, valid tokens) of items [32 chunk, 32 chunk + 64),
  // item k at k % 64, written as each 32-item chunk map is resolved
  __shared__ ItemEntry s_items[kNW][64];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  // the combine kernel may be scheduled now: its blocks take SMs as decode CTAs
  // retire and wait (griddepcontrol.wait) for the whole decode grid
  asm volatile("griddepcontrol.launch_dependents;");

  // ---- prologue: total work, zero outputs of empty sequences -------------------
  {
    // bring q and the page table into L2 early (each CTA a slice, 128-byte
    // lines): the first chunk maps and later pieces then find them there
    // instead of queueing behind the KV stream
    const long long step = (long long)gridDim.x * blockDim.x, first = (long long)blockIdx.x * blockDim.x + tid;
    const long long qlines = ((long long)p.batch * p.hq * kHeadDim * 2 + 127) / 128;
    for (long long l = first; l < qlines; l += step)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const uint8_t*>(p.q) + 128 * l));
    const long long plines = ((long long)p.batch * p.max_pages * 4 + 127) / 128;
    for (long long l = first; l < plines; l += step)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const uint8_t*>(p.page_table) + 128 * l));
  }
  long long W = 0;
  long long r0 = 0, r1 = 0;
  const long long N = gridDim.x;
  if (p.batch <= kNW * 32) {
    // one pass: every sequence's length is read once, by thread b
    const int b = tid;
    int np = 0;
    if (b < p.batch) {
      const int L = clamp_len(p, b);
      np = (L + kPage - 1) / kPage;
      if (L == 0 && (b % (int)gridDim.x) == (int)blockIdx.x) {
        float4* o = reinterpret_cast<float4*>(p.out + (long long)b * p.hq * kHeadDim);
        for (int j = 0; j < p.hq * kHeadDim / 4; ++j) o[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    int incl = np;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, off);
      if (lane >= off) incl += v;
    }
    if (lane == 31) red[warp] = incl;
    __syncthreads();
    long long before = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kNW; ++w) {
      if (w < warp) before += red[w];
      total += red[w];
    }
    W = total * p.hkv;
    if (W == 0) return;
    r0 = cta_start(blockIdx.x, W, N);
    r1 = cta_start((long long)blockIdx.x + 1, W, N);
    const int excl = (int)before + incl - np;
    if (blockIdx.x == 0 && b < p.batch) p.cu_pages[b] = excl;
    if (blockIdx.x == 0 && tid == 0) p.cu_pages[p.batch] = (int)total;
    if (np > 0) {
      for (int w2 = 0; w2 < kNW; ++w2) {
        const long long ws = r0 + (r1 - r0) * w2 / kNW, we = r0 + (r1 - r0) * (w2 + 1) / kNW;
        if (ws < we && ws >= (long long)excl * p.hkv && ws < (long long)(excl + np) * p.hkv) {
          wstart_b[w2] = b;
          wstart_cu[w2] = excl;
        }
      }
    }
    __syncthreads();
  } else {
    long long pages_local = 0;
    for (int b = tid; b < p.batch; b += kNW * 32) {
      const int L = clamp_len(p, b);
      pages_local += (L + kPage - 1) / kPage;
      if (L == 0 && (b % (int)gridDim.x) == (int)blockIdx.x) {
        float4* o = reinterpret_cast<float4*>(p.out + (long long)b * p.hq * kHeadDim);
        for (int j = 0; j < p.hq * kHeadDim / 4; ++j) o[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    W = block_sum_ll(pages_local, red, warp, lane) * p.hkv;
    if (W == 0) return;
    r0 = cta_start(blockIdx.x, W, N);
    r1 = cta_start((long long)blockIdx.x + 1, W, N);

    // locate the sequence holding each warp's first page-head
    int carry = 0;
    for (int base = 0; base < p.batch; base += kNW * 32) {
      const int b = base + tid;
      const int np = b < p.batch ? pages_of(p, b) : 0;
      int incl = np;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += v;
      }
      if (lane == 31) red[warp] = incl;
      __syncthreads();
      int before = carry, chunk = 0;
#pragma unroll
      for (int w = 0; w < kNW; ++w) {
        if (w < warp) before += (int)red[w];
        chunk += (int)red[w];
      }
      const int excl = before + incl - np;
      if (blockIdx.x == 0 && b < p.batch) p.cu_pages[b] = excl;
      if (np > 0) {
        for (int w2 = 0; w2 < kNW; ++w2) {
          const long long ws = r0 + (r1 - r0) * w2 / kNW, we = r0 + (r1 - r0) * (w2 + 1) / kNW;
          if (ws < we && ws >= (long long)excl * p.hkv && ws < (long long)(excl + np) * p.hkv) {
            wstart_b[w2] = b;
            wstart_cu[w2] = excl;
          }
        }
      }
      carry += chunk;
      __syncthreads();
    }
    if (blockIdx.x == 0 && tid == 0) p.cu_pages[p.batch] = carry;
  }

  // ---- per-warp streaming over its page-heads ----------------------------------
  const long long wr0 = r0 + (r1 - r0) * warp / kNW;
  const long long wr1 = r0 + (r1 - r0) * (warp + 1) / kNW;
  const int n = (int)(wr1 - wr0);
  uint8_t* wring = ring + warp * kStages * kStageBytes;
  const uint32_t wbar = smem_u32(bars + warp * kStages);
  const long long gwarp = (long long)blockIdx.x * kNW + warp;  // global warp index

  if (n == 0 && lane < kGMax) {
    // a warp with no items lies between the pieces of a cut pair when a CTA's
    // range is shorter than kNW: its first record is marked empty (m = -inf),
    // which the combine skips
    p.part[2 * gwarp * kRecFloats + kOffM + lane] = -INFINITY;
  }
  if (n > 0) {
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s) mbar_init(wbar + 8 * s, 32);
      fence_mbar_init();
    }
    __syncwarp();
    SeqCursor seq;
    seq.b = wstart_b[warp];
    seq.cu = wstart_cu[warp];
    seq.L = clamp_len(p, seq.b);
    ItemMap cur = map_chunk(p, wr0, 0, n, seq, lane);
    // the first piece's q goes out before the ring prefill, so it does not
    // queue behind the pages
    const QRaw q_first = fetch_q(p, __shfl_sync(0xFFFFFFFFu, cur.pair, 0), g, t);
    ItemMap nxt = cur;
    bool nres = true;  // nxt has been resolved (or is not used)
    if (n > 32) {
      nxt = map_chunk(p, wr0, 32, n, seq, lane);
      nres = false;
    }
    ItemEntry* const tab = s_items[warp];
    // an item's entry: computed by its lane once per chunk, used by the loop
    auto entry_of = [&](const ItemMap& m) {
      ItemEntry e;
      e.off = m.row < 0 ? 0 : (long long)m.row * ph_bytes(F);
      e.nv = m.nv;
      e.pad = 0;
      return e;
    };
    resolve_chunk(p, cur);
    tab[lane] = entry_of(cur);
    __syncwarp();

    // Launched right behind the append of the same decode step
    // (nvfp4kv_append_decode_attention), this grid ran everything above while
    // the append was still writing the new tokens' pages: wait for it before
    // the first page is read.  Without a prerequisite grid this returns at once.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // producer: prefill the ring (all within the first chunk: kStages < 32)
    const int pre = n < kStages ? n : kStages;
    const LaneCopy lc = lane_copy<F>(p, lane);
    const uint32_t wring_u32 = smem_u32(wring);
    for (int j = 0; j < pre; ++j) {
      issue_page_off<F>(lc, tab[j].off, tab[j].nv, wring_u32 + j * kStageBytes, wbar + 8 * j);
    }
    int issued = pre;
    int chunk = 0;   // the chunk `cur` maps
    int st = 0;      // ring stage of the next item
    uint32_t ph = 0; // its mbarrier phase parity
    WarpState s;
    load_q<F>(p, q_first, s, g, t);  // the first piece's q, fetched before the prefill
    int nseg = 0;
    int i = 0;
    // resolve the next chunk's map into the item table
#define NVFP4KV_RESOLVE_NXT()                                          \
  {                                                                     \
    resolve_chunk(p, nxt);                                              \
    tab[(32 * (chunk + 1) + lane) & 63] = entry_of(nxt);                \
    __syncwarp();                                                       \
  }
    // the chunk maps hold items [32 chunk, 32 chunk + 64): move them up to item k
#define NVFP4KV_ADVANCE_TO(k)                                   \
  while (((k) >> 5) != chunk) {                                 \
    if (!nres) NVFP4KV_RESOLVE_NXT();                           \
    cur = nxt;                                                  \
    ++chunk;                                                    \
    nres = true;                                                \
    if ((chunk + 1) * 32 < n) {                                 \
      nxt = map_chunk(p, wr0, (chunk + 1) * 32, n, seq, lane);  \
      nres = false;                                             \
    }                                                           \
  }
    while (i < n) {
      // ---- one piece: items [i, iend) of one (sequence, KV head) pair -------------
      NVFP4KV_ADVANCE_TO(i)
      const int li = i & 31;
      const int pair = __shfl_sync(0xFFFFFFFFu, cur.pair, li);
      const int page0 = __shfl_sync(0xFFFFFFFFu, cur.page, li);
      const int np = __shfl_sync(0xFFFFFFFFu, cur.np, li);
      const int iend = min(n, i + (np - page0));
      ++nseg;
      if (nseg > 1) load_q<F>(p, fetch_q(p, pair, g, t), s, g, t);
      int j = i;
      // the next item at which the chunk maps need work: the next chunk's start,
      // or half way through this chunk while the next one's rows are unresolved
#define NVFP4KV_NEXT_EVENT() (nres ? 32 * (chunk + 1) : min(32 * (chunk + 1), 32 * chunk + 16))
      int ev = NVFP4KV_NEXT_EVENT();
      // two pages per step
      for (; j + 1 < iend; j += 2) {
        if (j >= ev) {
          NVFP4KV_ADVANCE_TO(j)
          // the next chunk's rows are first needed at item 32 chunk + 32 - kStages - 1;
          // resolving them half way through the chunk leaves their loads time to land
          if (!nres && (j & 31) >= 16) {
            NVFP4KV_RESOLVE_NXT();
            nres = true;
          }
          ev = NVFP4KV_NEXT_EVENT();
        }
        const int st1 = st + 1 == kStages ? 0 : st + 1;
        const uint32_t ph1 = st1 == 0 ? ph ^ 1u : ph;
        // The second stage's barrier fires only after each lane's earlier copies
        // (those of the first stage) have landed too, so one wait covers both.
        if (!stage_wait(wbar + 8 * st1, ph1)) goto timed_out;
        {
          const int nv0 = tab[j & 63].nv, nv1 = tab[(j + 1) & 63].nv;
          const uint8_t* const stg[2] = {wring + st * kStageBytes, wring + st1 * kStageBytes};
          const int nvs[2] = {nv0, nv1};
          if ((nv0 & nv1) == kPage)
            process_pages<2, true, F>(stg, nvs, s, g, t);
          else if (nv0 | nv1)
            process_pages<2, false, F>(stg, nvs, s, g, t);
          __syncwarp();
          // refill the freed stages with items j + kStages and j + 1 + kStages
          const int ja = j + kStages, jb = ja + 1;
          if (jb < n) {
            const ItemEntry ea = tab[ja & 63], eb = tab[jb & 63];
            if constexpr (F == kFmtMxfp4) {
              issue_page_off<F>(lc, ea.off, ea.nv, wring_u32 + st * kStageBytes, wbar + 8 * st);
              issue_page_off<F>(lc, eb.off, eb.nv, wring_u32 + st1 * kStageBytes, wbar + 8 * st1);
            } else {
              issue_two_off(lc, ea, eb, wring_u32 + st * kStageBytes, wring_u32 + st1 * kStageBytes,
                            wbar + 8 * st, wbar + 8 * st1, lane < 16);
            }
            issued = jb + 1;
          } else if (ja < n) {
            issue_page_off<F>(lc, tab[ja & 63].off, tab[ja & 63].nv, wring_u32 + st * kStageBytes, wbar + 8 * st);
            issued = ja + 1;
          }
        }
        st = st1 + 1 == kStages ? 0 : st1 + 1;
        ph = st == 0 ? ph1 ^ 1u : ph1;
      }
      if (j < iend) {
        // the piece's last page on its own
        NVFP4KV_ADVANCE_TO(j)
        if (!nres && (j & 31) >= 16) {
          NVFP4KV_RESOLVE_NXT();
          nres = true;
        }
        if (!stage_wait(wbar + 8 * st, ph)) goto timed_out;
        {
          const int nv0 = tab[j & 63].nv;
          const uint8_t* const stg[2] = {wring + st * kStageBytes, wring + st * kStageBytes};
          const int nvs[2] = {nv0, 0};
          if (nv0) process_pages<2, false, F>(stg, nvs, s, g, t);
          __syncwarp();
          const int ja = j + kStages;
          if (ja < n) {
            issue_page_off<F>(lc, tab[ja & 63].off, tab[ja & 63].nv, wring_u32 + st * kStageBytes, wbar + 8 * st);
            issued = ja + 1;
          }
        }
        st = st + 1 == kStages ? 0 : st + 1;
        ph = st == 0 ? ph ^ 1u : ph;
        ++j;
      }
#undef NVFP4KV_NEXT_EVENT
#undef NVFP4KV_ADVANCE_TO
#undef NVFP4KV_RESOLVE_NXT
      __syncwarp();
      // a piece that ends before the warp range does is complete unless it is the
      // first; a cut piece becomes record 2 gwarp (the warp's first piece) or
      // 2 gwarp + 1 (its last piece), merged later by combine_kernel
      const int last_page = page0 + (iend - i) - 1;
      const bool complete = page0 == 0 && last_page == np - 1;
      const int slot = (iend == n && nseg > 1) ? 1 : 0;
      finish_piece<F>(p, s, pair, complete, p.part + (2 * gwarp + slot) * kRecFloats, g, t);
      i = iend;
    }
    return;
  timed_out:
    // a wait gave up: flag it, wait (bounded) for every copy still in flight so
    // that none lands after the warp has gone, and leave; the call's outputs
    // are then unspecified, but every access stays in bounds
    if (lane == 0) flag_error(p.status, kDevErrTimeout);
    for (int jj = issued - kStages; jj < issued; ++jj) {
      if (jj < 0) continue;
      mbar_wait(wbar + 8 * (jj % kStages), (uint32_t)((jj / kStages) & 1));
    }
  }
}

// Merge the records of every pair the warp ranges cut: block = (pair, a chunk
// of its query heads), warp = (query head, record group), thread = 4 columns.
// Group k of a head takes records k, k + groups, ... with an online rescale,
// then group 0 merges the groups' partial results.  Launched as a
// programmatic dependent of decode_kernel: griddepcontrol.wait returns once
// the decode grid has finished and its writes are visible; what comes before
// it reads only the call's inputs.
constexpr int kCombineMaxGroups = 16;

__device__ __forceinline__ void online_merge(float& M, float& L, float4& acc, float m, float l, float4 v) {
  const float Mn = fmaxf(M, m);
  const float a = M == -INFINITY ? 0.0f : ex2(M - Mn);
  const float b = m == -INFINITY ? 0.0f : ex2(m - Mn);
  L = L * a + l * b;
  acc.x = acc.x * a + v.x * b;
  acc.y = acc.y * a + v.y * b;
  acc.z = acc.z * a + v.z * b;
  acc.w = acc.w * a + v.w * b;
  M = Mn;
}

// The split's arithmetic in 32 bits, for W < 2^31 page-heads (the combine's use).
__device__ __forceinline__ int cta_start32(int c, int W, int N) {
  const int q = W / N, rem = W - q * N;
  return c * q + (c < rem ? c : rem);
}
__device__ __forceinline__ int warp_of_item32(int r, int W, int N) {
  const int q = W / N, rem = W - q * N, big = rem * (q + 1);
  const int c = r < big ? r / (q + 1) : rem + (r - big) / q;
  const int r0 = cta_start32(c, W, N), len = cta_start32(c + 1, W, N) - r0;
  return c * kNW + (int)(((long long)(r - r0 + 1) * kNW - 1) / len);
}

// A sequence's length as the decode clamps it (without flagging: the decode does).
__device__ __forceinline__ int clamped_len(const DecodeParams& p, int b) {
  const int L = __ldg(p.seq_lens + b), lmax = p.max_pages * kPage;
  return L < 0 ? 0 : (L > lmax ? lmax : L);
}

// Block = (pair, chunk of its query heads); warp = (head, record group).
constexpr int kCombineMaxWarps = 32;
constexpr int kCombineScanMax = 1024;  // batches up to this size: the combine sums the lengths itself

template <int F>
__global__ void __launch_bounds__(kCombineMaxWarps * 32) combine_kernel(const DecodeParams p) {
  __shared__ float s_m[kCombineMaxWarps][32], s_l[kCombineMaxWarps][32];
  __shared__ float4 s_o[kCombineMaxWarps][32];
  __shared__ int s_info[3];  // first record, first warp, record count (0: nothing to merge)
  const int pair = blockIdx.x;
  const int b = pair / p.hkv, hh = pair - b * p.hkv;
  const int warp = threadIdx.x >> 5, col = threadIdx.x & 31;
  const int hb = p.comb_heads;                 // query heads per block
  const int groups = (blockDim.x >> 5) / hb;   // record groups per head
  const int hl = warp % hb, grp = warp / hb;
  const int head = blockIdx.y * hb + hl;
  // Where the pair lies in the decode's split, worked out by warp 0 in 32-bit
  // arithmetic (page-head indices stay below 2^31): the pages of the sequences
  // before b and of all sequences, then the warps holding the pair's first and
  // last page-heads.  For up to kCombineScanMax sequences the pages come from
  // the lengths, inputs of the call, so this runs while the decode is still
  // streaming; for more, from the prefix the decode's CTA 0 wrote (after the
  // wait), which keeps the work per block independent of the batch.
  const bool scan = p.batch <= kCombineScanMax;
  if (warp == 0) {
    int before = 0, total = 0;
    if (scan) {
      for (int i = col; i < p.batch; i += 32) {
        const int npi = (clamped_len(p, i) + kPage - 1) / kPage;
        total += npi;
        before += i < b ? npi : 0;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        total += __shfl_xor_sync(0xFFFFFFFFu, total, off);
        before += __shfl_xor_sync(0xFFFFFFFFu, before, off);
      }
    }
    if (col == 0) {
      const int np = (clamped_len(p, b) + kPage - 1) / kPage;
      int rec0 = 0, wf = 0, cnt = 0;
      if (np > 0) {
        if (!scan) {
          asm volatile("griddepcontrol.wait;" ::: "memory");
          before = __ldcg(p.cu_pages + b);
          total = __ldcg(p.cu_pages + p.batch);
        }
        const int W = total * p.hkv, N = p.ncta;
        const int P0 = before * p.hkv + hh * np;  // the pair's first page-head
        wf = warp_of_item32(P0, W, N);
        const int wl = warp_of_item32(P0 + np - 1, W, N);
        if (wl != wf) {
          // the first piece is warp wf's last piece (record 2 wf + 1), or its
          // only one when the pair starts wf's range (record 2 wf); every later
          // warp up to wl holds one piece as its first (record 2 w)
          const int cf = wf / kNW, r0c = cta_start32(cf, W, N), r1c = cta_start32(cf + 1, W, N);
          const int wr0 = r0c + (int)((long long)(r1c - r0c) * (wf - cf * kNW) / kNW);
          rec0 = 2 * wf + (P0 > wr0 ? 1 : 0);
          cnt = wl - wf + 1;
        }
      }
      s_info[0] = rec0;
      s_info[1] = wf;
      s_info[2] = cnt;
    }
  }
  __syncthreads();
  const int rec0 = s_info[0], wf = s_info[1], cnt = s_info[2];
  if (cnt == 0) return;  // an empty sequence (the decode wrote its zeros) or one warp held the whole pair
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // warp (head, grp) merges the head's records grp, grp + groups, ...: four at
  // a time, all loads issued before any is used (a warp of the decode with no
  // items marked its record m = -inf)
  float M = -INFINITY, L = 0.0f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (head < p.group) {
    for (int c0 = grp; c0 < cnt; c0 += 4 * groups) {
      float m[4], l[4];
      float4 v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int c = c0 + i * groups;
        m[i] = -INFINITY;
        l[i] = 0.0f;
        v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c < cnt) {
          const float* r = p.part + (c == 0 ? (long long)rec0 : 2LL * (wf + c)) * kRecFloats;
          m[i] = __ldcg(r + kOffM + head);
          l[i] = __ldcg(r + kOffL + head);
          v[i] = __ldcg(reinterpret_cast<const float4*>(r + head * kHeadDim) + col);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) online_merge(M, L, acc, m[i], l[i], v[i]);
    }
  }
  s_m[warp][col] = M;
  s_l[warp][col] = L;
  s_o[warp][col] = acc;
  __syncthreads();
  if (grp != 0 || head >= p.group) return;
  for (int k = 1; k < groups; ++k) {
    const int w2 = k * hb + hl;
    online_merge(M, L, acc, s_m[w2][col], s_l[w2][col], s_o[w2][col]);
  }
  const float sc = L > 0.0f ? p.v_gscale / L : 0.0f;
  float v[4] = {acc.x * sc, acc.y * sc, acc.z * sc, acc.w * sc};
  if constexpr (F == kFmtHadamard) {
    // rotate the merged output back (d bits 0-1 in the thread, 2-6 across the warp's 32 columns)
    const int xs[5] = {1, 2, 4, 8, 16};
    hadamard_lanes<4, 5>(v, xs, col);
  }
  reinterpret_cast<float4*>(p.out + ((long long)pair * p.group + head) * kHeadDim)[col] =
      make_float4(v[0], v[1], v[2], v[3]);
}

}  // namespace

int decode_num_ctas(int num_sms) { return num_sms * kCtasPerSm; }

size_t decode_workspace_bytes(int num_sms, int32_t batch, int32_t num_kv_heads) {
  size_t rec = 2 * (size_t)decode_num_ctas(num_sms) * kNW * kRecFloats * sizeof(float);
  (void)num_kv_heads;
  rec = (rec + 255) / 256 * 256;
  return rec + ((size_t)batch + 1) * sizeof(int32_t);
}

size_t decode_workspace_bound(int num_sms, int32_t batch, int32_t num_q_heads) {
  return decode_workspace_bytes(num_sms, batch, num_q_heads);
}

namespace {

template <int F>
cudaError_t launch_decode_fmt(const nvfp4kv_cache& c, const uint16_t* q, float* out, const int32_t* page_table,
                              int32_t max_pages, const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                              float softmax_scale, void* workspace, int32_t* device_status, int num_sms,
                              cudaStream_t stream, bool after_kernel) {
  // the shared-memory limit is an attribute of the function on each device
  static PerDeviceOnce attr_once;
  const cudaError_t ae = attr_once.run([] {
    return cudaFuncSetAttribute(decode_kernel<F>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  });
  if (ae != cudaSuccess) return ae;
  const int num_ctas = decode_num_ctas(num_sms);
  DecodeParams p;
  p.pages = c.pages;
  p.num_pages = (int32_t)c.num_pages;
  p.hkv = c.num_kv_heads;
  p.q = q;
  p.out = out;
  p.page_table = page_table;
  p.max_pages = max_pages;
  p.seq_lens = seq_lens;
  p.batch = batch;
  p.hq = num_q_heads;
  p.group = num_q_heads / c.num_kv_heads;
  // MXFP4 has no global scales: its blocks carry power-of-two scales alone
  const float gk = F == kFmtMxfp4 ? 1.0f : c.k_global_scale, gv = F == kFmtMxfp4 ? 1.0f : c.v_global_scale;
  p.score_scale = softmax_scale * 1.4426950408889634f * gk;
  p.v_gscale = gv;
  const size_t pairs = (size_t)batch * (size_t)c.num_kv_heads;
  size_t rec = 2 * (size_t)num_ctas * kNW * kRecFloats * sizeof(float);
  rec = (rec + 255) / 256 * 256;
  p.part = static_cast<float*>(workspace);
  p.cu_pages = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + rec);
  p.status = device_status;
  p.ncta = num_ctas;
  cudaError_t e;
  if (after_kernel) {
    // a programmatic dependent of the kernel before it on the stream
    cudaLaunchConfig_t dc = {};
    dc.gridDim = dim3((unsigned)num_ctas);
    dc.blockDim = dim3(kNW * 32);
    dc.dynamicSmemBytes = kSmemBytes;
    dc.stream = stream;
    cudaLaunchAttribute da[1];
    da[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    da[0].val.programmaticStreamSerializationAllowed = 1;
    dc.attrs = da;
    dc.numAttrs = 1;
    e = cudaLaunchKernelEx(&dc, decode_kernel<F>, p);
  } else {
    decode_kernel<F><<<num_ctas, kNW * 32, kSmemBytes, stream>>>(p);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess || pairs == 0) return e;
  // the combine, as a programmatic dependent of the decode on the same stream
  // records per cut pair are about (warps / pairs) when the sequences are
  // alike: give each thread a handful of them
  // records per cut pair are about (warps / pairs) when the sequences are
  // alike: a record group per four to eight of them, up to 16 groups per head,
  // and as many of the pair's query heads per block as fit 32 warps
  const long long per_pair = (2LL * num_ctas * kNW) / (long long)pairs;
  int groups = 1;
  while (groups < kCombineMaxGroups && groups * 8 < per_pair) groups *= 2;
  const int hb = p.group < kCombineMaxWarps / groups ? p.group : kCombineMaxWarps / groups;
  p.comb_heads = hb;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)pairs, (unsigned)((p.group + hb - 1) / hb));
  cfg.blockDim = dim3(32 * hb * groups);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, combine_kernel<F>, p);
  return e;
}

}  // namespace

cudaError_t launch_decode(const nvfp4kv_cache& c, const uint16_t* q, float* out, const int32_t* page_table,
                          int32_t max_pages, const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                          float softmax_scale, void* workspace, int32_t* device_status, int num_sms,
                          cudaStream_t stream, bool after_kernel) {
  return launch_decode_fmt<kFmtNvfp4>(c, q, out, page_table, max_pages, seq_lens, batch, num_q_heads, softmax_scale,
                                      workspace, device_status, num_sms, stream, after_kernel);
}

cudaError_t launch_decode_variant(int variant, const nvfp4kv_cache& c, const uint16_t* q, float* out,
                                  const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                                  int32_t batch, int32_t num_q_heads, float softmax_scale, void* workspace,
                                  int32_t* device_status, int num_sms, cudaStream_t stream) {
  if (variant == NVFP4KV_VARIANT_HADAMARD)
    return launch_decode_fmt<kFmtHadamard>(c, q, out, page_table, max_pages, seq_lens, batch, num_q_heads,
                                           softmax_scale, workspace, device_status, num_sms, stream, false);
  if (variant == NVFP4KV_VARIANT_MXFP4)
    return launch_decode_fmt<kFmtMxfp4>(c, q, out, page_table, max_pages, seq_lens, batch, num_q_heads,
                                        softmax_scale, workspace, device_status, num_sms, stream, false);
  // stochastic rounding writes the plain NVFP4 format
  return launch_decode_fmt<kFmtNvfp4>(c, q, out, page_table, max_pages, seq_lens, batch, num_q_heads, softmax_scale,
                                      workspace, device_status, num_sms, stream, false);
}

}  // namespace nvfp4kv
