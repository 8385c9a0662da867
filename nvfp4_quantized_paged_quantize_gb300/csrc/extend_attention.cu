// extend_attention.cu -- chunked prefill / extend over the FP8 workspace
// ("nvfp4-kv-cache-memory-wall", section 3, item 2 and the data-flow figure:
// the cached NVFP4 prefix is dequantised into one FP8 workspace that every
// layer reuses; the chunk attends over that prefix and over itself, its own
// K/V taking part as FP8).
//
// chunk_to_ws_kernel: the chunk's bf16 K/V rows -> workspace rows
//   w = E4M3(fp32(x) / s_ws), signed, saturating.  HBM-bound: 2 B read and
//   1 B written per value.
//
// extend_attention_kernel: causal attention of the chunk's queries over their
// sequence's workspace rows (key j = row cu_prefix[b] + j; chunk token t sees
// keys 0 .. prefix + t), on the fifth-generation tensor cores, run by CTA
// pairs (clusters of two, on two SMs) with the pair form of the MMA.
//   - A CTA owns 128 query rows of one (sequence, KV head): 128 / G tokens x
//     the G query heads that share the KV head, so each K/V tile feeds all G;
//     a pair owns two adjacent such m-tiles (256 rows).
//   - Warps 4-7 of each CTA write its Q rows (f16) into its TMEM, then load
//     its half of each K/V tile of 128 keys (one tile ahead, into registers):
//     keys 64 rank .. +63 of K and head dims 64 rank .. +63 of V, convert E4M3
//     -> f16 (exact) and store them as B operands in shared memory (K K-major,
//     V MN-major) in a six-stage ring.  Each K/V byte is converted once per
//     256 query rows.
//   - Warp 8 of rank 0 issues, from one thread, S = Q K^T and O += P V for
//     the pair (M = 256): A (Q, P) is read from each CTA's TMEM, B from both
//     CTAs' halves, f32 accumulators land in each CTA's TMEM (two S buffers,
//     one O); each group is committed to the mbarrier of that name in both
//     CTAs.
//   - Warps 0-3 own one query row per thread (TMEM lane = row): they read the
//     S row, mask, run a lazy base-2 online softmax (the running max moves
//     only when it grows by 2^8, rescaling O in TMEM), and write P (f16) into
//     TMEM.  At the end: O * s_ws(V) / l -> fp32 out.
// Every wait is bounded: a stalled pipeline flags NVFP4KV_DEVERR_TIMEOUT,
// drains its MMAs, and both CTAs meet at a cluster barrier before freeing
// their TMEM.
#include "nvfp4kv_device.cuh"
#include "nvfp4kv_launch.h"
#include "fp8_quotient.cuh"
#include "tcgen05.cuh"

namespace nvfp4kv {
namespace {

// ---------------------------------------------------------------------------
// chunk K/V -> FP8 workspace rows
// ---------------------------------------------------------------------------

struct ChunkParams {
  const uint16_t* k;
  const uint16_t* v;
  const int64_t* rows;
  int64_t units;        // 16-byte input units of one tensor: tokens * hkv * 16
  int32_t units_per_token;
  int64_t total_rows;
  float sk, sv, rsk, rsv;
  bool sk_fast, sv_fast;
  uint8_t* ws_k;
  uint8_t* ws_v;
  int32_t* status;
};

constexpr int kChunkThreads = 256;

// fp32(x) / s rounded to E4M3 for 8 bf16 values; x / 1 is x itself.
__device__ __forceinline__ uint2 bf16x8_to_e4m3(const uint4& x, float s, float rs, bool fast, bool unit) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    o[i] = e4m3x2_from_quotients(bf16_to_f32(w[i] & 0xFFFFu), bf16_to_f32(w[i] >> 16), s, rs, fast, unit);
  return make_uint2(o[0] | (o[1] << 16), o[2] | (o[3] << 16));
}

template <bool kUnit>
__global__ void __launch_bounds__(kChunkThreads) chunk_to_ws_kernel(ChunkParams p) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < 2 * p.units; u += stride) {
    const int tensor = u >= p.units;  // 0: K, 1: V
    const int64_t uu = tensor ? u - p.units : u;
    const int64_t tok = uu / p.units_per_token;
    const int64_t row = __ldg(p.rows + tok);
    if (row < 0) continue;  // padding
    if (row >= p.total_rows) {
      flag_error(p.status, NVFP4KV_DEVERR_ROW);
      continue;
    }
    const uint4 x = __ldg(reinterpret_cast<const uint4*>(tensor ? p.v : p.k) + uu);
    const uint2 e = tensor ? bf16x8_to_e4m3(x, p.sv, p.rsv, p.sv_fast, kUnit)
                           : bf16x8_to_e4m3(x, p.sk, p.rsk, p.sk_fast, kUnit);
    uint8_t* ws = tensor ? p.ws_v : p.ws_k;
    // a token's workspace row holds units_per_token 8-byte outputs (hkv * 128 E4M3 bytes)
    reinterpret_cast<uint2*>(ws + row * (int64_t)p.units_per_token * 8)[uu - tok * p.units_per_token] = e;
  }
}

// ---------------------------------------------------------------------------
// extend attention
// ---------------------------------------------------------------------------

constexpr int kTileM = 128;          // query rows per CTA (TMEM lanes); a CTA pair takes 256
constexpr int kTileN = 128;          // keys per K/V tile
constexpr int kHalfN = kTileN / 2;   // keys of K, and head dims of V, that each CTA of the pair stages
constexpr int kSoftmaxWarps = 4;
constexpr int kLoadWarps = 4;
constexpr int kThreads = (kSoftmaxWarps + kLoadWarps + 1) * 32;  // + the MMA warp
constexpr int kMmaWarp = kSoftmaxWarps + kLoadWarps;
constexpr uint32_t kLBO = 128;   // next core matrix along K
constexpr uint32_t kSBO = 2048;  // next 8-row (N) group: 16 core matrices of 128 B
constexpr uint32_t kHalfBytes = kHalfN * kHeadDim * 2;  // a CTA's half of one f16 B tile, 16 KB
#ifndef NVFP4KV_EXTEND_STAGES
#define NVFP4KV_EXTEND_STAGES 6
#endif
constexpr int kStages = NVFP4KV_EXTEND_STAGES;  // K / V ring depth
constexpr uint32_t kOffK = 0, kOffV = kStages * kHalfBytes;
constexpr uint32_t kSmemBytes = 2 * kStages * kHalfBytes;  // 192 KB at 6 stages: one CTA per SM
// TMEM columns: S[0] 0-127, S[1] 128-255, O 256-383 (f32); Q 384-447 and
// P 448-511 (f16 pairs: the A operands of S = Q K^T and O += P V)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 256, kTmemQ = 384, kTmemP = 448;
constexpr float kLazy = 8.0f;  // the running max moves only when a row max exceeds it by this (base 2)
constexpr uint64_t kWaitNs = 1000000000ull;

struct ExtendParams {
  const uint16_t* q;
  const int64_t* cu_q;
  const uint8_t* ws_k;
  const uint8_t* ws_v;
  const int64_t* cu_prefix;
  const int32_t* prefix_lens;
  int32_t hq, hkv, group, log2_group;
  int32_t max_q_len;
  int64_t total_rows;
  float score_scale;  // softmax_scale * k_ws_scale * log2(e)
  float out_scale;    // v_ws_scale
  float* out;
  int32_t* status;
};

// byte offset of element (row, k) in a K-major f16 tile / (mn, k) in an MN-major one
__device__ __forceinline__ uint32_t kmajor_off(int row, int k) {
  return (uint32_t)(row >> 3) * kSBO + (uint32_t)(k >> 3) * kLBO + (uint32_t)(row & 7) * 16 + (uint32_t)(k & 7) * 2;
}
__device__ __forceinline__ uint32_t mnmajor_off(int mn, int k) {
  return (uint32_t)(mn >> 3) * kSBO + (uint32_t)(k >> 3) * kLBO + (uint32_t)(k & 7) * 16 + (uint32_t)(mn & 7) * 2;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, const uint4& v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// One arrival, released at cluster scope, on the mbarrier of cluster rank 0
// that sits at this shared-memory offset.
__device__ __forceinline__ void arrive_rank0(uint32_t bar) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(remote) : "r"(bar));
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote) : "memory");
}

// Every thread of both CTAs: arrive (release) and wait (acquire).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3; "
      "selp.u32 %0, 1, 0, p; }"
      : "=r"(done)
      : "r"(bar), "r"(parity), "r"(1000000u)
      : "memory");
  return done;
}

// Wait (acquire at cluster scope: the arrivals may come from the other CTA)
// until the phase of the given parity completes; false after about `limit_ns`.
__device__ __forceinline__ bool wait_cluster(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (try_wait_cluster(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

// The same for a whole warp, with one outcome for all its lanes.
__device__ __forceinline__ bool warp_wait_cluster(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (__all_sync(0xFFFFFFFFu, try_wait_cluster(bar, parity))) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (__all_sync(0xFFFFFFFFu, try_wait_cluster(bar, parity))) return true;
    if (__shfl_sync(0xFFFFFFFFu, global_timer_ns() - t0 > limit_ns ? 1 : 0, 0)) return false;
  }
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t f16x2_bits(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// 8 bf16 -> 8 f16 (round to nearest; exact for 2^-14 <= |x| <= 65504)
__device__ __forceinline__ uint4 bf16x8_to_f16x8(const uint4& x) {
  return make_uint4(f16x2_bits(bf16_to_f32(x.x & 0xFFFFu), bf16_to_f32(x.x >> 16)),
                    f16x2_bits(bf16_to_f32(x.y & 0xFFFFu), bf16_to_f32(x.y >> 16)),
                    f16x2_bits(bf16_to_f32(x.z & 0xFFFFu), bf16_to_f32(x.z >> 16)),
                    f16x2_bits(bf16_to_f32(x.w & 0xFFFFu), bf16_to_f32(x.w >> 16)));
}

// 8 E4M3 bytes (a uint2) -> 8 f16 (exact)
__device__ __forceinline__ uint4 e4m3x8_to_f16x8(uint32_t lo, uint32_t hi) {
  return make_uint4(e4m3x2_to_f16x2(lo & 0xFFFFu), e4m3x2_to_f16x2(lo >> 16), e4m3x2_to_f16x2(hi & 0xFFFFu),
                    e4m3x2_to_f16x2(hi >> 16));
}

struct Barriers {
  uint64_t q_full;
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t s_full[2];
  uint64_t p_full;
  uint64_t o_done;
  uint64_t drain;
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1) extend_attention_kernel(ExtendParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ Barriers bars;
  __shared__ uint32_t s_tmem;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();  // blockIdx.x & 1
  const int b = blockIdx.y, hk = blockIdx.z;
  const int tokens_per_tile = kTileM >> p.log2_group;
  // the pair takes m-tiles 2 mp (rank 0) and 2 mp + 1 (rank 1), the latest (longest) pairs first
  const int mp = (int)(gridDim.x >> 1) - 1 - (int)(blockIdx.x >> 1);
  const int tp = 2 * mp * tokens_per_tile;                  // the pair's first token
  const int t0 = tp + (int)rank * tokens_per_tile;          // this CTA's first token

  // the sequence: chunk length C, prefix P, first workspace row
  const int64_t q0 = __ldg(p.cu_q + b);
  int64_t C = __ldg(p.cu_q + b + 1) - q0;
  int64_t P = __ldg(p.prefix_lens + b);
  const int64_t row0 = __ldg(p.cu_prefix + b);
  if (C < 0 || C > p.max_q_len || P < 0) {
    if (threadIdx.x == 0 && blockIdx.x == 0) flag_error(p.status, NVFP4KV_DEVERR_LENGTH);
    C = C < 0 ? 0 : (C > p.max_q_len ? p.max_q_len : C);
    P = P < 0 ? 0 : P;
  }
  // no query in the pair: both CTAs leave before any set-up (the test is the same in both)
  if (tp >= C) return;
  const int64_t t_hi = (tp + 2 * tokens_per_tile < C ? tp + 2 * tokens_per_tile : C) - 1;
  const int64_t nkeys = P + t_hi + 1;  // keys 0 .. P + t_hi: the pair's last query sees them all
  const int ntiles = (int)((nkeys + kTileN - 1) / kTileN);

  const uint32_t sbase = smem_u32(smem);
  const uint32_t sK0 = sbase + kOffK, sV0 = sbase + kOffV;
  const uint32_t b_q = smem_u32(&bars.q_full), b_p = smem_u32(&bars.p_full), b_o = smem_u32(&bars.o_done);
  const uint32_t b_kvf0 = smem_u32(&bars.kv_full[0]), b_kve0 = smem_u32(&bars.kv_empty[0]);  // 8 bytes apart
  const uint32_t b_s[2] = {smem_u32(&bars.s_full[0]), smem_u32(&bars.s_full[1])};
  const uint32_t b_drain = smem_u32(&bars.drain);

  // Rank 0's q_full, kv_full and p_full take one arrival per loader or softmax
  // warp of both CTAs; s_full, o_done and kv_empty in both CTAs are arrived on
  // by rank 0's MMA commits, multicast to the pair.
  if (threadIdx.x == 0) {
    mbar_init(b_q, 2 * kLoadWarps);
    for (int st = 0; st < kStages; ++st) {
      mbar_init(b_kvf0 + 8 * st, 2 * kLoadWarps);
      mbar_init(b_kve0 + 8 * st, 1);
    }
    mbar_init(b_s[0], 1);
    mbar_init(b_s[1], 1);
    mbar_init(b_p, 2 * kSoftmaxWarps);
    mbar_init(b_o, 1);
    mbar_init(b_drain, 1);
    fence_mbar_init();
  }
  if (warp == 0) tc::tmem_alloc(smem_u32(&s_tmem), kTmemCols);
  // both CTAs' barriers and TMEM exist before either CTA signals the other
  tc::fence_before_sync();
  cluster_sync();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;
  const int G = p.group;

  if (warp >= kSoftmaxWarps && warp < kMmaWarp) {
    // ------------------------------------------------------------ loaders
    const int l = threadIdx.x - kSoftmaxWarps * 32;  // 0 .. 127
    // This CTA's half of each tile: K rows (keys) 64 rank .. 64 rank + 63 and V
    // columns (head dims) 64 rank .. 64 rank + 63 of all 128 keys.  Lane parts:
    //   K: key 16 lw + 8 g + (lane & 7) of the half (g < 2), bytes 16 part + 64 h (h < 2)
    //   V: key 32 lw + 8 g + (lane & 7) (g < 4), bytes 64 rank + 16 part
    // A tile's 16-byte loads are issued one step ahead (into registers) so that
    // their latency overlaps the wait for the stage they go to.
    const int lw = warp - kSoftmaxWarps;
    const int part = lane >> 3;
    uint4 xk[2][2], xv[4];
    auto load_tile = [&](int i) {
      const int64_t base = (int64_t)i * kTileN;
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        const int64_t j = base + kHalfN * (int)rank + lw * 16 + g * 8 + (lane & 7);
        const int64_t row = row0 + j;
        bool live = j < nkeys;
        if (live && (row < 0 || row >= p.total_rows)) {
          flag_error(p.status, NVFP4KV_DEVERR_ROW);
          live = false;
        }
        const int64_t off = (row * p.hkv + hk) * kHeadDim + part * 16;
#pragma unroll
        for (int h = 0; h < 2; ++h)
          xk[g][h] = live ? __ldg(reinterpret_cast<const uint4*>(p.ws_k + off + h * 64)) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const int64_t j = base + lw * 32 + g * 8 + (lane & 7);
        const int64_t row = row0 + j;
        bool live = j < nkeys;
        if (live && (row < 0 || row >= p.total_rows)) {
          flag_error(p.status, NVFP4KV_DEVERR_ROW);
          live = false;
        }
        const int64_t off = (row * p.hkv + hk) * kHeadDim + kHalfN * (int)rank + part * 16;
        xv[g] = live ? __ldg(reinterpret_cast<const uint4*>(p.ws_v + off)) : make_uint4(0, 0, 0, 0);
      }
    };
    load_tile(0);
    {
      // Q: thread l converts query row l (token t0 + l / G, head hk * G + l % G)
      // into TMEM lane l (this warp's lane quarter), two d values per column
      const int64_t t = t0 + (l >> p.log2_group);
      const bool live = t < C;
      const uint4* src =
          reinterpret_cast<const uint4*>(p.q + ((q0 + (live ? t : 0)) * p.hq + hk * G + (l & (G - 1))) * kHeadDim);
      const uint32_t tq = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + kTmemQ;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t w[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 h = bf16x8_to_f16x8(live ? __ldg(src + 8 * half + c) : make_uint4(0, 0, 0, 0));
          w[4 * c] = h.x;
          w[4 * c + 1] = h.y;
          w[4 * c + 2] = h.z;
          w[4 * c + 3] = h.w;
        }
        tc::tmem_st32(tq + 32 * half, w);
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) arrive_rank0(b_q);
    }
    bool ok = true;
    for (int i = 0; i < ntiles; ++i) {
      const int s = i % kStages;
      if (i >= kStages && !warp_wait_cluster(b_kve0 + 8 * s, ((i / kStages) - 1) & 1, kWaitNs)) {
        ok = false;
        break;
      }
      const uint32_t sK = sK0 + s * kHalfBytes, sV = sV0 + s * kHalfBytes;
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        const int key = lw * 16 + g * 8 + (lane & 7);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int d0 = h * 64 + part * 16;
          st_shared_v4(sK + kmajor_off(key, d0), e4m3x8_to_f16x8(xk[g][h].x, xk[g][h].y));
          st_shared_v4(sK + kmajor_off(key, d0 + 8), e4m3x8_to_f16x8(xk[g][h].z, xk[g][h].w));
        }
      }
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const int key = lw * 32 + g * 8 + (lane & 7);
        st_shared_v4(sV + mnmajor_off(part * 16, key), e4m3x8_to_f16x8(xv[g].x, xv[g].y));
        st_shared_v4(sV + mnmajor_off(part * 16 + 8, key), e4m3x8_to_f16x8(xv[g].z, xv[g].w));
      }
      tc::fence_smem_to_async();
      __syncwarp();
      if (lane == 0) arrive_rank0(b_kvf0 + 8 * s);
      if (i + 1 < ntiles) load_tile(i + 1);
    }
    if (!ok) flag_error(p.status, NVFP4KV_DEVERR_TIMEOUT);
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issue (rank 0)
    if (rank == 0 && lane == 0) {
      constexpr uint32_t id_qk = tc::idesc_f16_f32(2 * kTileM, kTileN, false, false);
      constexpr uint32_t id_pv = tc::idesc_f16_f32(2 * kTileM, kHeadDim, false, true);
      bool ok = wait_cluster(b_q, 0, kWaitNs);
      for (int i = 0; i <= ntiles && ok; ++i) {
        if (i < ntiles) {
          const int s = i % kStages;
          if (!wait_cluster(b_kvf0 + 8 * s, (i / kStages) & 1, kWaitNs)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t sK = sK0 + s * kHalfBytes;
#pragma unroll
          for (int kk = 0; kk < kHeadDim / 16; ++kk)
            tc::mma_f16_tmem_a(tmem + (i & 1) * kTileN, tmem + kTmemQ + kk * 8, tc::smem_desc(sK + kk * 256, kLBO, kSBO),
                               id_qk, kk > 0);
          tc::commit_multicast(b_s[i & 1], 3);
        }
        if (i >= 1) {
          const int pi = i - 1;  // P V of the previous tile
          if (!wait_cluster(b_p, pi & 1, kWaitNs)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t sV = sV0 + (pi % kStages) * kHalfBytes;
#pragma unroll
          for (int kk = 0; kk < kTileN / 16; ++kk)
            tc::mma_f16_tmem_a(tmem + kTmemO, tmem + kTmemP + kk * 8, tc::smem_desc(sV + kk * 256, kLBO, kSBO), id_pv,
                               (pi > 0 || kk > 0) ? 1u : 0u);
          tc::commit_multicast(b_o, 3);
          // the loaders of both CTAs wait for this stage
          if (pi + kStages < ntiles) tc::commit_multicast(b_kve0 + 8 * (pi % kStages), 3);
        }
      }
      if (!ok) flag_error(p.status, NVFP4KV_DEVERR_TIMEOUT);
      // nothing this thread issued may still be running when either CTA frees its TMEM
      tc::commit(b_drain);
      wait_cluster(b_drain, 0, kWaitNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax rows
    const int r = threadIdx.x;  // TMEM lane / query row
    const int64_t t = t0 + (r >> p.log2_group);
    const bool live = t < C;
    const int64_t kmax = P + t;  // last visible key
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    float m = -INFINITY, l = 0.0f;
    bool ok = true;
    for (int i = 0; i < ntiles; ++i) {
      if (!warp_wait_cluster(b_s[i & 1], (i >> 1) & 1, kWaitNs)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      float x[kTileN];
#pragma unroll
      for (int c4 = 0; c4 < kTileN / 32; ++c4) {
        uint32_t v[32];
        tc::tmem_ld32(tmem + lane_base + (i & 1) * kTileN + c4 * 32, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) x[c4 * 32 + j] = __uint_as_float(v[j]);
      }
      // keys c <= lim of this tile are visible to the row (all of them away from
      // the causal edge, none for a row past the chunk)
      const int64_t lim64 = live ? kmax - (int64_t)i * kTileN : -1;
      const int lim = lim64 >= kTileN - 1 ? kTileN - 1 : (int)(lim64 < -1 ? -1 : lim64);
      float mr[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if (lim == kTileN - 1) {
#pragma unroll
        for (int c = 0; c < kTileN; ++c) mr[c & 3] = fmaxf(mr[c & 3], x[c]);
      } else {
#pragma unroll
        for (int c = 0; c < kTileN; ++c) {
          if (c > lim) x[c] = -INFINITY;
          mr[c & 3] = fmaxf(mr[c & 3], x[c]);
        }
      }
      // the row max in base-2 units (the scale is positive, so it commutes with max)
      const float mx = fmaxf(fmaxf(mr[0], mr[1]), fmaxf(mr[2], mr[3])) * p.score_scale;
      float alpha = 1.0f;
      const bool grow = mx > m + kLazy;  // false for rows with nothing visible (mx = -inf)
      if (grow) {
        alpha = ex2(m - mx);  // 0 on the first visible tile (m = -inf)
        m = mx;
      }
      // p = 2^(s * scale - m); masked scores are -inf and give 0, and so does
      // every score of a row past the chunk (offset -inf)
      const float off = live ? -m : -INFINITY;
      uint32_t ph[kTileN / 2];
      float ls[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int c = 0; c < kTileN; c += 2) {
        const float p0 = ex2(fmaf(x[c], p.score_scale, off)), p1 = ex2(fmaf(x[c + 1], p.score_scale, off));
        ph[c / 2] = f16x2_bits(p0, p1);
        ls[(c >> 1) & 3] += p0 + p1;
      }
      const float lt = (ls[0] + ls[1]) + (ls[2] + ls[3]);
      if (i >= 1) {
        // the previous P V must be done before P is overwritten and O rescaled
        if (!warp_wait_cluster(b_o, (i - 1) & 1, kWaitNs)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        if (__any_sync(0xFFFFFFFFu, grow)) {
          const float a = grow ? alpha : 1.0f;
#pragma unroll
          for (int c4 = 0; c4 < kHeadDim / 32; ++c4) {
            uint32_t v[32];
            const uint32_t ta = tmem + lane_base + kTmemO + c4 * 32;
            tc::tmem_ld32(ta, v);
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * a);
            tc::tmem_st32(ta, v);
          }
        }
      }
      l = l * alpha + lt;
      // P into TMEM: the A operand of the next P V (two keys per column)
      tc::tmem_st32(tmem + lane_base + kTmemP, *reinterpret_cast<const uint32_t(*)[32]>(&ph[0]));
      tc::tmem_st32(tmem + lane_base + kTmemP + 32, *reinterpret_cast<const uint32_t(*)[32]>(&ph[32]));
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) arrive_rank0(b_p);
    }
    if (ok && warp_wait_cluster(b_o, (ntiles - 1) & 1, kWaitNs)) {
      tc::fence_after_sync();
      const float inv = live && l > 0.0f ? p.out_scale / l : 0.0f;
      float4* dst = reinterpret_cast<float4*>(
          p.out + ((q0 + (live ? t : 0)) * p.hq + hk * G + (r & (G - 1))) * kHeadDim);
#pragma unroll
      for (int c4 = 0; c4 < kHeadDim / 32; ++c4) {
        uint32_t v[32];
        tc::tmem_ld32(tmem + lane_base + kTmemO + c4 * 32, v);
        if (live) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            dst[c4 * 8 + j] = make_float4(__uint_as_float(v[4 * j]) * inv, __uint_as_float(v[4 * j + 1]) * inv,
                                          __uint_as_float(v[4 * j + 2]) * inv, __uint_as_float(v[4 * j + 3]) * inv);
        }
      }
    } else {
      flag_error(p.status, NVFP4KV_DEVERR_TIMEOUT);
    }
  }
  // Both CTAs are done with the pair's TMEM and barriers (rank 0's MMAs
  // drained, every signal to the other CTA sent) before either frees or leaves.
  tc::fence_before_sync();
  cluster_sync();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_chunk_to_ws(const uint16_t* k, const uint16_t* v, const int64_t* ws_rows, int64_t num_tokens,
                               int32_t num_kv_heads, int64_t total_rows, float k_ws_scale, float v_ws_scale,
                               uint8_t* ws_k, uint8_t* ws_v, int32_t* device_status, int num_sms,
                               cudaStream_t stream) {
  ChunkParams p;
  p.k = k;
  p.v = v;
  p.rows = ws_rows;
  p.units_per_token = num_kv_heads * (kHeadDim / 8);
  p.units = num_tokens * p.units_per_token;
  p.total_rows = total_rows;
  p.sk = k_ws_scale;
  p.sv = v_ws_scale;
  p.rsk = 1.0f / k_ws_scale;  // host IEEE division: RN(1 / s_ws)
  p.rsv = 1.0f / v_ws_scale;
  p.sk_fast = k_ws_scale >= 0x1p-100f && k_ws_scale <= 0x1p+100f;
  p.sv_fast = v_ws_scale >= 0x1p-100f && v_ws_scale <= 0x1p+100f;
  p.ws_k = ws_k;
  p.ws_v = ws_v;
  p.status = device_status;
  int64_t blocks = (2 * p.units + kChunkThreads - 1) / kChunkThreads;
  const int64_t max_blocks = (int64_t)num_sms * (2048 / kChunkThreads);
  if (blocks > max_blocks) blocks = max_blocks;
  if (blocks < 1) blocks = 1;
  if (k_ws_scale == 1.0f && v_ws_scale == 1.0f)
    chunk_to_ws_kernel<true><<<(unsigned)blocks, kChunkThreads, 0, stream>>>(p);
  else
    chunk_to_ws_kernel<false><<<(unsigned)blocks, kChunkThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_extend_attention(const uint16_t* q, const int64_t* cu_q, int32_t max_q_len, const uint8_t* ws_k,
                                    const uint8_t* ws_v, const int64_t* cu_prefix, const int32_t* prefix_lens,
                                    int32_t batch, int64_t total_rows, int32_t num_q_heads, int32_t num_kv_heads,
                                    float k_ws_scale, float v_ws_scale, float softmax_scale, float* out,
                                    int32_t* device_status, cudaStream_t stream) {
  ExtendParams p;
  p.q = q;
  p.cu_q = cu_q;
  p.ws_k = ws_k;
  p.ws_v = ws_v;
  p.cu_prefix = cu_prefix;
  p.prefix_lens = prefix_lens;
  p.hq = num_q_heads;
  p.hkv = num_kv_heads;
  p.group = num_q_heads / num_kv_heads;
  p.log2_group = 0;
  while ((1 << p.log2_group) < p.group) ++p.log2_group;
  p.max_q_len = max_q_len;
  p.total_rows = total_rows;
  p.score_scale = (float)((double)softmax_scale * (double)k_ws_scale * 1.4426950408889634);
  p.out_scale = v_ws_scale;
  p.out = out;
  p.status = device_status;
  // the shared-memory limit is an attribute of the function on each device
  static PerDeviceOnce attr_once;
  const cudaError_t attr = attr_once.run([] {
    return cudaFuncSetAttribute(extend_attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  });
  if (attr != cudaSuccess) return attr;
  // CTA pairs (clusters of two along x): an even number of m-tiles
  const int64_t tiles = ((int64_t)max_q_len * p.group + kTileM - 1) / kTileM;
  const dim3 grid((unsigned)((tiles + 1) / 2 * 2), (unsigned)batch, (unsigned)num_kv_heads);
  extend_attention_kernel<<<grid, kThreads, kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace nvfp4kv
