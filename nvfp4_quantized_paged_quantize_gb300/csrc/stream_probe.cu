// stream_probe.cu -- the memory stream of the decode with no attention math:
// a measurement aid that reads every cached page-head of a decode batch once,
// as the decode does, so that the time of the decode can be set against the
// time the same bytes take to stream on their own ("nvfp4-kv-cache-memory-
// wall", section 3, item 3: decode is bound by the KV read).
//
// Mode NVFP4KV_PROBE_DECODE_PATTERN copies exactly what decode_kernel copies,
// with its grid, its split of the (sequence, KV head, page) items over warps,
// its per-warp rings of 2304-byte stages filled by 16-byte cp.async pieces and
// its mbarrier waits; each page then costs one shared-memory load instead of
// the dequantisation and the two MMAs.  Mode NVFP4KV_PROBE_WHOLE_PAGES streams
// the same pages as whole pages (every KV head of a page, one contiguous
// run) with one bulk copy (TMA) each, one warp per CTA, two CTAs per SM: the
// fastest way the layout allows.  Both split the work statically and evenly.
// Every wait is bounded; a wait that gives up sets NVFP4KV_DEVERR_TIMEOUT.
#include <cstdint>

#include "nvfp4kv_device.cuh"
#include "nvfp4kv_launch.h"

namespace nvfp4kv {
namespace {

constexpr int kNW = 4;              // decode pattern: warps per CTA, as the decode
constexpr int kCtasPerSm = 3;       // decode pattern: CTAs per SM, as the decode
constexpr int kStages = 4;          // decode pattern: ring stages per warp, as the decode
constexpr int kPageStages = 6;      // whole pages: ring stages per CTA
constexpr int kPageCtasPerSm = 2;   // whole pages: CTAs (one warp each) per SM
constexpr int kMaxPageBytes = 16 * kPageHeadBytes;  // whole pages: up to 16 KV heads per stage

struct ProbeParams {
  const uint8_t* pages;
  int32_t num_pages;
  int32_t hkv;
  const int32_t* page_table;
  int32_t max_pages;
  const int32_t* seq_lens;
  int32_t batch;
  uint32_t* sink;
  int32_t* status;
};

__device__ __forceinline__ int clamp_len(const ProbeParams& p, int b) {
  int L = __ldg(p.seq_lens + b);
  const int lmax = p.max_pages * kPage;
  if (L < 0 || L > lmax) {
    flag_error(p.status, NVFP4KV_DEVERR_LENGTH);
    L = L < 0 ? 0 : lmax;
  }
  return L;
}

__device__ __forceinline__ long long range_start(long long c, long long W, long long N) {
  const long long q = W / N, rem = W % N;
  return c * q + (c < rem ? c : rem);
}

// Total pages of the batch (every CTA computes it) and the sequence holding
// unit r0 of a list whose sequence b spans `per_page * pages(b)` units.
__device__ void locate(const ProbeParams& p, long long per_page, long long r0, long long* W, int* b0, int* cu0) {
  __shared__ long long s_total;
  __shared__ int s_b, s_cu;
  if (threadIdx.x == 0) {
    long long cu = 0;
    int fb = 0, fcu = 0;
    bool found = false;
    for (int b = 0; b < p.batch; ++b) {
      const int np = (clamp_len(p, b) + kPage - 1) / kPage;
      if (!found && np > 0 && r0 < (cu + np) * per_page) {
        fb = b;
        fcu = (int)cu;
        found = true;
      }
      cu += np;
    }
    s_total = cu;
    s_b = fb;
    s_cu = fcu;
  }
  __syncthreads();
  *W = s_total;
  *b0 = s_b;
  *cu0 = s_cu;
}

// The page id of unit r (sequence-major), walking forward from (b, cu); units
// of a page are `per_page` consecutive heads (decode pattern) or one (pages).
__device__ __forceinline__ int unit_page(const ProbeParams& p, long long r, long long per_page, int& b, int& cu,
                                         int& np, int* head) {
  while (r >= (long long)(cu + np) * per_page) {
    cu += np;
    ++b;
    np = (clamp_len(p, b) + kPage - 1) / kPage;
  }
  const long long local = r - (long long)cu * per_page;
  const int h = (int)(local / np), pg = (int)(local - (long long)h * np);
  *head = h;
  const int id = __ldg(p.page_table + (long long)b * p.max_pages + pg);
  if (id < 0 || id >= p.num_pages) {
    flag_error(p.status, NVFP4KV_DEVERR_PAGE);
    return -1;
  }
  return id;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// The decode's pattern: warp ranges of page-heads, 2304-byte stages by cp.async.
__global__ void __launch_bounds__(kNW * 32) probe_decode_pattern(const ProbeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  long long W;
  int b, cu;
  const long long N = gridDim.x;
  // the CTA range needs W first: locate with r0 = 0, then again with the real r0
  locate(p, p.hkv, 0, &W, &b, &cu);
  W *= p.hkv;
  const long long r0 = range_start(blockIdx.x, W, N), r1 = range_start(blockIdx.x + 1, W, N);
  const long long wr0 = r0 + (r1 - r0) * warp / kNW, wr1 = r0 + (r1 - r0) * (warp + 1) / kNW;
  __syncthreads();
  long long Wd;
  locate(p, p.hkv, wr0 < W ? r0 : 0, &Wd, &b, &cu);
  const int n = (int)(wr1 - wr0);
  uint8_t* ring = smem + warp * kStages * kPageHeadBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kNW * kStages * kPageHeadBytes) + warp * kStages;
  if (n <= 0) return;
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(bars + s), 32);
    fence_mbar_init();
  }
  __syncwarp();
  // walk from the CTA's first unit to the warp's
  int np = (clamp_len(p, b) + kPage - 1) / kPage;
  int head = 0;
  {
    int bb = b, cc = cu, nn = np;
    if (wr0 > r0) unit_page(p, wr0, p.hkv, bb, cc, nn, &head);
    b = bb;
    cu = cc;
    np = nn;
  }
  uint32_t acc = 0;
  auto issue = [&](int i) {
    const int id = unit_page(p, wr0 + i, p.hkv, b, cu, np, &head);
    const uint32_t st = smem_u32(ring + (i % kStages) * kPageHeadBytes);
    if (id >= 0) {
      const uint8_t* src = p.pages + ((size_t)id * p.hkv + head) * kPageHeadBytes;
      for (int c = lane; c < kPageHeadBytes / 16; c += 32) cp_async16(st + 16 * c, src + 16 * c);
    }
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bars + i % kStages))
                 : "memory");
  };
  const int pre = n < kStages ? n : kStages;
  for (int i = 0; i < pre; ++i) issue(i);
  int issued = pre;
  bool ok = true;
  for (int i = 0; i < n; ++i) {
    const bool done = mbar_wait(smem_u32(bars + i % kStages), (uint32_t)((i / kStages) & 1));
    if (!__all_sync(0xFFFFFFFFu, done)) {
      ok = false;
      if (lane == 0) flag_error(p.status, kDevErrTimeout);
      break;
    }
    acc ^= *reinterpret_cast<const uint32_t*>(ring + (i % kStages) * kPageHeadBytes + 4 * lane);
    __syncwarp();
    if (i + kStages < n) {
      issue(i + kStages);
      issued = i + kStages + 1;
    }
  }
  if (!ok) {
    for (int j = issued - kStages; j < issued; ++j)
      if (j >= 0) mbar_wait(smem_u32(bars + j % kStages), (uint32_t)((j / kStages) & 1));
  }
  if (acc != 0) atomicXor(p.sink, acc);
}

// Whole pages: one warp per CTA streams its range of pages with bulk copies.
__global__ void __launch_bounds__(32) probe_whole_pages(const ProbeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[kPageStages];
  const int lane = threadIdx.x;
  long long W;
  int b, cu;
  const long long N = gridDim.x;
  locate(p, 1, 0, &W, &b, &cu);
  const long long r0 = range_start(blockIdx.x, W, N), r1 = range_start(blockIdx.x + 1, W, N);
  const int n = (int)(r1 - r0);
  if (n <= 0) return;
  long long Wd;
  locate(p, 1, r0, &Wd, &b, &cu);
  const uint32_t bytes = (uint32_t)p.hkv * kPageHeadBytes;
  if (lane == 0) {
    for (int s = 0; s < kPageStages; ++s) mbar_init(smem_u32(bars + s), 1);
    fence_mbar_init();
  }
  __syncwarp();
  int np = (clamp_len(p, b) + kPage - 1) / kPage;
  int head = 0;
  uint32_t acc = 0;
  auto issue = [&](int i) {
    const int id = unit_page(p, r0 + i, 1, b, cu, np, &head);  // lane-uniform
    if (lane != 0) return;
    const uint32_t bar = smem_u32(bars + i % kPageStages);
    if (id >= 0) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
      asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                   ::"r"(smem_u32(smem + (size_t)(i % kPageStages) * bytes)),
                   "l"(p.pages + (size_t)id * bytes), "r"(bytes), "r"(bar)
                   : "memory");
    } else {
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
    }
  };
  const int pre = n < kPageStages ? n : kPageStages;
  for (int i = 0; i < pre; ++i) issue(i);
  int issued = pre;
  bool ok = true;
  for (int i = 0; i < n; ++i) {
    const bool done = mbar_wait(smem_u32(bars + i % kPageStages), (uint32_t)((i / kPageStages) & 1));
    if (!__all_sync(0xFFFFFFFFu, done)) {
      ok = false;
      if (lane == 0) flag_error(p.status, kDevErrTimeout);
      break;
    }
    acc ^= *reinterpret_cast<const uint32_t*>(smem + (size_t)(i % kPageStages) * bytes + 4 * lane);
    __syncwarp();
    if (i + kPageStages < n) {
      issue(i + kPageStages);
      issued = i + kPageStages + 1;
    }
  }
  if (!ok) {
    for (int j = issued - kPageStages; j < issued; ++j)
      if (j >= 0) mbar_wait(smem_u32(bars + j % kPageStages), (uint32_t)((j / kPageStages) & 1));
  }
  if (acc != 0) atomicXor(p.sink, acc);
}

}  // namespace

cudaError_t launch_stream_probe(const nvfp4kv_cache& c, const int32_t* page_table, int32_t max_pages,
                                const int32_t* seq_lens, int32_t batch, int mode, uint32_t* sink,
                                int32_t* device_status, int num_sms, cudaStream_t stream) {
  ProbeParams p;
  p.pages = c.pages;
  p.num_pages = (int32_t)c.num_pages;
  p.hkv = c.num_kv_heads;
  p.page_table = page_table;
  p.max_pages = max_pages;
  p.seq_lens = seq_lens;
  p.batch = batch;
  p.sink = sink;
  p.status = device_status;
  if (mode == NVFP4KV_PROBE_DECODE_PATTERN) {
    const int smem = kNW * kStages * (kPageHeadBytes + 8);
    static PerDeviceOnce once;
    const cudaError_t e = once.run([smem] {
      return cudaFuncSetAttribute(probe_decode_pattern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (e != cudaSuccess) return e;
    probe_decode_pattern<<<num_sms * kCtasPerSm, kNW * 32, smem, stream>>>(p);
  } else {
    const int smem = kPageStages * c.num_kv_heads * kPageHeadBytes;
    static PerDeviceOnce once;
    const cudaError_t e = once.run([] {
      return cudaFuncSetAttribute(probe_whole_pages, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  kPageStages * kMaxPageBytes);
    });
    if (e != cudaSuccess) return e;
    probe_whole_pages<<<num_sms * kPageCtasPerSm, 32, smem, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace nvfp4kv
