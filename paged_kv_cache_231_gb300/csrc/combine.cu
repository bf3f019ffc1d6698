// Log-sum-exp combine of (o, m, l) partials: the AttendSplitKMerge pass of
// "com.microsoft.PagedAttention manifest.json" and the merge of the block-sparse
// partials of "alice-llm sparse_attention_forward.wgsl" (partial layout block).
//
// One warp per output row; each lane owns head_dim / 32 consecutive elements, so a
// partial row is read as one coalesced 512-byte (D = 128) transaction. Pass 1 finds
// the max m over non-empty partials (l > 0); pass 2 accumulates w = exp(m - M) with
// w*l into L and w*o into the row, 32 partials at a time so that the o rows of a chunk
// are all in flight together; out = row / L, lse = M + ln L.
#include <math.h>

#include <atomic>

#include "device_common.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr int kCombineWarps = 4;

template <int D, bool PAGED, bool OUT_F16>
__device__ __forceinline__ void combine_row(const CombineParams& p, int64_t row, int lane) {
  constexpr int V = D / 32;  // elements per lane
  int64_t g0, g1, out_row;
  int64_t lanes = p.lanes, c = 0;
  if (PAGED) {
    const int64_t nrow = (int64_t)p.slot_count[0] * p.Hq;
    if (row >= nrow) return;
    const int64_t slot = row / p.Hq;
    const int hq = (int)(row % p.Hq);
    g0 = row * p.uniform;
    g1 = g0 + p.slot_splits[slot];
    out_row = (int64_t)p.slot_token[slot] * p.Hq + hq;
    lanes = 1;
  } else {
    if (row >= p.num_segments * p.lanes) return;
    const int64_t seg = row / p.lanes;
    c = row % p.lanes;
    if (p.seg_off) {
      g0 = p.seg_off[seg];
      g1 = p.seg_off[seg + 1];
    } else {
      g0 = seg * p.uniform;
      g1 = g0 + p.uniform;
    }
    out_row = row;
  }
  float M = -INFINITY;
  for (int64_t e = g0 + lane; e < g1; e += 32) {
    const int64_t pr = e * lanes + c;
    if (p.l[pr] > 0.f) M = fmaxf(M, p.m[pr]);
  }
  M = warp_max(M);
  float acc[V];
#pragma unroll
  for (int v = 0; v < V; ++v) acc[v] = 0.f;
  float Lpart = 0.f;
  if (M != -INFINITY) {
    // 32 partials at a time: lane k computes the weight of partial base + k, then every
    // o row of the chunk is loaded without waiting on another load (an empty partial's
    // load is pointed at a non-empty row of the chunk and weighted 0, so its o is never
    // used)
    for (int64_t base = g0; base < g1; base += 32) {
      const int64_t e = base + lane;
      float w = 0.f;
      if (e < g1) {
        const int64_t pr = e * lanes + c;
        const float lv = p.l[pr];
        if (lv > 0.f) {
          w = ex2((p.m[pr] - M) * kLog2e);
          Lpart += w * lv;
        }
      }
      const uint32_t live = __ballot_sync(0xffffffffu, w > 0.f);
      if (!live) continue;
      const int64_t fallback = (base + (__ffs(live) - 1)) * lanes + c;
      const int n = g1 - base < 32 ? (int)(g1 - base) : 32;
#pragma unroll 8
      for (int k = 0; k < n; ++k) {
        const float wk = __shfl_sync(0xffffffffu, w, k);
        const int64_t pr = wk > 0.f ? (base + k) * lanes + c : fallback;
        const float* orow = p.o + pr * D + lane * V;
        if constexpr (V == 4) {
          const float4 x = __ldg(reinterpret_cast<const float4*>(orow));
          acc[0] += wk * x.x;
          acc[1] += wk * x.y;
          acc[2] += wk * x.z;
          acc[3] += wk * x.w;
        } else {
#pragma unroll
          for (int v = 0; v < V; ++v) acc[v] += wk * __ldg(orow + v);
        }
      }
    }
  }
  const float L = warp_sum(Lpart);
  const float inv = L > 0.f ? 1.f / L : 0.f;
  if (OUT_F16) {
    __half* dst = reinterpret_cast<__half*>(p.out) + out_row * D + lane * V;
#pragma unroll
    for (int v = 0; v < V; v += 2)
      *reinterpret_cast<__half2*>(dst + v) = __floats2half2_rn(acc[v] * inv, acc[v + 1] * inv);
  } else {
    float* dst = reinterpret_cast<float*>(p.out) + out_row * D + lane * V;
#pragma unroll
    for (int v = 0; v < V; ++v) dst[v] = acc[v] * inv;
  }
  if (p.lse && lane == 0) p.lse[out_row] = L > 0.f ? M + logf(L) : -INFINITY;
}

// Persistent: each warp takes rows warp, warp + W, ... (W = the grid's warps), so the
// whole merge runs in one wave of resident blocks instead of one short block per 4 rows.
template <int D, bool PAGED, bool OUT_F16>
__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(CombineParams p,
                                                                      int64_t rows) {
  const int lane = threadIdx.x & 31;
  const int64_t W = (int64_t)gridDim.x * kCombineWarps;
  for (int64_t row = (int64_t)blockIdx.x * kCombineWarps + (threadIdx.x >> 5); row < rows;
       row += W)
    combine_row<D, PAGED, OUT_F16>(p, row, lane);
}

// resident blocks of the combine kernel per SM (2048 threads / 128)
constexpr int kCombineBlocksPerSm = 16;

template <int D>
cudaError_t launch_d(const CombineParams& p, int64_t rows, cudaStream_t s) {
  static std::atomic<int> sms_cache{0};
  int sms = sms_cache.load(std::memory_order_relaxed);
  if (sms <= 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0)
      sms = 152;
    sms_cache.store(sms, std::memory_order_relaxed);
  }
  const int64_t need = (rows + kCombineWarps - 1) / kCombineWarps;
  const int64_t cap = (int64_t)sms * kCombineBlocksPerSm;
  const unsigned grid = (unsigned)(need < cap ? need : cap);
  if (grid == 0) return cudaSuccess;
  const bool paged = p.slot_token != nullptr;
  ProfScope ps("combine", s);
  if (paged)
    combine_kernel<D, true, true><<<grid, kCombineWarps * 32, 0, s>>>(p, rows);
  else if (p.out_f16)
    combine_kernel<D, false, true><<<grid, kCombineWarps * 32, 0, s>>>(p, rows);
  else
    combine_kernel<D, false, false><<<grid, kCombineWarps * 32, 0, s>>>(p, rows);
  return cudaGetLastError();
}

}  // namespace

// rows: number of output rows to cover (an upper bound in the paged mode).
cudaError_t launch_combine(const CombineParams& p, cudaStream_t s) {
  const int64_t rows = p.slot_token ? p.num_segments * p.Hq : p.num_segments * p.lanes;
  switch (p.D) {
    case 64:
      return launch_d<64>(p, rows, s);
    case 128:
      return launch_d<128>(p, rows, s);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
