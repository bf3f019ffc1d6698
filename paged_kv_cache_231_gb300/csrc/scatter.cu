// KV writes into the caches.
//
// paged_scatter_kernel: the ScatterKV pass of "com.microsoft.PagedAttention
//   manifest.json" - each new token's K and V rows go to the paged cache
//   [num_blocks, block_size, kv_heads, head] at the row slot_mapping names, or at the
//   block-table row of the token's absolute position past + t. Optionally the key is
//   rotated first at that position (rotation rule of the SparseAttention append page).
// append_kernel: the KV-append main of "com.microsoft.SparseAttention
//   sparse-kv-append.wgsl.jinja" - writes new rows into a [batch, kv_heads,
//   max_cache_seq, head] cache at position history(b) + t, rotating K with the
//   sparse_rotary rule; optionally the query heads are rotated at the same position
//   into a separate output (the page rotates keys only).
//
// Row path (head size <= 128, chunk-aligned rotation pairs): half a warp moves a (token,
// kv head) row pair, rotation partners exchanged between lanes. Otherwise one thread moves
// one 16-byte chunk (8 halves) of a K row and the matching V chunk; consecutive threads
// take consecutive chunks of a row, so loads and stores coalesce.
// The page's one-invocation-per-component dispatch and its 2-D dispatch folding
// (a WebGPU grid limit) are not needed: CUDA's grid is 1-D up to 2^31 - 1 blocks.
#include "device_common.cuh"
#include "internal.h"
#include "scatter_dev.cuh"

namespace pkv {
namespace {

constexpr int kScatterThreads = 256;

__global__ void __launch_bounds__(kScatterThreads) paged_scatter_kernel(ScatterParams p) {
  paged_scatter_thread<false>(p, (int64_t)blockIdx.x * kScatterThreads + threadIdx.x);
}

__global__ void __launch_bounds__(kScatterThreads) paged_scatter_rows_kernel(ScatterParams p) {
  const int64_t row = ((int64_t)blockIdx.x * kScatterThreads + threadIdx.x) >> 4;
  paged_scatter_row<false>(p, row, threadIdx.x & 31);
}

// Row path of the append: half-warp `row` of the (batch, kv head, new token) grid; with kQ
// also the query heads (the kernels without kQ carry none of that code).
template <bool kQ>
__global__ void __launch_bounds__(kScatterThreads) append_rows_kernel(AppendParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t row = ((int64_t)blockIdx.x * kScatterThreads + threadIdx.x) >> 4;
  if (row >= (int64_t)p.B * p.Hkv * p.S) return;
  const int t = (int)(row % p.S);
  const int64_t r = row / p.S;
  const int h = (int)(r % p.Hkv);
  const int b = (int)(r / p.Hkv);
  // history length: prompt mode when the scalar total equals the new-token count
  const uint32_t total0 = (uint32_t)p.total_seq[0];
  const uint32_t S = (uint32_t)p.S;
  uint32_t past = 0;
  if (total0 != S) {
    const uint32_t tb = (uint32_t)p.key_totals[b];
    past = tb >= S ? tb - S : 0u;
  }
  const int64_t pos = (int64_t)past + t;
  if constexpr (kQ) {   // the G query heads of kv head h (copied unrotated past the table)
    const int G = p.Hq / p.Hkv;
    const int64_t qr = (int64_t)b * p.S + t;
    rotate_query_rows(p.q_src + qr * p.q_stride + (int64_t)h * G * p.D,
                      p.q_dst + (qr * p.Hq + (int64_t)h * G) * p.D, G, p.D, pos, p.cos, p.sin,
                      pos < p.rotary_positions ? p.rotary_dim : 0, p.interleaved, lane);
  }
  if (pos >= p.MCS || (p.rotary_dim > 0 && pos >= p.rotary_positions)) {
    if ((lane & 15) == 0) flag_status(p.status, PKV_DEV_BAD_POSITION);
    return;
  }
  const int64_t src = ((int64_t)b * p.S + t) * p.src_stride + (int64_t)h * p.D;
  const int64_t dst = (((int64_t)b * p.Hkv + h) * p.MCS + pos) * p.D;
  move_row_pair(p.k_src + src, p.v_src + src, p.pk + dst, p.pv + dst, p.D, pos, p.cos, p.sin,
                p.rotary_dim, p.interleaved, lane);
}

template <bool kQ>
__global__ void __launch_bounds__(kScatterThreads) append_kernel(AppendParams p) {
  const int CPR = p.D / 8;
  const int64_t gid = (int64_t)blockIdx.x * kScatterThreads + threadIdx.x;
  const int64_t total = (int64_t)p.B * p.Hkv * p.S * CPR;
  if (gid >= total) return;
  const int c = (int)(gid % CPR);
  int64_t r = gid / CPR;
  const int t = (int)(r % p.S);
  r /= p.S;
  const int h = (int)(r % p.Hkv);
  const int b = (int)(r / p.Hkv);

  // history length: prompt mode when the scalar total equals the new-token count
  const uint32_t total0 = (uint32_t)p.total_seq[0];
  const uint32_t S = (uint32_t)p.S;
  uint32_t past = 0;
  if (total0 != S) {
    const uint32_t tb = (uint32_t)p.key_totals[b];
    past = tb >= S ? tb - S : 0u;
  }
  const int64_t pos = (int64_t)past + t;
  if constexpr (kQ) {   // the G query heads of kv head h, chunk c (unrotated past the table)
    const int G = p.Hq / p.Hkv;
    const int64_t qr = (int64_t)b * p.S + t;
    const bool rot = p.rotary_dim > 0 && c * 8 < p.rotary_dim && pos < p.rotary_positions;
#pragma unroll 1
    for (int g = 0; g < G; ++g) {
      const int hq = h * G + g;
      const __half* qrow = p.q_src + qr * p.q_stride + (int64_t)hq * p.D;
      __half x[8];
      *reinterpret_cast<uint4*>(x) = *reinterpret_cast<const uint4*>(qrow + c * 8);
      if (rot) rotate_chunk(x, qrow, c * 8, pos, p.cos, p.sin, p.rotary_dim, p.interleaved);
      *reinterpret_cast<uint4*>(p.q_dst + (qr * p.Hq + hq) * p.D + c * 8) =
          *reinterpret_cast<uint4*>(x);
    }
  }
  if (pos >= p.MCS || (p.rotary_dim > 0 && pos >= p.rotary_positions)) {
    if (c == 0) flag_status(p.status, PKV_DEV_BAD_POSITION);
    return;
  }
  const __half* krow = p.k_src + ((int64_t)b * p.S + t) * p.src_stride + (int64_t)h * p.D;
  const __half* vrow = p.v_src + ((int64_t)b * p.S + t) * p.src_stride + (int64_t)h * p.D;
  const int64_t dst = (((int64_t)b * p.Hkv + h) * p.MCS + pos) * p.D + c * 8;
  uint4 kv = *reinterpret_cast<const uint4*>(krow + c * 8);
  const uint4 vv = *reinterpret_cast<const uint4*>(vrow + c * 8);
  if (p.rotary_dim > 0 && c * 8 < p.rotary_dim) {
    __half x[8];
    *reinterpret_cast<uint4*>(x) = kv;
    rotate_chunk(x, krow, c * 8, pos, p.cos, p.sin, p.rotary_dim, p.interleaved);
    kv = *reinterpret_cast<uint4*>(x);
  }
  *reinterpret_cast<uint4*>(p.pk + dst) = kv;
  *reinterpret_cast<uint4*>(p.pv + dst) = vv;
}

}  // namespace

cudaError_t launch_paged_scatter(const ScatterParams& p, cudaStream_t s) {
  const int64_t total = scatter_threads(p);
  if (total == 0) return cudaSuccess;
  ProfScope ps("scatter", s);
  const unsigned grid = (unsigned)((total + kScatterThreads - 1) / kScatterThreads);
  if (p.row_path)
    paged_scatter_rows_kernel<<<grid, kScatterThreads, 0, s>>>(p);
  else
    paged_scatter_kernel<<<grid, kScatterThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_append(const AppendParams& p, cudaStream_t s) {
  const int64_t rows = (int64_t)p.B * p.Hkv * p.S;
  const int64_t total = p.row_path ? rows * 16 : rows * (p.D / 8);
  if (total == 0) return cudaSuccess;
  ProfScope ps("append", s);
  const unsigned grid = (unsigned)((total + kScatterThreads - 1) / kScatterThreads);
  if (p.row_path) {
    if (p.q_dst)
      append_rows_kernel<true><<<grid, kScatterThreads, 0, s>>>(p);
    else
      append_rows_kernel<false><<<grid, kScatterThreads, 0, s>>>(p);
  } else {
    if (p.q_dst)
      append_kernel<true><<<grid, kScatterThreads, 0, s>>>(p);
    else
      append_kernel<false><<<grid, kScatterThreads, 0, s>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace pkv
