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
//   sparse_rotary rule.
//
// One thread moves one 16-byte chunk (8 halves) of a K row and the matching V chunk;
// consecutive threads take consecutive chunks of a row, so loads and stores coalesce.
// The page's one-invocation-per-component dispatch and its 2-D dispatch folding
// (a WebGPU grid limit) are not needed: CUDA's grid is 1-D up to 2^31 - 1 blocks.
#include "device_common.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr int kScatterThreads = 256;

// rotated value of component d of a head row held as 8-element chunk `own` starting at
// d0, reading a partner outside the chunk from `row` (global memory).
__device__ __forceinline__ void rotate_chunk(__half (&x)[8], const __half* row, int d0,
                                             int64_t pos, const __half* cos_t,
                                             const __half* sin_t, int rotary_dim,
                                             int interleaved) {
  const int half = rotary_dim / 2;
  float out[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int d = d0 + e;
    const float own = __half2float(x[e]);
    out[e] = own;
    if (d < rotary_dim) {
      int slot, partner;
      bool first;
      if (interleaved) {
        slot = d >> 1;
        first = (d & 1) == 0;
        partner = first ? d + 1 : d - 1;
      } else {
        first = d < half;
        slot = first ? d : d - half;
        partner = first ? d + half : d - half;
      }
      const float pv = (partner >= d0 && partner < d0 + 8)
                           ? __half2float(x[partner - d0])
                           : __half2float(row[partner]);
      const float cs = __half2float(cos_t[pos * half + slot]);
      const float sn = __half2float(sin_t[pos * half + slot]);
      out[e] = first ? own * cs - pv * sn : own * cs + pv * sn;
    }
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) x[e] = __float2half_rn(out[e]);
}

__global__ void __launch_bounds__(kScatterThreads) paged_scatter_kernel(ScatterParams p) {
  const int CPR = p.D / 8;
  const int64_t gid = (int64_t)blockIdx.x * kScatterThreads + threadIdx.x;
  const int64_t total = (int64_t)p.T * p.Hkv * CPR;
  if (gid >= total) return;
  const int c = (int)(gid % CPR);
  const int64_t rh = gid / CPR;
  const int h = (int)(rh % p.Hkv);
  const int i = (int)(rh / p.Hkv);

  // sequence of token i: the last b with cu[b] <= i
  int lo = 0, hi = p.B - 1, b = -1;
  while (lo <= hi) {
    const int mid = (lo + hi) >> 1;
    if (p.cu[mid] <= i) {
      b = mid;
      lo = mid + 1;
    } else {
      hi = mid - 1;
    }
  }
  if (b < 0) return;
  const int s0 = p.cu[b], s1 = p.cu[b + 1], P = p.past[b];
  const bool valid = s0 >= 0 && s1 >= s0 && s1 <= p.T && P >= 0;
  if (!valid) {
    if (c == 0 && h == 0) flag_status(p.status, PKV_DEV_BAD_SEQUENCE);
    return;
  }
  if (i >= s1) return;  // token past the last sequence: not part of the batch
  const int64_t pos = (int64_t)P + (i - s0);

  int64_t blk, off;
  if (p.slot_mapping) {
    const int slot = p.slot_mapping[i];
    if (slot < 0) return;  // padding
    blk = slot / p.BS;
    off = slot % p.BS;
    if (blk >= p.NB) {
      if (c == 0) flag_status(p.status, PKV_DEV_BAD_SLOT);
      return;
    }
  } else {
    const int64_t col = pos / p.BS;
    if (col >= p.MB) {
      if (c == 0) flag_status(p.status, PKV_DEV_BAD_BLOCK);
      return;
    }
    blk = p.block_table[(int64_t)b * p.MB + col];
    off = pos % p.BS;
    if (blk < 0 || blk >= p.NB) {
      if (c == 0) flag_status(p.status, PKV_DEV_BAD_BLOCK);
      return;
    }
  }
  if (p.rotary_dim > 0 && pos >= p.rotary_positions) {
    if (c == 0) flag_status(p.status, PKV_DEV_BAD_POSITION);
    return;
  }
  const __half* krow = p.k_src + (int64_t)i * p.src_stride + (int64_t)h * p.D;
  const __half* vrow = p.v_src + (int64_t)i * p.src_stride + (int64_t)h * p.D;
  const int64_t dst = ((blk * p.BS + off) * p.Hkv + h) * p.D + c * 8;
  uint4 kv = *reinterpret_cast<const uint4*>(krow + c * 8);
  const uint4 vv = *reinterpret_cast<const uint4*>(vrow + c * 8);
  if (p.rotary_dim > 0 && c * 8 < p.rotary_dim) {
    __half x[8];
    *reinterpret_cast<uint4*>(x) = kv;
    rotate_chunk(x, krow, c * 8, pos, p.cos, p.sin, p.rotary_dim, p.interleaved);
    kv = *reinterpret_cast<uint4*>(x);
  }
  *reinterpret_cast<uint4*>(p.kc + dst) = kv;
  *reinterpret_cast<uint4*>(p.vc + dst) = vv;
}

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
  const int64_t total = (int64_t)p.T * p.Hkv * (p.D / 8);
  if (total == 0) return cudaSuccess;
  ProfScope ps("scatter", s);
  paged_scatter_kernel<<<(unsigned)((total + kScatterThreads - 1) / kScatterThreads),
                         kScatterThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_append(const AppendParams& p, cudaStream_t s) {
  const int64_t total = (int64_t)p.B * p.Hkv * p.S * (p.D / 8);
  if (total == 0) return cudaSuccess;
  ProfScope ps("append", s);
  append_kernel<<<(unsigned)((total + kScatterThreads - 1) / kScatterThreads),
                  kScatterThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace pkv
