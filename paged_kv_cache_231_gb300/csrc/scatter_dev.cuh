// Device code of the ScatterKV pass, shared by the standalone scatter kernel and the
// attention prologue kernel (which plans in block 0 and scatters in the others).
//
// "com.microsoft.PagedAttention manifest.json", ScatterKV: each new token's K and V
// rows go to the paged cache [num_blocks, block_size, kv_heads, head] at the row
// slot_mapping names, or at the block-table row of the token's absolute position
// past + t. Optionally the key is first rotated at that position with the rotation
// rule of "com.microsoft.SparseAttention sparse-kv-append.wgsl.jinja" (sparse_rotary),
// and the token's query heads are rotated at the same position into a separate buffer
// (the page rotates keys only; the query uses the same rule and tables).
#pragma once

#include "device_common.cuh"
#include "internal.h"

namespace pkv {

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

// Half a warp rotates one head row at position pos: lane c (of 16) holds chunk c (eight
// elements) in `x` and gets it back rotated when R > 0. A NeoX partner chunk comes from the
// lane of the half-warp that holds it and an interleaved partner from the same chunk; the
// cos/sin values of a chunk's slots are one vector load each. Needs row_path_ok(D, R, ...);
// every lane of the half-warp calls it (the two halves may take different rows).
__device__ __forceinline__ uint4 rope_chunk_half(uint4 x, bool live, int64_t pos,
                                                 const __half* cos_t, const __half* sin_t,
                                                 int R, int interleaved, int lane) {
  if (R <= 0) return x;
  const int c = lane & 15;
  const unsigned hmask = 0xFFFFu << (lane & 16);
  const int half = R / 2;
  const int hc = half / 8;   // NeoX: chunks per half
  const int pc = interleaved ? c : (c < hc ? c + hc : c - hc);
  const int src = (lane & 16) | (pc & 15);
  uint4 px;
  px.x = __shfl_sync(hmask, x.x, src);
  px.y = __shfl_sync(hmask, x.y, src);
  px.z = __shfl_sync(hmask, x.z, src);
  px.w = __shfl_sync(hmask, x.w, src);
  if (!live || c * 8 >= R) return x;
  __half own[8], par[8], cs[8], sn[8];
  *reinterpret_cast<uint4*>(own) = x;
  *reinterpret_cast<uint4*>(par) = px;
  bool first[8];
  if (interleaved) {   // pairs (2i, 2i+1), slot i
    const uint2 c2 = *reinterpret_cast<const uint2*>(cos_t + pos * half + c * 4);
    const uint2 s2 = *reinterpret_cast<const uint2*>(sin_t + pos * half + c * 4);
    __half c4[4], s4[4];
    *reinterpret_cast<uint2*>(c4) = c2;
    *reinterpret_cast<uint2*>(s4) = s2;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      first[e] = (e & 1) == 0;
      par[e] = own[e ^ 1];
      cs[e] = c4[e >> 1];
      sn[e] = s4[e >> 1];
    }
  } else {              // pairs (d, d + half), slot d mod half
    const bool f = c < hc;
    const int slot0 = f ? c * 8 : c * 8 - half;
    *reinterpret_cast<uint4*>(cs) = *reinterpret_cast<const uint4*>(cos_t + pos * half + slot0);
    *reinterpret_cast<uint4*>(sn) = *reinterpret_cast<const uint4*>(sin_t + pos * half + slot0);
#pragma unroll
    for (int e = 0; e < 8; ++e) first[e] = f;
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float o = __half2float(own[e]), pv = __half2float(par[e]);
    const float cf = __half2float(cs[e]), sf = __half2float(sn[e]);
    own[e] = __float2half_rn(first[e] ? o * cf - pv * sf : o * cf + pv * sf);
  }
  return *reinterpret_cast<uint4*>(own);
}

// Half a warp moves one (token, kv head) row pair: lane c (of 16) the K chunk c (rotated
// at position pos when R > 0) and the V chunk c.
__device__ __forceinline__ void move_row_pair(const __half* krow, const __half* vrow,
                                              __half* kdst, __half* vdst, int D, int64_t pos,
                                              const __half* cos_t, const __half* sin_t, int R,
                                              int interleaved, int lane) {
  const int c = lane & 15;
  const bool live = c < D / 8;
  uint4 x = make_uint4(0u, 0u, 0u, 0u), v = make_uint4(0u, 0u, 0u, 0u);
  if (live) {
    x = *reinterpret_cast<const uint4*>(krow + c * 8);
    v = *reinterpret_cast<const uint4*>(vrow + c * 8);
  }
  x = rope_chunk_half(x, live, pos, cos_t, sin_t, R, interleaved, lane);
  if (live) {
    *reinterpret_cast<uint4*>(kdst + c * 8) = x;
    *reinterpret_cast<uint4*>(vdst + c * 8) = v;
  }
}

// Half a warp rotates the G query heads of one (token, kv head) at position pos (R = 0:
// plain copy). Head g's row is at qsrc + g*D and goes to qdst + g*D; four heads' chunks
// are loaded before any is stored. Only the query-rotating kernels carry this code.
__device__ __forceinline__ void rotate_query_rows(const __half* qsrc, __half* qdst, int G,
                                                  int D, int64_t pos, const __half* cos_t,
                                                  const __half* sin_t, int R, int interleaved,
                                                  int lane) {
  const int c = lane & 15;
  const bool live = c < D / 8;
  for (int g0 = 0; g0 < G; g0 += 4) {
    uint4 x[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[j] = make_uint4(0u, 0u, 0u, 0u);
      if (live && g0 + j < G)
        x[j] = *reinterpret_cast<const uint4*>(qsrc + (int64_t)(g0 + j) * D + c * 8);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (g0 + j < G) {   // uniform over the half-warp
        x[j] = rope_chunk_half(x[j], live, pos, cos_t, sin_t, R, interleaved, lane);
        if (live) *reinterpret_cast<uint4*>(qdst + (int64_t)(g0 + j) * D + c * 8) = x[j];
      }
    }
  }
}

// Chunk c of the G query heads of kv head h of token i (copied unrotated past the table).
__device__ __forceinline__ void rotate_query_chunks(const ScatterParams& p, int i, int h, int c,
                                                 int64_t pos) {
  const int G = p.Hq / p.Hkv;
  const bool rot = p.rotary_dim > 0 && c * 8 < p.rotary_dim && pos < p.rotary_positions;
#pragma unroll 1
  for (int g = 0; g < G; ++g) {
    const int hq = h * G + g;
    const __half* qrow = p.q_src + (int64_t)i * p.q_stride + (int64_t)hq * p.D;
    __half x[8];
    *reinterpret_cast<uint4*>(x) = *reinterpret_cast<const uint4*>(qrow + c * 8);
    if (rot) rotate_chunk(x, qrow, c * 8, pos, p.cos, p.sin, p.rotary_dim, p.interleaved);
    *reinterpret_cast<uint4*>(p.q_dst + ((int64_t)i * p.Hq + hq) * p.D + c * 8) =
        *reinterpret_cast<uint4*>(x);
  }
}

// One thread of the ScatterKV pass: 16-byte chunk `gid` of the (token, kv head, chunk)
// grid moves K (rotated when asked) and V into the paged cache; with kQ, also the chunk of
// the token's query heads (the kernels without kQ carry none of that code).
template <bool kQ>
__device__ __forceinline__ void paged_scatter_thread(const ScatterParams& p, int64_t gid) {
  const int CPR = p.D / 8;
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
  if constexpr (kQ) rotate_query_chunks(p, i, h, c, pos);

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

// Half a warp of the ScatterKV pass on the row path: (token, kv head) row pair `row`;
// with kQ also the token's query heads of that kv head.
template <bool kQ>
__device__ __forceinline__ void paged_scatter_row(const ScatterParams& p, int64_t row,
                                                  int lane) {
  if (row >= (int64_t)p.T * p.Hkv) return;
  const int h = (int)(row % p.Hkv);
  const int i = (int)(row / p.Hkv);
  int lo = 0, hi = p.B - 1, b = -1;   // sequence of token i: the last b with cu[b] <= i
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
  if (!(s0 >= 0 && s1 >= s0 && s1 <= p.T && P >= 0)) {
    if ((lane & 15) == 0 && h == 0) flag_status(p.status, PKV_DEV_BAD_SEQUENCE);
    return;
  }
  if (i >= s1) return;
  const int64_t pos = (int64_t)P + (i - s0);
  if constexpr (kQ) {   // the G query heads of kv head h (copied unrotated past the table)
    const int G = p.Hq / p.Hkv;
    rotate_query_rows(p.q_src + (int64_t)i * p.q_stride + (int64_t)h * G * p.D,
                      p.q_dst + ((int64_t)i * p.Hq + (int64_t)h * G) * p.D, G, p.D, pos,
                      p.cos, p.sin, pos < p.rotary_positions ? p.rotary_dim : 0,
                      p.interleaved, lane);
  }
  int64_t blk, off;
  if (p.slot_mapping) {
    const int slot = p.slot_mapping[i];
    if (slot < 0) return;
    blk = slot / p.BS;
    off = slot % p.BS;
    if (blk >= p.NB) {
      if ((lane & 15) == 0) flag_status(p.status, PKV_DEV_BAD_SLOT);
      return;
    }
  } else {
    const int64_t col = pos / p.BS;
    if (col >= p.MB) {
      if ((lane & 15) == 0) flag_status(p.status, PKV_DEV_BAD_BLOCK);
      return;
    }
    blk = p.block_table[(int64_t)b * p.MB + col];
    off = pos % p.BS;
    if (blk < 0 || blk >= p.NB) {
      if ((lane & 15) == 0) flag_status(p.status, PKV_DEV_BAD_BLOCK);
      return;
    }
  }
  if (p.rotary_dim > 0 && pos >= p.rotary_positions) {
    if ((lane & 15) == 0) flag_status(p.status, PKV_DEV_BAD_POSITION);
    return;
  }
  const int64_t dst = ((blk * p.BS + off) * p.Hkv + h) * p.D;
  move_row_pair(p.k_src + (int64_t)i * p.src_stride + (int64_t)h * p.D,
                p.v_src + (int64_t)i * p.src_stride + (int64_t)h * p.D, p.kc + dst, p.vc + dst,
                p.D, pos, p.cos, p.sin, p.rotary_dim, p.interleaved, lane);
}

}  // namespace pkv
