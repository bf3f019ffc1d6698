// Block-sparse attention partials, from "alice-llm src/shaders/sparse_attention_forward.wgsl"
// (sparse_forward): per (edge, query-head lane) an fp32 partial (o, m, l) over the
// keys t < block_len of one KV block, unmapped pages scoring -1e30, weights exp(s - m)
// for s > -5e29, o unnormalised, empty edges giving (0, -1e30, 0).
//
// The page runs one 64-lane workgroup per partial and re-reads the block's K and V
// rows for every lane and edge. Here the edges are first grouped by (batch, kv head,
// block) with a device counting sort; one CTA stages a block's K and V in shared
// memory once and computes the partials of every edge that names it, 64 query rows
// (edges x lanes) at a time, with register-tiled fp32 FMA for both QK^T and PV.
#include <math.h>

#include "device_common.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr int kSpThreads = 256;
constexpr int kSpRows = 64;

__device__ __forceinline__ void write_sentinel(const SparseParams& p, int64_t e) {
  for (int qh = 0; qh < p.qhead; ++qh) {
    const int64_t pi = e * p.qhead + qh;
    float4* o = reinterpret_cast<float4*>(p.o + pi * p.D);
    for (int d = 0; d < p.D / 4; ++d) o[d] = make_float4(0.f, 0.f, 0.f, 0.f);
    p.m[pi] = kNegLarge;
    p.l[pi] = 0.f;
  }
}

// Returns the group key of edge e, or -1 if the edge is handled without a group
// (empty or invalid: its sentinel partials are written here when `write` is set).
__device__ __forceinline__ int64_t edge_group(const SparseParams& p, int64_t e, bool write) {
  const int32_t* m = p.meta + e * 5;
  const int q_idx = m[0], h = m[1], blk = m[2], batch = m[3], bl = m[4];
  if (bl <= 0) {
    if (write) write_sentinel(p, e);
    return -1;
  }
  const bool ok = q_idx >= 0 && q_idx < p.Tq && h >= 0 && h < p.hkv && batch >= 0 &&
                  batch < p.nseq && blk >= 0 && blk < p.nblk;
  if (!ok) {
    if (write) {
      write_sentinel(p, e);
      flag_status(p.status, PKV_DEV_BAD_EDGE);
    }
    return -1;
  }
  if (write && bl > p.block_size) flag_status(p.status, PKV_DEV_BAD_EDGE);
  return ((int64_t)batch * p.nblk + blk) * p.hkv + h;
}

__global__ void sparse_count_kernel(SparseParams p) {
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= p.E) return;
  const int64_t key = edge_group(p, e, true);
  if (key >= 0) atomicAdd(&p.group_count[key], 1);
}

// exclusive scan of group_count into group_off (one CTA); clears the fill cursors
__global__ void __launch_bounds__(1024) sparse_scan_kernel(SparseParams p) {
  __shared__ int s[1024];
  __shared__ int carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int64_t c0 = 0; c0 < p.ngroups; c0 += 1024) {
    const int64_t g = c0 + threadIdx.x;
    const int v = g < p.ngroups ? p.group_count[g] : 0;
    s[threadIdx.x] = v;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {
      const int x = threadIdx.x >= off ? s[threadIdx.x - off] : 0;
      __syncthreads();
      s[threadIdx.x] += x;
      __syncthreads();
    }
    if (g < p.ngroups) {
      p.group_off[g] = carry + s[threadIdx.x] - v;
      p.group_cursor[g] = 0;
    }
    __syncthreads();
    if (threadIdx.x == 1023) carry += s[1023];
    __syncthreads();
  }
  if (threadIdx.x == 0) p.group_off[p.ngroups] = carry;
}

__global__ void sparse_fill_kernel(SparseParams p) {
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= p.E) return;
  const int64_t key = edge_group(p, e, false);
  if (key < 0) return;
  const int at = atomicAdd(&p.group_cursor[key], 1);
  p.perm[p.group_off[key] + at] = (int32_t)e;
}

// One CTA per (batch, block, kv head) group. Thread (tr, tk) owns rows tr + 16 i and
// keys tk + 16 j (QK^T), then rows tr + 16 i and columns 4 td .. of each 64-wide slab
// (PV), td = tk.
template <int D, int KB>
__global__ void __launch_bounds__(kSpThreads, 2) sparse_partials_kernel(SparseParams p) {
  constexpr int KS = D + 4;                // padded row stride (floats) of K and Q
  constexpr int PS = KB + 4;               // padded row stride of P
  constexpr int KPT = KB / 16;             // keys per thread
  constexpr int DPT = D / 64;              // float4 columns per thread in PV
  extern __shared__ __align__(16) float sm[];
  float* sK = sm;                          // [KB][KS]
  float* sV = sK + KB * KS;                // [KB][D]
  float* sQ = sV + KB * D;                 // [kSpRows][KS]
  float* sP = (KB <= D) ? sQ : sQ + kSpRows * KS;  // [kSpRows][PS]
  __shared__ uint8_t sValid[KB];           // key state, see the staging loop
  __shared__ int sBL[kSpRows];
  __shared__ int sPI[kSpRows];             // partial index of each row, -1 = padding

  const int64_t grp = blockIdx.x;
  const int e0 = p.group_off[grp], e1 = p.group_off[grp + 1];
  if (e0 >= e1) return;
  const int h = (int)(grp % p.hkv);
  const int64_t bb = grp / p.hkv;
  const int blk = (int)(bb % p.nblk);
  const int batch = (int)(bb / p.nblk);
  const int tid = threadIdx.x;
  bool bad = false;

  // stage the block's K / V rows (unmapped or past the block: zero, invalid)
  for (int i = tid; i < KB * (D / 4); i += kSpThreads) {
    const int t = i / (D / 4), c = i % (D / 4);
    const int64_t slot = (int64_t)blk * p.ppb + t / p.page_size;
    int64_t page = -1;
    uint8_t state = 0;   // 0 unmapped, 1 mapped, 2 invalid reference (flag if used)
    if (t < p.block_size) {
      if (slot < p.max_pages) {
        page = p.bt[(int64_t)batch * p.max_pages + slot];
        if (page >= p.num_pages) {
          page = -1;
          state = 2;
        }
      } else {
        state = 2;
      }
    }
    if (page >= 0) state = 1;
    const float* gk = p.kp;
    const float* gv = p.vp;
    int nb = 0;
    if (page >= 0) {
      const int64_t row = ((page * p.hkv + h) * p.page_size + t % p.page_size) * D + c * 4;
      gk += row;
      gv += row;
      nb = 16;
    }
    cp_async_16(sK + t * KS + c * 4, gk, nb);
    cp_async_16(sV + t * D + c * 4, gv, nb);
    if (c == 0) sValid[t] = state;
  }
  cp_async_commit();

  const int epc = kSpRows / p.qhead;       // edges per chunk
  const int rows_pc = epc * p.qhead;
  const int tr = tid >> 4, tk = tid & 15;
  for (int c0 = e0; c0 < e1; c0 += epc) {
    // gather the chunk's query rows
    for (int i = tid; i < kSpRows * (D / 4); i += kSpThreads) {
      const int r = i / (D / 4), c = i % (D / 4);
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      const int er = r / p.qhead;
      if (r < rows_pc && c0 + er < e1) {
        const int64_t e = p.perm[c0 + er];
        const int qh = r - er * p.qhead;
        const int q_idx = p.meta[e * 5];
        v = *reinterpret_cast<const float4*>(
            p.q + ((int64_t)q_idx * p.hq + h * p.qhead + qh) * D + c * 4);
        if (c == 0) {
          sBL[r] = min(p.meta[e * 5 + 4], p.block_size);
          sPI[r] = (int)(e * p.qhead + qh);
        }
      } else if (c == 0) {
        sBL[r] = 0;
        sPI[r] = -1;
      }
      *reinterpret_cast<float4*>(sQ + r * KS + c * 4) = v;
    }
    cp_async_wait<0>();
    __syncthreads();

    // S = Q K^T
    float acc[4][KPT];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < KPT; ++j) acc[i][j] = 0.f;
#pragma unroll 4
    for (int d = 0; d < D; d += 4) {
      float4 qv[4], kv[KPT];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        qv[i] = *reinterpret_cast<const float4*>(sQ + (tr + 16 * i) * KS + d);
#pragma unroll
      for (int j = 0; j < KPT; ++j)
        kv[j] = *reinterpret_cast<const float4*>(sK + (tk + 16 * j) * KS + d);
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < KPT; ++j) {
          acc[i][j] = fmaf(qv[i].x, kv[j].x, acc[i][j]);
          acc[i][j] = fmaf(qv[i].y, kv[j].y, acc[i][j]);
          acc[i][j] = fmaf(qv[i].z, kv[j].z, acc[i][j]);
          acc[i][j] = fmaf(qv[i].w, kv[j].w, acc[i][j]);
        }
    }
    // softmax pieces per row (the 16 threads of a row are one half-warp)
    float mrow[4], lrow[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = tr + 16 * i;
      const int bl = sBL[r];
      float mx = kNegLarge;
#pragma unroll
      for (int j = 0; j < KPT; ++j) {
        const int t = tk + 16 * j;
        float s = -INFINITY;
        if (t < bl) {
          const uint8_t st = sValid[t];
          s = st == 1 ? acc[i][j] * p.scale : kNegLarge;
          if (st == 2) bad = true;
        }
        acc[i][j] = s;
        mx = fmaxf(mx, s);
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < KPT; ++j) {
        const float s = acc[i][j];
        const float w = s > 0.5f * kNegLarge ? ex2((s - mx) * kLog2e) : 0.f;
        acc[i][j] = w;
        sum += w;
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      mrow[i] = mx;
      lrow[i] = sum;
    }
    __syncthreads();   // all reads of sQ done before P overwrites it
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < KPT; ++j) sP[(tr + 16 * i) * PS + tk + 16 * j] = acc[i][j];
    __syncthreads();

    // O = P V (unnormalised)
    float o[4][DPT][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int c = 0; c < DPT; ++c) o[i][c][0] = o[i][c][1] = o[i][c][2] = o[i][c][3] = 0.f;
#pragma unroll 4
    for (int t = 0; t < KB; ++t) {
      float pw[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) pw[i] = sP[(tr + 16 * i) * PS + t];
#pragma unroll
      for (int c = 0; c < DPT; ++c) {
        const float4 v = *reinterpret_cast<const float4*>(sV + t * D + c * 64 + tk * 4);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          o[i][c][0] = fmaf(pw[i], v.x, o[i][c][0]);
          o[i][c][1] = fmaf(pw[i], v.y, o[i][c][1]);
          o[i][c][2] = fmaf(pw[i], v.z, o[i][c][2]);
          o[i][c][3] = fmaf(pw[i], v.w, o[i][c][3]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = tr + 16 * i;
      const int pi = sPI[r];
      if (pi < 0) continue;
#pragma unroll
      for (int c = 0; c < DPT; ++c)
        *reinterpret_cast<float4*>(p.o + (int64_t)pi * D + c * 64 + tk * 4) =
            make_float4(o[i][c][0], o[i][c][1], o[i][c][2], o[i][c][3]);
      if (tk == 0) {
        p.m[pi] = mrow[i];
        p.l[pi] = lrow[i];
      }
    }
    __syncthreads();   // sQ / sP / sBL / sPI reused by the next chunk
  }
  if (bad) flag_status(p.status, PKV_DEV_BAD_EDGE);
}

template <int D, int KB>
cudaError_t launch_partials(const SparseParams& p, cudaStream_t s) {
  constexpr int KS = D + 4, PS = KB + 4;
  const size_t smem = sizeof(float) * ((size_t)KB * KS + (size_t)KB * D + kSpRows * KS +
                                       (KB <= D ? 0 : (size_t)kSpRows * PS));
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(sparse_partials_kernel<D, KB>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  ProfScope ps("sparse_partials", s);
  sparse_partials_kernel<D, KB><<<(unsigned)p.ngroups, kSpThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_sparse(const SparseParams& p, cudaStream_t s) {
  if (p.E == 0) return cudaSuccess;
  const unsigned eg = (unsigned)((p.E + 255) / 256);
  cudaError_t e = cudaMemsetAsync(p.group_count, 0, sizeof(int32_t) * (p.ngroups + 1), s);
  if (e != cudaSuccess) return e;
  {
    ProfScope ps("sparse_group", s);
    sparse_count_kernel<<<eg, 256, 0, s>>>(p);
  }
  {
    ProfScope ps("sparse_group", s);
    sparse_scan_kernel<<<1, 1024, 0, s>>>(p);
  }
  {
    ProfScope ps("sparse_group", s);
    sparse_fill_kernel<<<eg, 256, 0, s>>>(p);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.ngroups == 0) return cudaSuccess;
  const int kb = p.block_size <= 64 ? 64 : 128;
  if (p.D == 64) return kb == 64 ? launch_partials<64, 64>(p, s) : launch_partials<64, 128>(p, s);
  if (p.D == 128)
    return kb == 64 ? launch_partials<128, 64>(p, s) : launch_partials<128, 128>(p, s);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
