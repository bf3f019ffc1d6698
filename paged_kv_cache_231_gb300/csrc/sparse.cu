// Block-sparse attention partials, from "alice-llm src/shaders/sparse_attention_forward.wgsl"
// (sparse_forward): per (edge, query-head lane) an fp32 partial (o, m, l) over the
// keys t < block_len of one KV block, unmapped pages scoring -1e30, weights exp(s - m)
// for s > -5e29, o unnormalised, empty edges giving (0, -1e30, 0).
//
// The page runs one 64-lane workgroup per partial and re-reads the block's K and V
// rows for every lane and edge. Here the edges are first grouped by (batch, kv head,
// block) with a device counting sort; the block's K and V are staged in shared memory
// once for the partials of every edge that names it. Head sizes 64 / 128 with blocks of
// at most 64 keys run both products on the tensor core in 3xTF32 (sparse_tc_kernel);
// other shapes take 64 query rows (edges x lanes) at a time with register-tiled fp32 FMA.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include "device_common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

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
  if (edge_keys(p, q_idx, blk, bl) <= 0) {   // every key after the query (causal)
    if (write) write_sentinel(p, e);
    return -1;
  }
  return ((int64_t)batch * p.nblk + blk) * p.hkv + h;
}

__global__ void sparse_count_kernel(SparseParams p) {
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= p.E) return;
  const int64_t key = edge_group(p, e, true);
  if (key >= 0) atomicAdd(&p.group_count[key], 1);
}

// exclusive scan of group_count into group_off (one CTA); clears the fill cursors. Thread i
// owns the i-th run of ceil(ngroups / 1024) consecutive groups: the run totals are scanned
// across the block (warp shuffles), then each thread walks its run.
__global__ void __launch_bounds__(1024) sparse_scan_kernel(SparseParams p) {
  __shared__ int warp_tot[32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t per = (p.ngroups + 1023) / 1024;
  const int64_t g0 = (int64_t)threadIdx.x * per;
  const int64_t g1 = g0 + per < p.ngroups ? g0 + per : p.ngroups;
  int run = 0;
  for (int64_t g = g0; g < g1; ++g) run += p.group_count[g];
  int x = run;   // inclusive scan of the run totals
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[w] = x;
  __syncthreads();
  if (w == 0) {
    int s = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_tot[lane] = s;
  }
  __syncthreads();
  int off = (w > 0 ? warp_tot[w - 1] : 0) + x - run;
  for (int64_t g = g0; g < g1; ++g) {
    p.group_off[g] = off;
    p.group_cursor[g] = 0;
    off += p.group_count[g];
  }
  if (threadIdx.x == 1023) p.group_off[p.ngroups] = warp_tot[31];
}

__global__ void sparse_fill_kernel(SparseParams p) {
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= p.E) return;
  const int64_t key = edge_group(p, e, false);
  if (key < 0) return;
  const int at = atomicAdd(&p.group_cursor[key], 1);
  const int pos = p.group_off[key] + at;
  p.perm[pos] = (int32_t)e;
  const int32_t* m = p.meta + e * 5;
  p.edge_rec[pos] = make_int4((int)e, m[0], edge_keys(p, m[0], m[2], m[4]), 0);
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
          sBL[r] = edge_keys(p, q_idx, p.meta[e * 5 + 2], p.meta[e * 5 + 4]);
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

// ---- tensor-core partials: 3xTF32 on tcgen05 ----------------------------------------
// For head size 64/128 and blocks of at most 64 keys. A persistent CTA per SM takes
// (batch, block, kv head) groups from a counter. The group's raw fp32 K and V rows are
// staged with cp.async while the previous group computes, then split into tf32 pairs
// x = hi + lo (hi = x rounded to tf32, lo = x - hi) in 128-byte-swizzled K-major tiles:
// K [64 keys][D] and V^T [D][64 keys]. For each tile of 128 query rows (edges x query
// heads) Q (hi, lo) goes to TMEM and S = Q K^T is accumulated from three tf32 products
// (hi*hi + hi*lo + lo*hi, relative error about 2^-22, i.e. fp32 level); one thread per row
// forms the partial's max, weights and sum, writes the weights (hi, lo) back to TMEM,
// and O = P V is accumulated the same way. TMEM: S 0..63, O 64.., Q hi 256.., Q lo 384..,
// P hi 256..319, P lo 320..383 (P replaces Q once S is complete).
namespace tcs {
constexpr int kThreads = 256;
constexpr int kNK = 64;                 // keys per block tile
constexpr uint32_t kTries = 1u << 24;   // default bound of each wait (polls)

__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
  return (1u << 4)                      // D format: f32
         | (2u << 7) | (2u << 10)       // A, B format: tf32
         | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "setp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n"
      "}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// L2 residency: the partials stream through once (evict first on store); Q rows are
// re-read by every edge that names their query (evict last).
__device__ __forceinline__ uint64_t l2_policy_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;\n" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ float4 ldg_hint(const float* gmem, uint64_t pol) {
  float4 v;
  asm volatile("ld.global.nc.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;\n"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(gmem), "l"(pol));
  return v;
}

// x rounded to the nearest tf32 (low 13 mantissa bits cleared)
__device__ __forceinline__ float tf32_hi(float x) {
  return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xffffe000u);
}

template <int D>
struct Layout {   // byte offsets from a 1024-byte-aligned base
  static constexpr uint32_t kKhi = 0;                       // [64][D]: D/32 x [64][128 B]
  static constexpr uint32_t kKlo = kKhi + D * 256;
  static constexpr uint32_t kVhi = kKlo + D * 256;          // [D][64]: 2 x [D][128 B]
  static constexpr uint32_t kVlo = kVhi + D * 256;
  static constexpr uint32_t kRawK = kVlo + D * 256;         // raw K, V as loaded by TMA:
  static constexpr uint32_t kRawV = kRawK + D * 256;        //   D/32 x [64 keys][128 B], swizzled
  static constexpr uint32_t kXfer = kRawV + D * 256;        // 8 warps x [32][32] fp32 transpose
  static constexpr uint32_t kValid = kXfer + 8 * 4096;      // key masks, current group (16 B)
  static constexpr uint32_t kRValid = kValid + 64;          // [64] key state, staged group
  static constexpr uint32_t kBar = kRValid + 64;            // MMA completion, drain, raw K/V
  static constexpr uint32_t kTmem = kBar + 24;
  static constexpr uint32_t kNext = kTmem + 8;              // int64, 8-byte aligned
  static constexpr uint32_t kEnd = kNext + 8;
};

struct SpMaps {     // TMA descriptors of the K and V pages (kernel parameters)
  CUtensorMap k;    // [pages * hkv * page_size rows][D] fp32, box 32 x page_size
  CUtensorMap v;
};

// One warp: group g's K and V pages by TMA (one box per page and 32-column slice, landing
// in the 128-byte-swizzled layout of the raw tiles) onto rbar; key states into rValid
// (0 unmapped or past the block, 1 mapped, 2 invalid table reference). Unmapped pages get
// no copy: the conversion writes zeros for their keys.
template <int D>
__device__ void stage_raw(const SparseParams& p, const SpMaps& maps, unsigned char* sm,
                          int64_t g, uint64_t* rbar, bool withhold = false) {
  using L = Layout<D>;
  const int lane = threadIdx.x & 31;
  uint8_t* rValid = sm + L::kRValid;
  const int h = (int)(g % p.hkv);
  const int64_t bb = g / p.hkv;
  const int blk = (int)(bb % p.nblk);
  const int batch = (int)(bb / p.nblk);
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int t = lane + 32 * k;
    uint8_t state = 0;
    if (t < p.block_size) {
      const int64_t slot = (int64_t)blk * p.ppb + t / p.page_size;
      if (slot < p.max_pages) {
        const int64_t page = p.bt[(int64_t)batch * p.max_pages + slot];
        state = page >= p.num_pages ? 2 : page >= 0 ? 1 : 0;
      } else {
        state = 2;
      }
    }
    rValid[t] = state;
  }
  int row0 = -1;   // first row of page `lane` of the block in the page tensors
  if (lane < p.ppb) {
    const int64_t slot = (int64_t)blk * p.ppb + lane;
    if (slot < p.max_pages) {
      const int64_t page = p.bt[(int64_t)batch * p.max_pages + slot];
      if (page >= 0 && page < p.num_pages) row0 = (int)((page * p.hkv + h) * p.page_size);
    }
  }
  const uint32_t bits = __ballot_sync(0xffffffffu, row0 >= 0);
  __syncwarp();   // the key states are published by lane 0's arrive
  if (lane == 0)
    tc::mbar_arrive_expect_tx(rbar, (uint32_t)__popc(bits) * (uint32_t)p.page_size * D * 4u * 2u);
  __syncwarp();
  if (row0 >= 0 && !withhold) {
#pragma unroll
    for (int q = 0; q < D / 32; ++q) {
      const uint32_t off = (uint32_t)q * (kNK * 128) + (uint32_t)(lane * p.page_size) * 128u;
      tc::tma_load_2d(sm + L::kRawK + off, &maps.k, q * 32, row0, rbar);
      tc::tma_load_2d(sm + L::kRawV + off, &maps.v, q * 32, row0, rbar);
    }
  }
}

// next group (in counter order) that has edges, or ngroups
__device__ __forceinline__ int64_t next_group(const SparseParams& p) {
  int* counter = p.group_count + p.ngroups;
  while (true) {
    const int64_t g = atomicAdd(counter, 1);
    if (g >= p.ngroups) return p.ngroups;
    if (p.group_off[g + 1] > p.group_off[g]) return g;
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    sparse_tc_kernel(SparseParams p, const __grid_constant__ SpMaps maps) {
  using L = Layout<D>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint32_t* sMask = reinterpret_cast<uint32_t*>(sm + L::kValid);   // {mapped, invalid} x 64 bits
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::kBar);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L::kTmem);
  volatile int64_t* snext = reinterpret_cast<volatile int64_t*>(sm + L::kNext);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, half = warp >> 2;
  const int r = quarter * 32 + lane;   // TMEM lane / tile row of this thread
  const uint32_t tries = p.wait_tries ? p.wait_tries : kTries;
  if (tid == 0) {
    tc::mbar_init(bar, 1);
    tc::mbar_init(bar + 1, 1);
    tc::mbar_init(bar + 2, 1);   // raw K / V landed (count 1 + tx)
    tc::mbar_init_fence();
    *snext = next_group(p);
  }
  if (warp == 0) {
    tc::tmem_alloc(tslot, 512);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;
  const uint32_t lane_tm = tmem + ((uint32_t)(quarter * 32) << 16);
  int64_t g = *snext;
  uint64_t* rbar = bar + 2;
  constexpr int kStageWarp = 7;
  if (warp == kStageWarp && g < p.ngroups) {
    if (lane == 0) {
      tc::tma_prefetch_desc(&maps.k);
      tc::tma_prefetch_desc(&maps.v);
    }
    // testing hook: the first staging is announced but never copied, so the wait for it
    // gives up with nothing in flight
    stage_raw<D>(p, maps, sm, g, rbar, p.withhold_copy != 0);
  }
  uint32_t raw_issued = g < p.ngroups ? 1u : 0u, raw_used = 0;
  uint32_t phase = 0;
  bool ok = true, bad = false;
  const uint64_t keep = l2_policy_last();
  // edge of this thread's row in a tile starting at edge c0 of a group ending at e1:
  // (edge, query index, block_len), fetched one tile ahead of its use
  const int epc = 128 / p.qhead;
  const int my_er = r / p.qhead, my_qh = r - my_er * p.qhead;
  auto row_edge = [&](int c0, int e1, int& e, int& qi, int& bl) {
    e = -1;
    qi = 0;
    bl = 0;
    if (my_er < epc && c0 + my_er < e1) {
      e = p.perm[c0 + my_er];
      qi = p.meta[(int64_t)e * 5];
      bl = edge_keys(p, qi, p.meta[(int64_t)e * 5 + 2], p.meta[(int64_t)e * 5 + 4]);
    }
  };
  int nx_e, nx_q, nx_bl;
  if (g < p.ngroups) row_edge(p.group_off[g], p.group_off[g + 1], nx_e, nx_q, nx_bl);
  // Row r of the warp's [32][32] fp32 transpose buffer holds its 16-byte chunk q at chunk
  // q ^ (r & 7): a lane's own row and a warp-wide 4-row x 128-byte slab both map to
  // distinct banks. Global rows are read and written whole (128 bytes per 8 lanes)
  // instead of one row per lane.
  float* xf = reinterpret_cast<float*>(sm + L::kXfer) + warp * 1024;
  // columns [col0, col0 + ncols) of the Q rows of this warp's 32 TMEM lanes (hi, lo) into
  // TMEM; zeros for padding rows
  auto load_q = [&](int h, int e, int qi, int col0, int ncols) {
    const float* myrow = e >= 0 ? p.q + ((int64_t)qi * p.hq + h * p.qhead + my_qh) * D : nullptr;
    const int q4 = lane & 7;
    for (int ch = 0; ch < ncols / 32; ++ch) {
      const int cbase = col0 + ch * 32;
#pragma unroll
      for (int i = 0; i < 8; ++i) {   // 4 rows x 32 floats per instruction
        const int rr = i * 4 + (lane >> 3);
        const float* src = reinterpret_cast<const float*>(
            __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(myrow), rr));
        const float4 v = src ? ldg_hint(src + cbase + q4 * 4, keep) : make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4*>(xf + rr * 32 + ((q4 ^ (rr & 7)) << 2)) = v;
      }
      __syncwarp();
      float vh[32], vl[32];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 v = *reinterpret_cast<const float4*>(xf + lane * 32 + ((q ^ (lane & 7)) << 2));
        const float x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) vh[q * 4 + j] = tf32_hi(x[j]);
        sub2(vl[q * 4], vl[q * 4 + 1], x[0], x[1], vh[q * 4], vh[q * 4 + 1]);
        sub2(vl[q * 4 + 2], vl[q * 4 + 3], x[2], x[3], vh[q * 4 + 2], vh[q * 4 + 3]);
      }
      __syncwarp();
      tc::tmem_st32(lane_tm + 256 + cbase, vh);
      tc::tmem_st32(lane_tm + 384 + cbase, vl);
    }
    tc::tmem_wait_st();
  };
  const uint32_t idesc_s = idesc_tf32(128, kNK), idesc_o = idesc_tf32(128, D);
  while (g < p.ngroups && ok) {
    ok = __syncthreads_and(tc::mbar_wait(rbar, raw_used & 1u, tries));
    ++raw_used;
    if (!ok) break;
    const uint8_t* rValid = sm + L::kRValid;
    // raw -> tf32 (hi, lo) tiles: K in place (the raw layout is the K-major tile layout),
    // V transposed (lane = key, conflict-free); keys not mapped become zeros
    for (int i = tid; i < kNK * (D / 4); i += kThreads) {
      const int t = i / (D / 4), c = i % (D / 4);
      const uint32_t off = (uint32_t)(c >> 3) * (kNK * 128) + tc::sw128(t, c & 7);
      float4 v = *reinterpret_cast<const float4*>(sm + L::kRawK + off);
      if (rValid[t] != 1) v = make_float4(0.f, 0.f, 0.f, 0.f);
      const float4 hi = make_float4(tf32_hi(v.x), tf32_hi(v.y), tf32_hi(v.z), tf32_hi(v.w));
      float4 lo;
      sub2(lo.x, lo.y, v.x, v.y, hi.x, hi.y);
      sub2(lo.z, lo.w, v.z, v.w, hi.z, hi.w);
      *reinterpret_cast<float4*>(sm + L::kKhi + off) = hi;
      *reinterpret_cast<float4*>(sm + L::kKlo + off) = lo;
    }
    {
      const int t = lane + 32 * (warp & 1);
      const bool live = rValid[t] == 1;
      for (int c = warp >> 1; c < D / 4; c += kThreads / 64) {
        float4 v = *reinterpret_cast<const float4*>(sm + L::kRawV + (uint32_t)(c >> 3) * (kNK * 128) +
                                                    tc::sw128(t, c & 7));
        if (!live) v = make_float4(0.f, 0.f, 0.f, 0.f);
        const float x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int d = c * 4 + k;
          const uint32_t off = (uint32_t)(t >> 5) * (D * 128) + (uint32_t)d * 128u +
                               ((uint32_t)(((t & 31) >> 2) ^ (d & 7)) << 4) + (uint32_t)(t & 3) * 4u;
          const float hi = tf32_hi(x[k]);
          *reinterpret_cast<float*>(sm + L::kVhi + off) = hi;
          *reinterpret_cast<float*>(sm + L::kVlo + off) = x[k] - hi;
        }
      }
    }
    if (warp < 2) {   // the key masks of this group, 32 keys per warp
      const uint8_t st = rValid[tid];
      const uint32_t vb = __ballot_sync(0xffffffffu, st == 1);
      const uint32_t ib = __ballot_sync(0xffffffffu, st == 2);
      if (lane == 0) {
        sMask[warp] = vb;
        sMask[2 + warp] = ib;
      }
    }
    tc::fence_async_shared();
    if (tid == 0) *snext = next_group(p);
    __syncthreads();
    // the raw buffers are free: stage the next group behind this one's compute
    const int64_t gn = *snext;
    if (gn < p.ngroups) {
      if (warp == kStageWarp) stage_raw<D>(p, maps, sm, gn, rbar);
      ++raw_issued;
    }
    // key masks of this group: bit t of vmask = mapped, of imask = invalid reference
    const uint64_t vmask = reinterpret_cast<const uint64_t*>(sMask)[0];
    const uint64_t imask = reinterpret_cast<const uint64_t*>(sMask)[1];
    const int e0 = p.group_off[g], e1 = p.group_off[g + 1];
    const int h = (int)(g % p.hkv);
    for (int c0 = e0; c0 < e1 && ok; c0 += epc) {
      // this tile's rows (fetched one tile ahead); Q of a group's first tile is loaded here
      // by all warps (column halves), later tiles' Q during the previous tile's epilogue
      const int cur_bl = nx_e >= 0 ? nx_bl : 0;
      const int cur_pi = nx_e >= 0 ? nx_e * p.qhead + my_qh : -1;
      if (c0 == e0) load_q(h, nx_e, nx_q, half * (D / 2), D / 2);
      tc::fence_before_sync();
      __syncthreads();
      if (tid == 0) {   // S = Qhi Khi + Qhi Klo + Qlo Khi
        tc::fence_after_sync();
        int n = 0;
#pragma unroll
        for (int pass = 0; pass < 3; ++pass) {
          const uint32_t a = tmem + (pass == 2 ? 384u : 256u);
          const uint32_t b = smem_u32(sm + (pass == 1 ? L::kKlo : L::kKhi));
#pragma unroll
          for (int ks = 0; ks < D / 8; ++ks, ++n)
            mma_tf32(tmem, a + ks * 8,
                     tc::smem_desc(b + (ks >> 2) * (kNK * 128) + (ks & 3) * 32, 16, 1024),
                     idesc_s, n > 0 ? 1u : 0u);
        }
        tc::commit(bar);
      }
      // the next tile's rows (later in this group, else the first tile of the next one),
      // fetched while S is computed: the dependent loads stall here, not on the next tile
      if (c0 + epc < e1) row_edge(c0 + epc, e1, nx_e, nx_q, nx_bl);
      else if (gn < p.ngroups) row_edge(p.group_off[gn], p.group_off[gn + 1], nx_e, nx_q, nx_bl);
      ok = __syncthreads_and(tc::mbar_wait(bar, phase & 1u, tries));
      ++phase;
      if (!ok) break;
      tc::fence_after_sync();
      float mrow = kNegLarge, lrow = 0.f;
      if (half == 0) {   // softmax of row r over the block's keys
        float s[64];
        float (*s32)[32] = reinterpret_cast<float (*)[32]>(s);
        tc::tmem_ld32(lane_tm, s32[0]);
        tc::tmem_ld32(lane_tm + 32, s32[1]);
        tc::tmem_wait_ld();
        const int bl = cur_bl;
        const uint64_t used = bl >= 64 ? ~0ull : ((1ull << bl) - 1ull);
        if (imask & used) bad = true;
        // keys that take part: mapped and inside the block (the rest score -1e30, and keys
        // past the block never raise m above that sentinel either)
        const uint64_t live = vmask & used;
        const uint32_t live_lo = (uint32_t)live, live_hi = (uint32_t)(live >> 32);
        // scores in base-2 units (scale * log2(e) * <q, k>): the weights are 2^(s - max);
        // four partial maxima and sums keep the dependency chains short
        // (pairs of keys go through one f32x2 instruction, each rounded as the scalar one)
        const float sl2 = p.scale * kLog2e;
        float mp[4] = {kNegLarge, kNegLarge, kNegLarge, kNegLarge};
#pragma unroll
        for (int t = 0; t < 64; t += 2) {
          const uint32_t word = t < 32 ? live_lo : live_hi;
          float x0, x1;
          fma2(x0, x1, s[t], s[t + 1], sl2, 0.f);
          s[t] = ((word >> (t & 31)) & 1u) ? x0 : kNegLarge;
          s[t + 1] = ((word >> ((t + 1) & 31)) & 1u) ? x1 : kNegLarge;
          mp[t & 3] = fmaxf(mp[t & 3], s[t]);
          mp[(t + 1) & 3] = fmaxf(mp[(t + 1) & 3], s[t + 1]);
        }
        const float m2 = fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3]));
        // 2^(-1e30 - m) is exactly 0 for every finite m; with no key taking part m is the
        // sentinel itself, and subtracting 0 instead keeps every weight 0
        const float msub = m2 > 0.5f * kNegLarge ? m2 : 0.f;
        float la[4] = {0.f, 0.f, 0.f, 0.f}, lb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int t = 0; t < 64; t += 2) {
          float d0, d1;
          fma2(d0, d1, s[t], s[t + 1], 1.f, -msub);   // s - m, exactly as a subtraction
          s[t] = ex2(d0);
          s[t + 1] = ex2(d1);
          add2(la[(t >> 1) & 3], lb[(t >> 1) & 3], s[t], s[t + 1]);
        }
        lrow = ((la[0] + lb[0]) + (la[1] + lb[1])) + ((la[2] + lb[2]) + (la[3] + lb[3]));
        // m in natural-log units (the -1e30 sentinel as is when no key takes part)
        mrow = m2 > 0.5f * kNegLarge ? m2 * 0.6931471805599453f : kNegLarge;
        float ph[32], pl[32];
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
#pragma unroll
          for (int k = 0; k < 32; k += 2) {
            ph[k] = tf32_hi(s[ch * 32 + k]);
            ph[k + 1] = tf32_hi(s[ch * 32 + k + 1]);
            sub2(pl[k], pl[k + 1], s[ch * 32 + k], s[ch * 32 + k + 1], ph[k], ph[k + 1]);
          }
          tc::tmem_st32(lane_tm + 256 + ch * 32, ph);
          tc::tmem_st32(lane_tm + 320 + ch * 32, pl);
        }
        tc::tmem_wait_st();
      }
      tc::fence_before_sync();
      __syncthreads();
      if (tid == 0) {   // O = Phi Vhi + Phi Vlo + Plo Vhi
        tc::fence_after_sync();
        int n = 0;
#pragma unroll
        for (int pass = 0; pass < 3; ++pass) {
          const uint32_t a = tmem + (pass == 2 ? 320u : 256u);
          const uint32_t b = smem_u32(sm + (pass == 1 ? L::kVlo : L::kVhi));
#pragma unroll
          for (int ks = 0; ks < kNK / 8; ++ks, ++n)
            mma_tf32(tmem + 64, a + ks * 8,
                     tc::smem_desc(b + (ks >> 2) * (D * 128) + (ks & 3) * 32, 16, 1024),
                     idesc_o, n > 0 ? 1u : 0u);
        }
        tc::commit(bar);
      }
      ok = __syncthreads_and(tc::mbar_wait(bar, phase & 1u, tries));
      ++phase;
      if (!ok) break;
      tc::fence_after_sync();
      if (half == 0) {   // write the partials of this tile (full rows, 128 bytes per 8 lanes)
        const int q4 = lane & 7;
#pragma unroll 1
        for (int ch = 0; ch < D / 32; ++ch) {
          float o[32];
          tc::tmem_ld32(lane_tm + 64 + ch * 32, o);
          tc::tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4*>(xf + lane * 32 + ((q ^ (lane & 7)) << 2)) =
                make_float4(o[q * 4], o[q * 4 + 1], o[q * 4 + 2], o[q * 4 + 3]);
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rr = i * 4 + (lane >> 3);
            const int pi = __shfl_sync(0xffffffffu, cur_pi, rr);
            const float4 v = *reinterpret_cast<const float4*>(xf + rr * 32 + ((q4 ^ (rr & 7)) << 2));
            if (pi >= 0) __stcs(reinterpret_cast<float4*>(p.o + (int64_t)pi * D + ch * 32 + q4 * 4), v);
          }
          __syncwarp();
        }
        if (cur_pi >= 0) {
          __stcs(p.m + cur_pi, mrow);
          __stcs(p.l + cur_pi, lrow);
        }
      } else if (c0 + epc < e1) {   // meanwhile the next tile's Q replaces P
        load_q(h, nx_e, nx_q, 0, D);
      }
      tc::fence_before_sync();
      __syncthreads();   // the next tile's S = Q K^T follows
      tc::fence_after_sync();
    }
    g = gn;
  }
  if (!ok) {
    // a wait gave up: let what this CTA issued finish before leaving
    if (tid == 0) {
      flag_status(p.status, PKV_DEV_TIMEOUT);
      tc::commit(bar + 1);
      tc::mbar_wait(bar + 1, 0, tries);
      if (raw_issued > raw_used) tc::mbar_wait(rbar, raw_used & 1u, tries);
    }
  }
  if (bad) flag_status(p.status, PKV_DEV_BAD_EDGE);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// [pages * hkv * page_size rows][D] fp32 pages, boxes of 32 columns x page_size rows in the
// 128-byte swizzle
bool encode_pages(CUtensorMap* m, const void* base, const SparseParams& p) {
  const PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)p.D, (cuuint64_t)(p.num_pages * p.hkv * p.page_size)};
  const cuuint64_t strides[1] = {(cuuint64_t)p.D * 4};
  const cuuint32_t box[2] = {32, (cuuint32_t)p.page_size};
  const cuuint32_t unit[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box,
            unit, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Shapes the tensor-core kernel takes: head size 64/128, blocks of at most 64 keys made of
// whole pages of a multiple of 8 rows (each page's box starts on a 1024-byte boundary)
bool eligible(const SparseParams& p) {
  return (p.D == 64 || p.D == 128) && p.block_size <= kNK && p.qhead <= 128 &&
         p.page_size % 8 == 0 && (int64_t)p.ppb * p.page_size <= kNK &&
         p.num_pages * p.hkv * p.page_size <= INT32_MAX;
}

template <int D>
cudaError_t launch_tc(const SparseParams& p, cudaStream_t s) {
  constexpr size_t smem = Layout<D>::kEnd + 1024;
  static_assert(smem <= 232448, "shared memory over the per-block limit");
  static std::atomic<uint64_t> configured{0};
  int dev = -1;
  if (needs_configure(configured, &dev)) {
    cudaError_t e = cudaFuncSetAttribute(sparse_tc_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    mark_configured(configured, dev);
  }
  int sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  SpMaps maps;
  if (!encode_pages(&maps.k, p.kp, p) || !encode_pages(&maps.v, p.vp, p))
    return cudaErrorInvalidValue;
  const int64_t grid = p.ngroups < sms ? p.ngroups : sms;
  ProfScope ps("sparse_partials", s);
  sparse_tc_kernel<D><<<(unsigned)grid, kThreads, smem, s>>>(p, maps);
  return cudaGetLastError();
}
}  // namespace tcs

template <int D, int KB>
cudaError_t launch_partials(const SparseParams& p, cudaStream_t s) {
  constexpr int KS = D + 4, PS = KB + 4;
  const size_t smem = sizeof(float) * ((size_t)KB * KS + (size_t)KB * D + kSpRows * KS +
                                       (KB <= D ? 0 : (size_t)kSpRows * PS));
  static std::atomic<uint64_t> configured{0};
  int dev = -1;
  if (needs_configure(configured, &dev)) {
    cudaError_t e = cudaFuncSetAttribute(sparse_partials_kernel<D, KB>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    mark_configured(configured, dev);
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
  if (p.f16) return launch_sparse_tc16(p, s);   // fp16 on the tensor core
  if (tcs::eligible(p)) {   // 3xTF32 on the tensor core
    if (p.D == 64) return tcs::launch_tc<64>(p, s);
    if (p.D == 128) return tcs::launch_tc<128>(p, s);
  }
  const int kb = p.block_size <= 64 ? 64 : 128;
  if (p.D == 64) return kb == 64 ? launch_partials<64, 64>(p, s) : launch_partials<64, 128>(p, s);
  if (p.D == 128)
    return kb == 64 ? launch_partials<128, 64>(p, s) : launch_partials<128, 128>(p, s);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
