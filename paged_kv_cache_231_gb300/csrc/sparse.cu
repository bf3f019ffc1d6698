// Block-sparse attention partials, from "alice-llm src/shaders/sparse_attention_forward.wgsl"
// (sparse_forward): per (edge, query-head lane) an fp32 partial (o, m, l) over the
// keys t < block_len of one KV block, unmapped pages scoring -1e30, weights exp(s - m)
// for s > -5e29, o unnormalised, empty edges giving (0, -1e30, 0).
//
// The page runs one 64-lane workgroup per partial and re-reads the block's K and V
// rows for every lane and edge. Here the edges are first grouped by (batch, kv head,
// block) with a device counting sort; the block's K and V are staged in shared memory
// once for the partials of every edge that names it. Head sizes 64 / 128 with blocks of
// at most 64 keys run both products on the tensor core from fp16 (hi, lo) splits of the
// fp32 operands, each block or half row scaled by a power of two (sparse_tc_kernel);
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
// across the block (warp shuffles), then each thread walks its run. Runs of 16 groups (the
// common case) are read and written as four 16-byte vectors, so a thread's run costs one
// memory round trip instead of sixteen.
__global__ void __launch_bounds__(1024) sparse_scan_kernel(SparseParams p) {
  __shared__ int warp_tot[32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t per = (p.ngroups + 1023) / 1024;
  const int64_t g0 = (int64_t)threadIdx.x * per;
  const int64_t g1 = g0 + per < p.ngroups ? g0 + per : p.ngroups;
  // whole vectors: the workspace arrays are 256-byte aligned, g0 is a multiple of 16
  const bool vec = per == 16 && g1 == g0 + 16;
  int4 c4[4];
  int run = 0;
  if (vec) {
    const int4* src = reinterpret_cast<const int4*>(p.group_count + g0);
#pragma unroll
    for (int k = 0; k < 4; ++k) c4[k] = src[k];
#pragma unroll
    for (int k = 0; k < 4; ++k) run += c4[k].x + c4[k].y + c4[k].z + c4[k].w;
  } else {
    for (int64_t g = g0; g < g1; ++g) run += p.group_count[g];
  }
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
  if (vec) {
    int4* dst = reinterpret_cast<int4*>(p.group_off + g0);
    int4* cur = reinterpret_cast<int4*>(p.group_cursor + g0);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      int4 o4;
      o4.x = off;
      o4.y = o4.x + c4[k].x;
      o4.z = o4.y + c4[k].y;
      o4.w = o4.z + c4[k].z;
      off = o4.w + c4[k].w;
      dst[k] = o4;
      cur[k] = make_int4(0, 0, 0, 0);
    }
  } else {
    for (int64_t g = g0; g < g1; ++g) {
      p.group_off[g] = off;
      p.group_cursor[g] = 0;
      off += p.group_count[g];
    }
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
  // the fp32 FMA kernel reads perm, the tensor-core kernels the edge records: the launch
  // passes only the array its partials kernel reads
  if (p.perm != nullptr) p.perm[pos] = (int32_t)e;
  if (p.edge_rec == nullptr) return;
  const int32_t* m = p.meta + e * 5;
  // with split Q rows (already written), the Q shifts of the edge's query heads as signed
  // bytes (up to four heads), so that the tensor-core kernel reads them with the record
  int shifts = 0;
  if (p.qshift != nullptr && p.qhead <= 4) {
    const int32_t* qs = p.qshift + ((int64_t)m[0] * p.hq + (int64_t)m[1] * p.qhead);
    for (int j = 0; j < p.qhead; ++j) shifts |= (qs[j] & 0xff) << (8 * j);
  }
  p.edge_rec[pos] = make_int4((int)e, m[0], edge_keys(p, m[0], m[2], m[4]), shifts);
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

// ---- tensor-core partials from split fp16 operands on tcgen05 -----------------------
// For head size 64/128 and blocks of at most 64 keys. A persistent CTA per SM takes
// (batch, block, kv head) groups from a counter. The group's raw fp32 K and V rows are
// staged by TMA and split in place into fp16 pairs x 2^s = hi + lo (s a power-of-two
// scale per block) in 128-byte-swizzled K-major tiles [64 keys][D]. For each tile of 128
// query rows (edges x query heads) Q (hi, lo), scaled per half row, goes to TMEM and
// S = Q K^T is accumulated from three fp16 products (hi*hi + hi*lo + lo*hi, relative
// error about 2^-21, i.e. fp32 level); one thread per row forms the partial's max,
// weights and sum, writes the weights (hi, lo) back to TMEM, and O = P V is accumulated
// the same way.
namespace tcs {
// L2 residency: Q rows are re-read by every edge that names their query (evict last).
__device__ __forceinline__ uint64_t l2_policy_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;\n" : "=l"(pol));
  return pol;
}

// ---- fp32 products from split fp16 operands ------------------------------------------
// An fp32 operand (a row of Q, a block of K or V) is scaled by a power of two 2^s,
// chosen from its largest magnitude so that the scaled values lie below 2^15 and the
// largest at or above 2^14, and written as two fp16 numbers: hi = fp16(x 2^s) and
// lo = fp16(x 2^s - hi). Their sum keeps 22 significant bits (as a tf32 pair does), and a
// product takes three fp16 MMAs with fp32 accumulation (hi*hi + hi*lo + lo*hi); the
// dropped lo*lo term is below 2^-22 of the product. The result is scaled back by the exact
// power of two.

// shift s that brings a largest magnitude m into [2^14, 2^15), kept within [-114, 120] so
// that 2^s and 2^-s are finite fp32 numbers
__device__ __forceinline__ int scale_shift(float m) {
  const int e = (int)((__float_as_uint(m) >> 23) & 0xffu);   // biased exponent
  const int s = 141 - e;                                      // 14 - (e - 127)
  return s > 120 ? 120 : s;
}
// 2^s for s in [-126, 127]
__device__ __forceinline__ float pow2f(int s) {
  return __uint_as_float((uint32_t)(s + 127) << 23);
}
// (hi, lo) fp16 pairs of two scaled values
__device__ __forceinline__ void split_pair(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = pack_half2(x0, x1);
  const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hi));
  float r0, r1;
  sub2(r0, r1, x0, x1, hf.x, hf.y);
  lo = pack_half2(r0, r1);
}
// 16 or 32 consecutive 32-bit columns of this thread's TMEM lane
template <int N>
__device__ __forceinline__ void tmem_st_u32(uint32_t taddr, const uint32_t (&v)[N]);
template <>
__device__ __forceinline__ void tmem_st_u32<32>(uint32_t taddr, const uint32_t (&v)[32]) {
  tc::tmem_st32(taddr, *reinterpret_cast<const float(*)[32]>(v));
}
template <>
__device__ __forceinline__ void tmem_st_u32<16>(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem], kind::f16, issued by one thread
__device__ __forceinline__ void mma_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "setp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n"
      "}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

struct SpMaps {     // TMA descriptors of the K and V pages (kernel parameters)
  CUtensorMap k;    // [pages * hkv * page_size rows][D] fp32, box 32 x page_size
  CUtensorMap v;
};

// next group (in counter order) that has edges, or ngroups
__device__ __forceinline__ int64_t next_group(const SparseParams& p) {
  int* counter = p.group_count + p.ngroups;
  while (true) {
    const int64_t g = atomicAdd(counter, 1);
    if (g >= p.ngroups) return p.ngroups;
    if (p.group_off[g + 1] > p.group_off[g]) return g;
  }
}

// Split pass over Q: every fp32 row (query, head) scaled by 2^s with s from the row's
// largest magnitude and written as fp16 (hi, lo), with s. The split arrays hold each
// 8-column chunk of all rows together (chunk-major), so that the threads of a tile (one row
// each) loading the same chunk of an edge's consecutive head rows read one contiguous run.
// A warp takes 8 consecutive rows, 4 lanes a row (D/4 columns each): every store then
// writes one chunk of 8 consecutive rows, 128 contiguous bytes.
template <int D>
__global__ void __launch_bounds__(256) qsplit_kernel(SparseParams p) {
  constexpr int PER = D / 4;    // values per lane
  constexpr int NCH = PER / 8;  // 8-column chunks per lane
  const int lane = threadIdx.x & 31;
  const int r8 = lane >> 2, j = lane & 3;
  const int64_t rows = p.Tq * p.hq;
  const int64_t stride = (int64_t)gridDim.x * 64;
  for (int64_t row0 = (int64_t)blockIdx.x * 64 + (threadIdx.x >> 5) * 8; row0 < rows;
       row0 += stride) {
    const int64_t row = row0 + r8;
    const bool ok = row < rows;
    float v[PER];
#pragma unroll
    for (int k = 0; k < PER / 4; ++k) {
      float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
      if (ok) x = *reinterpret_cast<const float4*>(p.q + row * D + j * PER + 4 * k);
      v[4 * k] = x.x; v[4 * k + 1] = x.y; v[4 * k + 2] = x.z; v[4 * k + 3] = x.w;
    }
    float mx = 0.f;
#pragma unroll
    for (int k = 0; k < PER; ++k) mx = fmaxf(mx, fabsf(v[k]));
    // the row's maximum over its 4 lanes (non-negative floats order as their bit patterns)
    uint32_t mb = __float_as_uint(mx);
    mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
    mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
    const int s = scale_shift(__uint_as_float(mb));
    const float f = pow2f(s);
    if (!ok) continue;
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float x0, x1;
        fma2(x0, x1, v[8 * c + 2 * k], v[8 * c + 2 * k + 1], f, 0.f);
        split_pair(x0, x1, hi[k], lo[k]);
      }
      // chunk-major: 8-column chunk ch of every row together ([D / 8][rows][8])
      const int64_t at = ((int64_t)(j * NCH + c) * rows + row) * 8;
      *reinterpret_cast<uint4*>(p.qhi + at) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(p.qlo + at) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    if (j == 0) p.qshift[row] = s;
  }
}

// Q arrives split: a pass before the kernel writes every fp32 Q row as fp16 (hi, lo), in
// chunk-major arrays, scaled by the row's own power of two, and that shift (which the
// grouping pass also packs into the edge records).
//
// Warp-specialised form: a persistent CTA of 16 warps per SM, every hand-off on an
// mbarrier.
//   warp 12 (scheduler): takes groups from the counter, publishes each in a 4-entry ring
//     with its 64-bit key masks (mapped, invalid reference), a group ahead of its staging,
//     and stages the group's raw fp32 K and V pages by TMA (one box per page and 32-column
//     slice) into one of two stages, once every product of the group that used the stage
//     last is done.
//   warps 8-11 (convert): at the first tile of a group, the raw K, then V, of its stage
//     split in place into (hi, lo) fp16 tiles (both in the K-major layout: K is the K-major
//     operand of S = Q K^T and V the MN-major operand of O = P V), each block scaled by its
//     own power of two; keys not mapped become zeros. The tile's K and V shifts go to a
//     ring of slots that the softmax and store warps release.
//   warps 4-7 (lower Q halves + store): per tile, the lower half of every split Q row; the
//     O rows of the previous tile from TMEM to memory, scaled back (through a per-warp
//     staging area, so that each store instruction writes whole 128-byte row segments).
//   warps 13, 14, lane 0 (S issuers): S = Q K^T of the even / odd tiles (24 MMAs of
//     128 x 64 x 16 for head size 128 into the tile parity's accumulator).
//   warp 15, lane 0 (O issuer): O = P V, P (hi, lo) read from TMEM (12 MMAs).
//   warps 0-3 (softmax, one thread per row): the row's scores from S and the shifts, m,
//     the weights and l; P' = 2^14 P (hi, lo) over the S columns; m and l to memory; then
//     the upper half of the split Q row of the tile two ahead into TMEM (its L2 round trip
//     off the chain of the converter warps).
// TMEM: S of tile parity b at 64 b (P' hi at +0 and lo at +32 once the scores are read), O
// at 128, Q (hi, lo) of tile parity b at 256 + D b (hi D/2 columns, then lo). With two S
// and two Q buffers the next tile's Q copy and S run while the softmax and O of this one
// do. Registers: warps 12-15 run on 72 a thread, the other twelve on 144 (setmaxnreg).
constexpr int kThreads = 512;
constexpr int kNK = 64;                 // keys per block tile
constexpr uint32_t kTries = 1u << 22;   // default bound of each wait (polls)
constexpr int kRing = 4;                // group ring entries
constexpr int kStages = 2;              // K/V stages (raw fp32 landed, then split in place)
constexpr int kScaleRing = 8;           // tile scale entries
constexpr int kSchedWarp = 12, kIssueS0 = 13, kIssueS1 = 14, kIssuePv = 15;
constexpr uint32_t kTmS = 0, kTmO = 128, kTmQ = 256;
constexpr int kPLog2 = 14;              // P' = 2^14 P keeps the lo parts of the weights normal
constexpr int kRegsIssue = 72, kRegsData = 144;   // registers per thread after the split
// bound of this CTA's waits (kTries unless a test lowered it), set before the first barrier
__shared__ uint32_t s_tries;

enum : int {
  kGFull = 0,                     // [kRing] entry published (scheduler, count 1)
  kGEmpty = kGFull + kRing,       // [kRing] entry released (15 consumer warps / threads)
  kRawFull = kGEmpty + kRing,     // [kStages] raw K/V of a group landed (1 arrival + tx)
  kKReady = kRawFull + kStages,   // [kStages] K (hi, lo) in place (4 converter warps)
  kVReady = kKReady + kStages,    // [kStages] V (hi, lo) in place (4 converter warps)
  kKFree = kVReady + kStages,     // [kStages] every S of the stage's group done (2 commits)
  kVFree = kKFree + kStages,      // [kStages] every O of the stage's group done (commit)
  kCvtK = kVFree + kStages,       // the converter warps' K block maxima posted (4 warps)
  kCvtV,                          // the same for V
  kQReady,                        // [2] Q (hi, lo) of a tile in buffer b (8 warps)
  kScale = kQReady + 2,           // [kScaleRing] K and V shifts of a tile posted (4 warps)
  kScaleFree = kScale + kScaleRing,   // [kScaleRing] a tile's shifts read (8 warps)
  kSFull = kScaleFree + kScaleRing,   // [2] S of a tile in buffer b (issuer b commits)
  kPFull = kSFull + 2,            // [2] P of a tile in buffer b (4 softmax warps)
  kPvDone = kPFull + 2,           // [2] O of a tile of parity b complete (commit)
  kOEmpty = kPvDone + 2,          // O read out of TMEM (4 store warps)
  kDrainS0, kDrainS1, kDrainPv,
  kNumBars
};

struct GroupEntry {   // ring entry: group (ngroups = end of work), edges, key masks
  long long g;
  int e0, e1;
  unsigned long long vmask, imask;
};
struct TileScales {   // scale shifts of one tile: K and V block of the tile's group
  int32_t sk, sv;
};

template <int D>
struct Layout {   // byte offsets from a 1024-byte-aligned base
  static constexpr uint32_t kHalf = D * 256;     // raw fp32 K (or V) of a block; its (hi, lo)
  static constexpr uint32_t kStage = 2 * kHalf;  // K, then V
  static constexpr uint32_t kSub = kNK * 128;    // a 32-column fp32 box or 64-column fp16 tile
  static constexpr uint32_t kLo = D * 128;       // lo tile after the hi tile
  static constexpr uint32_t kStgWarp = 32 * 128;  // a store warp's O staging: 32 rows x 128 B
  static constexpr uint32_t kStgOff = kStages * kStage;
  static constexpr uint32_t kRingOff = kStgOff + 4 * kStgWarp;
  static constexpr uint32_t kScaleOff = kRingOff + kRing * sizeof(GroupEntry);
  static constexpr uint32_t kMaxOff = kScaleOff + kScaleRing * sizeof(TileScales);
  static constexpr uint32_t kBar = kMaxOff + 8 * sizeof(float);
  static constexpr uint32_t kAbort = kBar + kNumBars * 8;
  static constexpr uint32_t kTmem = kAbort + 4;
  static constexpr uint32_t kEnd = kTmem + 4;
};

__device__ __forceinline__ void bar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
// Bounded wait for the phase of parity `parity`; false (and the abort flag raised) when the
// bound runs out or another role raised the flag.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort) {
  const uint32_t addr = smem_u32(bar);
  const uint32_t tries = s_tries;
  for (uint32_t i = 0; i < tries; ++i) {
    uint32_t done;
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) return true;
    if ((i & 255u) == 255u && *abort) return false;
  }
  *abort = 1;
  return false;
}
// the same for a whole warp (every lane polls; all agree on the outcome)
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  return __all_sync(0xffffffffu, wait_bar(bar, parity, abort));
}

// Ring entry gi (waiting for it); false at the end of the work or on abort.
__device__ __forceinline__ bool read_entry(const SparseParams& p, uint64_t* bars,
                                           const volatile GroupEntry* ring, uint32_t gi,
                                           volatile int* abort, bool whole_warp, GroupEntry& e) {
  const int slot = (int)(gi % kRing);
  const bool ok = whole_warp ? warp_wait(bars + kGFull + slot, (gi / kRing) & 1u, abort)
                             : wait_bar(bars + kGFull + slot, (gi / kRing) & 1u, abort);
  if (!ok) return false;
  e.g = ring[slot].g;
  e.e0 = ring[slot].e0;
  e.e1 = ring[slot].e1;
  e.vmask = ring[slot].vmask;
  e.imask = ring[slot].imask;
  return e.g < p.ngroups;
}

// Edge record of row `er` of the tile starting at edge c0 of a group ending at e1:
// (edge, query index, keys taking part, 0); x = -1 for a row past the group.
__device__ __forceinline__ int4 row_record(const SparseParams& p, int c0, int e1, int er,
                                           int epc) {
  if (er < epc && c0 + er < e1) return __ldg(p.edge_rec + c0 + er);
  return make_int4(-1, 0, 0, 0);
}
// Marks the point where a record loaded ahead is first used, so that no arithmetic on it
// (and no wait for its load) is moved up to the load.
__device__ __forceinline__ void settle(int4& r) {
  asm volatile("" : "+r"(r.x), "+r"(r.y), "+r"(r.z), "+r"(r.w));
}

// Warp 12: group scheduling, key masks and raw K/V staging. Ring entries are published one
// group ahead of the staging, so that the Q rows of a group's first tile can be fetched
// while the stage of the group two back is still in use.
template <int D>
__device__ void sched_role(const SparseParams& p, const SpMaps& maps, unsigned char* sm,
                           uint32_t (&issued)[kStages]) {
  using L = Layout<D>;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBar);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + L::kAbort);
  volatile GroupEntry* ring = reinterpret_cast<volatile GroupEntry*>(sm + L::kRingOff);
  const int lane = threadIdx.x & 31;
  if (lane == 0) {
    tc::tma_prefetch_desc(&maps.k);
    tc::tma_prefetch_desc(&maps.v);
  }
  // ring entry gi: the next group with edges (or the end) with its key masks; row0 = first
  // row of the group's page `lane` in the page tensors (-1: none)
  auto publish = [&](uint32_t gi, long long& g, int& row0) -> bool {
    g = 0;
    if (lane == 0) g = next_group(p);
    g = __shfl_sync(0xffffffffu, g, 0);
    const int slot = (int)(gi % kRing);
    if (gi >= kRing && !warp_wait(bars + kGEmpty + slot, ((gi / kRing) - 1) & 1u, abort))
      return false;
    uint64_t vmask = 0, imask = 0;
    int e0 = 0, e1 = 0;
    row0 = -1;
    if (g < p.ngroups) {
      const int h = (int)(g % p.hkv);
      const int64_t bb = g / p.hkv;
      const int blk = (int)(bb % p.nblk);
      const int batch = (int)(bb / p.nblk);
      // key states: 1 mapped, 2 invalid table reference, 0 unmapped or past the block
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int t = lane + 32 * k;
        int state = 0;
        if (t < p.block_size) {
          const int64_t slot_t = (int64_t)blk * p.ppb + t / p.page_size;
          if (slot_t < p.max_pages) {
            const int64_t page = p.bt[(int64_t)batch * p.max_pages + slot_t];
            state = page >= p.num_pages ? 2 : page >= 0 ? 1 : 0;
          } else {
            state = 2;
          }
        }
        vmask |= (uint64_t)__ballot_sync(0xffffffffu, state == 1) << (32 * k);
        imask |= (uint64_t)__ballot_sync(0xffffffffu, state == 2) << (32 * k);
      }
      if (lane < p.ppb) {
        const int64_t slot_t = (int64_t)blk * p.ppb + lane;
        if (slot_t < p.max_pages) {
          const int64_t page = p.bt[(int64_t)batch * p.max_pages + slot_t];
          if (page >= 0 && page < p.num_pages) row0 = (int)((page * p.hkv + h) * p.page_size);
        }
      }
      e0 = p.group_off[g];
      e1 = p.group_off[g + 1];
    }
    if (lane == 0) {
      ring[slot].g = g;
      ring[slot].e0 = e0;
      ring[slot].e1 = e1;
      ring[slot].vmask = vmask;
      ring[slot].imask = imask;
      bar_arrive(bars + kGFull + slot);   // release: the entry is visible to the waiters
    }
    return true;
  };
  long long g;
  int row0;
  if (!publish(0, g, row0)) return;
  for (uint32_t gi = 0; g < p.ngroups; ++gi) {
    long long g_next;
    int row0_next;
    if (!publish(gi + 1, g_next, row0_next)) return;
    // the stage is free once every S and every O of the group that used it last are done
    const uint32_t st = gi % kStages;
    if (gi >= kStages) {
      const uint32_t par = ((gi / kStages) - 1) & 1u;
      if (!warp_wait(bars + kKFree + st, par, abort)) return;
      if (!warp_wait(bars + kVFree + st, par, abort)) return;
    }
    const uint32_t bits = __ballot_sync(0xffffffffu, row0 >= 0);
    if (lane == 0)
      tc::mbar_arrive_expect_tx(bars + kRawFull + st,
                                (uint32_t)__popc(bits) * (uint32_t)p.page_size * D * 4u * 2u);
    __syncwarp();
    // testing hook: the first staging is announced but never copied, so the waits for it
    // give up with nothing in flight
    const bool withhold = p.withhold_copy && gi == 0;
    if (row0 >= 0 && !withhold) {
      unsigned char* kb = sm + st * L::kStage;
#pragma unroll
      for (int q = 0; q < D / 32; ++q) {
        const uint32_t off = (uint32_t)q * L::kSub + (uint32_t)(lane * p.page_size) * 128u;
        tc::tma_load_2d(kb + off, &maps.k, q * 32, row0, bars + kRawFull + st);
        tc::tma_load_2d(kb + L::kHalf + off, &maps.v, q * 32, row0, bars + kRawFull + st);
      }
    }
    ++issued[st];
    g = g_next;
    row0 = row0_next;
  }
}

// Splits the raw fp32 block at buf (64 keys x D as landed by TMA: D/32 boxes of
// [64 keys][128 B] in the 128-byte swizzle) in place into an fp16 hi tile at buf and a lo
// tile at buf + D*128 (64-column sub-tiles [64 keys][128 B] in the 128-byte swizzle), both
// scaled by 2^s with s from the block's largest magnitude (over the four warps that split it,
// posted on `bar`); keys not mapped become zeros. Every raw element is read before any
// warp writes. False on abort.
template <int D>
__device__ bool split_block(unsigned char* buf, uint64_t vmask, float* wmax, uint64_t* bar,
                            uint32_t parity, volatile int* abort, int ct, int& s_out) {
  using L = Layout<D>;
  constexpr int kItems = kNK * (D / 8) / 128;   // 8-column chunks per thread
  const int lane = ct & 31, wq = ct >> 5;
  float v[kItems][8];
  float mxs[kItems];
#pragma unroll
  for (int j = 0; j < kItems; ++j) {
    const int i = j * 128 + ct;
    const int tk = i & (kNK - 1), c8 = i >> 6;   // key, 8-column chunk
    const uint32_t box = (uint32_t)(c8 >> 2) * L::kSub;
    const uint32_t c16 = (uint32_t)(c8 & 3) * 2u;
    float4 a = *reinterpret_cast<const float4*>(buf + box + tc::sw128(tk, c16));
    float4 b = *reinterpret_cast<const float4*>(buf + box + tc::sw128(tk, c16 + 1u));
    if (!((vmask >> tk) & 1ull)) a = b = make_float4(0.f, 0.f, 0.f, 0.f);
    v[j][0] = a.x; v[j][1] = a.y; v[j][2] = a.z; v[j][3] = a.w;
    v[j][4] = b.x; v[j][5] = b.y; v[j][6] = b.z; v[j][7] = b.w;
    mxs[j] = fmaxf(fmaxf(fmaxf(fabsf(v[j][0]), fabsf(v[j][1])), fmaxf(fabsf(v[j][2]), fabsf(v[j][3]))),
                   fmaxf(fmaxf(fabsf(v[j][4]), fabsf(v[j][5])), fmaxf(fabsf(v[j][6]), fabsf(v[j][7]))));
  }
  float mx = mxs[0];
#pragma unroll
  for (int j = 1; j < kItems; ++j) mx = fmaxf(mx, mxs[j]);
  // non-negative floats order as their bit patterns
  const uint32_t wm = __reduce_max_sync(0xffffffffu, __float_as_uint(mx));
  if (lane == 0) {
    wmax[wq] = __uint_as_float(wm);
    bar_arrive(bar);   // release: this warp's maximum, and its reads of the raw block done
  }
  if (!warp_wait(bar, parity, abort)) return false;
  const float bm = fmaxf(fmaxf(wmax[0], wmax[1]), fmaxf(wmax[2], wmax[3]));
  const int s = scale_shift(bm);
  const float f = pow2f(s);
#pragma unroll
  for (int j = 0; j < kItems; ++j) {
    const int i = j * 128 + ct;
    const int tk = i & (kNK - 1), c8 = i >> 6;
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float x0, x1;
      fma2(x0, x1, v[j][2 * k], v[j][2 * k + 1], f, 0.f);
      split_pair(x0, x1, hi[k], lo[k]);
    }
    const uint32_t off = (uint32_t)(c8 >> 3) * L::kSub + tc::sw128(tk, (uint32_t)(c8 & 7));
    *reinterpret_cast<uint4*>(buf + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(buf + L::kLo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
  s_out = s;
  return true;
}

__device__ __forceinline__ uint4 ldg_hint_u4(const void* gmem, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(gmem), "l"(pol));
  return v;
}
// Half H (0: columns [0, D/2), 1: [D/2, D)) of a split Q row (hi and lo) into this
// thread's TMEM lane at q_tm (hi at + H*D/4, lo at + D/2 + H*D/4). The split arrays are
// chunk-major: 8-column chunk c of row r at (c * rows + r) * 8, so that the lanes of an
// edge's consecutive head rows read one contiguous run per load; hi0 / lo0 point at chunk 0
// of the row (nullptr: padding row, zeros). The row's loads are all issued before any is
// used (one round trip).
template <int D, int H>
__device__ __forceinline__ void copy_q_half(uint32_t q_tm, const __half* hi0, const __half* lo0,
                                            int64_t rows, uint64_t pol) {
  constexpr int NV = D / 16;   // 8-column chunks in half a row
  uint32_t h[NV * 4], l[NV * 4];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int64_t at = (int64_t)(H * NV + k) * rows * 8;
    const uint4 x = hi0 ? ldg_hint_u4(hi0 + at, pol) : make_uint4(0u, 0u, 0u, 0u);
    const uint4 y = lo0 ? ldg_hint_u4(lo0 + at, pol) : make_uint4(0u, 0u, 0u, 0u);
    h[4 * k] = x.x; h[4 * k + 1] = x.y; h[4 * k + 2] = x.z; h[4 * k + 3] = x.w;
    l[4 * k] = y.x; l[4 * k + 1] = y.y; l[4 * k + 2] = y.z; l[4 * k + 3] = y.w;
  }
  tmem_st_u32<NV * 4>(q_tm + H * (D / 4), h);
  tmem_st_u32<NV * 4>(q_tm + D / 2 + H * (D / 4), l);
  tc::tmem_wait_st();
}

// Walks the tiles in work order (ring entries read as needed) for this thread's row: the
// tile's edge record (load left in flight) and kv head; ok = false past the last tile or on
// abort.
struct TileCursor {
  uint32_t gi;
  int c0, e1;
  long long g;
  bool ok;
};
__device__ __forceinline__ void cursor_first(const SparseParams& p, uint64_t* bars,
                                             const volatile GroupEntry* ring,
                                             volatile int* abort, TileCursor& c) {
  GroupEntry e;
  c.ok = read_entry(p, bars, ring, 0, abort, true, e);
  c.gi = 0;
  c.c0 = e.e0;
  c.e1 = e.e1;
  c.g = e.g;
}
__device__ __forceinline__ void cursor_next(const SparseParams& p, uint64_t* bars,
                                            const volatile GroupEntry* ring, volatile int* abort,
                                            TileCursor& c) {
  if (!c.ok) return;
  const int epc = 128 / p.qhead;
  if (c.c0 + epc < c.e1) {
    c.c0 += epc;
    return;
  }
  GroupEntry e;
  c.ok = read_entry(p, bars, ring, c.gi + 1, abort, true, e);
  c.gi += 1;
  c.c0 = e.e0;
  c.e1 = e.e1;
  c.g = e.g;
}
// split Q row of this thread in the cursor's tile (-1: padding row or no tile)
__device__ __forceinline__ int64_t cursor_qrow(const SparseParams& p, const TileCursor& c,
                                               int4 rec, int my_qh) {
  if (!c.ok || rec.x < 0) return -1;
  return (int64_t)rec.y * p.hq + (int)(c.g % p.hkv) * p.qhead + my_qh;
}
__device__ __forceinline__ int4 cursor_record(const SparseParams& p, const TileCursor& c,
                                              int my_er) {
  const int epc = 128 / p.qhead;
  return c.ok ? row_record(p, c.c0, c.e1, my_er, epc) : make_int4(-1, 0, 0, 0);
}

// O rows (D columns) of this warp's 32 tile rows, 32 columns from column c, written out
// through the warp's staging area so that every store instruction writes whole 128-byte row
// segments: each lane puts its row (o, scaled by f) in place, then lanes copy 4 rows x 128
// bytes per instruction. `pj` holds, for lane i, the partial index of tile row 4 j + i / 8
// in slot j (-1: padding row).
template <int D>
__device__ __forceinline__ void store_o_chunk(unsigned char* stg, const float (&o)[32], float f,
                                              float* out, const int (&pj)[8], int c, int lane) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t off = (uint32_t)lane * 128u + (uint32_t)((k ^ (lane & 7)) * 16);
    *reinterpret_cast<float4*>(stg + off) =
        make_float4(o[4 * k] * f, o[4 * k + 1] * f, o[4 * k + 2] * f, o[4 * k + 3] * f);
  }
  __syncwarp();
  const int kk = lane & 7;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int row = 4 * j + (lane >> 3);
    const float4 v = *reinterpret_cast<const float4*>(
        stg + (uint32_t)row * 128u + (uint32_t)((kk ^ (row & 7)) * 16));
    if (pj[j] >= 0) __stcs(reinterpret_cast<float4*>(out + (int64_t)pj[j] * D + c) + kk, v);
  }
  __syncwarp();
}

// Warps 8-11: the K and V split of each group at its first tile; the tile's K and V shifts.
template <int D>
__device__ void convert_role(const SparseParams& p, unsigned char* sm) {
  using L = Layout<D>;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBar);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + L::kAbort);
  const volatile GroupEntry* ring = reinterpret_cast<const volatile GroupEntry*>(sm + L::kRingOff);
  TileScales* scales = reinterpret_cast<TileScales*>(sm + L::kScaleOff);
  float* wmax = reinterpret_cast<float*>(sm + L::kMaxOff);   // [K: 4][V: 4]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ct = (warp & 3) * 32 + lane;   // thread of the 128
  const int epc = 128 / p.qhead;
  uint32_t t = 0;
  for (uint32_t gi = 0;; ++gi) {
    GroupEntry e;
    if (!read_entry(p, bars, ring, gi, abort, true, e)) return;
    const uint32_t st = gi % kStages;
    unsigned char* kb = sm + st * L::kStage;
    int sk = 0, sv = 0;
    for (int c0 = e.e0; c0 < e.e1; c0 += epc, ++t) {
      // scale slot t % kScaleRing is free once both readers are done with tile t - kScaleRing
      if (t >= kScaleRing &&
          !warp_wait(bars + kScaleFree + t % kScaleRing, ((t / kScaleRing) - 1) & 1u, abort))
        return;
      if (c0 == e.e0) {   // K, then V, of this group once its raw block landed
        if (!warp_wait(bars + kRawFull + st, (gi / kStages) & 1u, abort)) return;
        if (!split_block<D>(kb, e.vmask, wmax, bars + kCvtK, gi & 1u, abort, ct, sk)) return;
        tc::fence_async_shared();
        __syncwarp();
        if (lane == 0) bar_arrive(bars + kKReady + st);
        if (!split_block<D>(kb + L::kHalf, e.vmask, wmax + 4, bars + kCvtV, gi & 1u, abort, ct,
                            sv))
          return;
        tc::fence_async_shared();
        __syncwarp();
        if (lane == 0) bar_arrive(bars + kVReady + st);
      }
      if (ct == 0) {
        scales[t % kScaleRing].sk = sk;
        scales[t % kScaleRing].sv = sv;
      }
      __syncwarp();
      if (lane == 0) bar_arrive(bars + kScale + t % kScaleRing);
    }
    __syncwarp();
    if (lane == 0) bar_arrive(bars + kGEmpty + (gi % kRing));
  }
}

// Warps 4-7: the lower Q half rows per tile; the O rows of the previous tile.
template <int D>
__device__ void store_role(const SparseParams& p, unsigned char* sm, uint32_t tmem) {
  using L = Layout<D>;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBar);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + L::kAbort);
  const volatile GroupEntry* ring = reinterpret_cast<const volatile GroupEntry*>(sm + L::kRingOff);
  const TileScales* scales = reinterpret_cast<const TileScales*>(sm + L::kScaleOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wq = warp & 3, r = wq * 32 + lane;
  const uint32_t lane_tm = tmem + ((uint32_t)(wq * 32) << 16);
  const int epc = 128 / p.qhead, my_er = r / p.qhead, my_qh = r - (r / p.qhead) * p.qhead;
  const uint64_t keep = l2_policy_last();
  unsigned char* stg = sm + L::kStgOff + (uint32_t)wq * L::kStgWarp;
  // O rows of tile tt (partial index pi, -1 = padding row) to memory: O' = 2^(14 + sv) O
  auto store = [&](uint32_t tt, int pi) -> bool {
    if (!warp_wait(bars + kPvDone + (tt & 1u), (tt >> 1) & 1u, abort)) return false;
    if (!warp_wait(bars + kScale + tt % kScaleRing, (tt / kScaleRing) & 1u, abort)) return false;
    tc::fence_after_sync();
    const float f = ldexpf(1.f, -(kPLog2 + scales[tt % kScaleRing].sv));
    __syncwarp();
    if (lane == 0) bar_arrive(bars + kScaleFree + tt % kScaleRing);
    int pj[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) pj[j] = __shfl_sync(0xffffffffu, pi, 4 * j + (lane >> 3));
#pragma unroll 1
    for (int ch = 0; ch < D / 32; ++ch) {
      float o[32];
      tc::tmem_ld32(lane_tm + kTmO + ch * 32, o);
      tc::tmem_wait_ld();
      store_o_chunk<D>(stg, o, f, p.o, pj, ch * 32, lane);
    }
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) bar_arrive(bars + kOEmpty);
    return true;
  };
  uint32_t t = 0;
  int prev_pi = -1;
  for (uint32_t gi = 0;; ++gi) {
    GroupEntry e;
    if (!read_entry(p, bars, ring, gi, abort, true, e)) break;
    const int h = (int)(e.g % p.hkv);
    int4 rec = row_record(p, e.e0, e.e1, my_er, epc);
    for (int c0 = e.e0; c0 < e.e1; c0 += epc, ++t) {
      const uint32_t b = t & 1u;
      if (t >= 2 && !warp_wait(bars + kSFull + b, ((t >> 1) - 1) & 1u, abort)) return;
      tc::fence_after_sync();
      settle(rec);
      const int64_t qrow = (int64_t)rec.y * p.hq + h * p.qhead + my_qh;
      copy_q_half<D, 0>(lane_tm + kTmQ + b * (uint32_t)D, rec.x >= 0 ? p.qhi + qrow * 8 : nullptr,
                        rec.x >= 0 ? p.qlo + qrow * 8 : nullptr, p.Tq * p.hq, keep);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) bar_arrive(bars + kQReady + b);
      const int pi = rec.x >= 0 ? rec.x * p.qhead + my_qh : -1;
      if (c0 + epc < e.e1) rec = row_record(p, c0 + epc, e.e1, my_er, epc);
      if (t > 0 && !store(t - 1, prev_pi)) return;
      prev_pi = pi;
    }
    __syncwarp();
    if (lane == 0) bar_arrive(bars + kGEmpty + (gi % kRing));
  }
  if (t > 0 && !*abort) store(t - 1, prev_pi);
}

// Warps 0-3: the softmax of each tile row over the block's keys.
template <int D>
__device__ void softmax_role(const SparseParams& p, unsigned char* sm, uint32_t tmem,
                             bool& bad) {
  using L = Layout<D>;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBar);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + L::kAbort);
  const volatile GroupEntry* ring = reinterpret_cast<const volatile GroupEntry*>(sm + L::kRingOff);
  const TileScales* scales = reinterpret_cast<const TileScales*>(sm + L::kScaleOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = warp * 32 + lane;
  const uint32_t lane_tm = tmem + ((uint32_t)(warp * 32) << 16);
  const int epc = 128 / p.qhead, my_er = r / p.qhead, my_qh = r - (r / p.qhead) * p.qhead;
  const float sl2 = p.scale * kLog2e;
  const float p_scale = (float)(1 << kPLog2);
  const uint64_t keep = l2_policy_last();
  // Upper Q half of the cursor's tile (if any) into TMEM buffer b, then QReady of that
  // buffer; the row's partial index, key count and Q shift join the queue of the tiles
  // ahead (entry 1 after entry 0; partial index -1: padding row).
  int pi0 = -1, pi1 = -1, keys0 = 0, keys1 = 0, sq0 = 0, sq1 = 0;
  auto q_upper = [&](const TileCursor& c, int4 rq, uint32_t b) {
    settle(rq);
    const int64_t qr = cursor_qrow(p, c, rq, my_qh);
    if (c.ok) {
      copy_q_half<D, 1>(lane_tm + kTmQ + b * (uint32_t)D, qr >= 0 ? p.qhi + qr * 8 : nullptr,
                        qr >= 0 ? p.qlo + qr * 8 : nullptr, p.Tq * p.hq, keep);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) bar_arrive(bars + kQReady + b);
    }
    pi0 = pi1;
    keys0 = keys1;
    sq0 = sq1;
    pi1 = qr >= 0 ? rq.x * p.qhead + my_qh : -1;
    keys1 = qr >= 0 ? rq.z : 0;
    sq1 = qr < 0 ? 0 : p.qhead <= 4 ? (int)(signed char)((uint32_t)rq.w >> (8 * my_qh))
                                    : __ldg(p.qshift + qr);
  };
  // tiles 0 and 1 now; tile t + 2 once the weights of tile t are out (S of tile t, the last
  // reader of buffer t & 1, is done), from a record loaded a tile before
  TileCursor cq;
  cursor_first(p, bars, ring, abort, cq);
  for (uint32_t k = 0; k < 2; ++k) {
    q_upper(cq, cursor_record(p, cq, my_er), k);
    cursor_next(p, bars, ring, abort, cq);
  }
  if (*abort) return;
  int4 rec_q = cursor_record(p, cq, my_er);
  uint32_t t = 0;
  for (uint32_t gi = 0;; ++gi) {
    GroupEntry e;
    if (!read_entry(p, bars, ring, gi, abort, true, e)) return;
    for (int c0 = e.e0; c0 < e.e1; c0 += epc, ++t) {
      const uint32_t b = t & 1u;
      // this tile's partial index, key count and Q shift lead the queue
      const int keys = keys0, pi = pi0, sq_t = sq0;
      // the shifts of this row's Q and of the block's K: S' = 2^(sq + sk) S
      if (!warp_wait(bars + kScale + t % kScaleRing, (t / kScaleRing) & 1u, abort)) return;
      const float f = ldexpf(sl2, -(sq_t + scales[t % kScaleRing].sk));
      __syncwarp();
      if (lane == 0) bar_arrive(bars + kScaleFree + t % kScaleRing);
      if (!warp_wait(bars + kSFull + b, (t >> 1) & 1u, abort)) return;
      tc::fence_after_sync();
      const uint32_t s_tm = lane_tm + kTmS + b * 64u;
      float s[64];
      float (*s32)[32] = reinterpret_cast<float (*)[32]>(s);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) tc::tmem_ld32(s_tm + hf * 32, s32[hf]);
      tc::tmem_wait_ld();
#pragma unroll
      for (int k = 0; k < 64; k += 2) fma2(s[k], s[k + 1], s[k], s[k + 1], f, 0.f);   // base-2 units
      const uint64_t used = keys >= 64 ? ~0ull : ((1ull << keys) - 1ull);
      if (e.imask & used) bad = true;
      // keys that take part: mapped and inside the block (the rest score -1e30, and keys
      // past the block never raise m above that sentinel either)
      const uint64_t live = e.vmask & used;
      const uint32_t live_lo = (uint32_t)live, live_hi = (uint32_t)(live >> 32);
      // the weights are 2^(s - max); four partial maxima and sums keep the chains short
      float mp[4] = {kNegLarge, kNegLarge, kNegLarge, kNegLarge};
#pragma unroll
      for (int k = 0; k < 64; ++k) {
        const uint32_t word = k < 32 ? live_lo : live_hi;
        s[k] = ((word >> (k & 31)) & 1u) ? s[k] : kNegLarge;
        mp[k & 3] = fmaxf(mp[k & 3], s[k]);
      }
      const float m2 = fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3]));
      // 2^(-1e30 - m) is exactly 0 for every finite m; with no key taking part m is the
      // sentinel itself, and subtracting 0 instead keeps every weight 0
      const float msub = m2 > 0.5f * kNegLarge ? m2 : 0.f;
      // the record of the tile two ahead is taken in hand before the exponentials, so that
      // the copy after the weights finds it loaded
      if (cq.ok) settle(rec_q);
      float la[4] = {0.f, 0.f, 0.f, 0.f}, lb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int k = 0; k < 64; k += 2) {
        float d0, d1;
        fma2(d0, d1, s[k], s[k + 1], 1.f, -msub);   // s - m, exactly as a subtraction
        s[k] = ex2(d0);
        s[k + 1] = ex2(d1);
        add2(la[(k >> 1) & 3], lb[(k >> 1) & 3], s[k], s[k + 1]);
      }
      const float lrow = ((la[0] + lb[0]) + (la[1] + lb[1])) + ((la[2] + lb[2]) + (la[3] + lb[3]));
      // m in natural-log units (the -1e30 sentinel as is when no key takes part)
      const float mrow = m2 > 0.5f * kNegLarge ? m2 * kLn2 : kNegLarge;
      uint32_t ph[32], pl[32];   // P' = 2^14 P as (hi, lo) fp16 pairs of keys
#pragma unroll
      for (int k = 0; k < 64; k += 2) {
        float w0, w1;
        fma2(w0, w1, s[k], s[k + 1], p_scale, 0.f);
        split_pair(w0, w1, ph[k / 2], pl[k / 2]);
      }
      tmem_st_u32<32>(s_tm, ph);
      tmem_st_u32<32>(s_tm + 32, pl);
      tc::tmem_wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) bar_arrive(bars + kPFull + b);
      if (pi >= 0) {
        __stcs(p.m + pi, mrow);
        __stcs(p.l + pi, lrow);
      }
      q_upper(cq, rec_q, b);
      if (cq.ok) {
        cursor_next(p, bars, ring, abort, cq);
        if (*abort) return;
        rec_q = cursor_record(p, cq, my_er);
      }
    }
    __syncwarp();
    if (lane == 0) bar_arrive(bars + kGEmpty + (gi % kRing));
  }
}

// Lane 0 of warps 13, 14: S = Q K^T of the tiles of parity `which`.
template <int D>
__device__ void s_issue_role(const SparseParams& p, unsigned char* sm, uint32_t tmem, int which) {
  using L = Layout<D>;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBar);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + L::kAbort);
  const volatile GroupEntry* ring = reinterpret_cast<const volatile GroupEntry*>(sm + L::kRingOff);
  const int epc = 128 / p.qhead;
  constexpr int KS = D / 16;   // k-steps of 16 along the head
  const uint32_t idesc = tc::idesc_f16(128, kNK, false, false);
  uint32_t t = 0;
  for (uint32_t gi = 0;; ++gi) {
    GroupEntry e;
    if (!read_entry(p, bars, ring, gi, abort, false, e)) return;
    const uint32_t st = gi % kStages;
    if (!wait_bar(bars + kKReady + st, (gi / kStages) & 1u, abort)) return;
    const uint32_t khi = smem_u32(sm + st * L::kStage), klo = khi + L::kLo;
    for (int c0 = e.e0; c0 < e.e1; c0 += epc, ++t) {
      const uint32_t b = t & 1u;
      if (b != (uint32_t)which) continue;
      if (!wait_bar(bars + kQReady + b, (t >> 1) & 1u, abort)) return;
      // buffer b holds P of tile t - 2 until its O is done
      if (t >= 2 && !wait_bar(bars + kPvDone + b, ((t >> 1) - 1) & 1u, abort)) return;
      tc::fence_after_sync();
      const uint32_t d_tm = tmem + kTmS + b * 64u;
      const uint32_t q_tm = tmem + kTmQ + b * (uint32_t)D;
      int n = 0;
#pragma unroll
      for (int pass = 0; pass < 3; ++pass) {   // Qhi Khi, Qhi Klo, Qlo Khi
#pragma unroll
        for (int kk = 0; kk < KS; ++kk, ++n) {
          const uint32_t a = q_tm + (pass == 2 ? (uint32_t)(D / 2) : 0u) + (uint32_t)kk * 8u;
          const uint32_t kbase = (pass == 1 ? klo : khi) + (uint32_t)(kk >> 2) * L::kSub +
                                 (uint32_t)(kk & 3) * 32u;
          mma_tmem_a(d_tm, a, tc::smem_desc(kbase, 16, 1024), idesc, n > 0 ? 1u : 0u);
        }
      }
      tc::commit(bars + kSFull + b);
    }
    // both issuers: every S of the group (of either parity) complete frees the K tiles
    tc::commit(bars + kKFree + st);
    bar_arrive(bars + kGEmpty + (gi % kRing));
  }
}

// Lane 0 of warp 15: O = P V (P' hi and lo from the first S accumulator's columns).
template <int D>
__device__ void pv_issue_role(const SparseParams& p, unsigned char* sm, uint32_t tmem) {
  using L = Layout<D>;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBar);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + L::kAbort);
  const volatile GroupEntry* ring = reinterpret_cast<const volatile GroupEntry*>(sm + L::kRingOff);
  const int epc = 128 / p.qhead;
  const uint32_t idesc = tc::idesc_f16(128, D, false, true);
  uint32_t t = 0;
  for (uint32_t gi = 0;; ++gi) {
    GroupEntry e;
    if (!read_entry(p, bars, ring, gi, abort, false, e)) return;
    const uint32_t st = gi % kStages;
    if (!wait_bar(bars + kVReady + st, (gi / kStages) & 1u, abort)) return;
    const uint32_t vhi = smem_u32(sm + st * L::kStage + L::kHalf), vlo = vhi + L::kLo;
    for (int c0 = e.e0; c0 < e.e1; c0 += epc, ++t) {
      const uint32_t b = t & 1u;
      if (!wait_bar(bars + kPFull + b, (t >> 1) & 1u, abort)) return;
      if (t > 0 && !wait_bar(bars + kOEmpty, (t - 1) & 1u, abort)) return;
      tc::fence_after_sync();
      int n = 0;
#pragma unroll
      for (int pass = 0; pass < 3; ++pass) {   // Phi Vhi, Phi Vlo, Plo Vhi
        const uint32_t a = tmem + kTmS + b * 64u + (pass == 2 ? 32u : 0u);
        const uint32_t vb = pass == 1 ? vlo : vhi;
#pragma unroll
        for (int ks = 0; ks < kNK / 16; ++ks, ++n)
          mma_tmem_a(tmem + kTmO, a + (uint32_t)ks * 8u,
                     tc::smem_desc(vb + (uint32_t)ks * 2048u, L::kSub, 1024), idesc,
                     n > 0 ? 1u : 0u);
      }
      tc::commit(bars + kPvDone + b);
      if (c0 + epc >= e.e1) tc::commit(bars + kVFree + st);
    }
    bar_arrive(bars + kGEmpty + (gi % kRing));
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    sparse_tc_kernel(SparseParams p, const __grid_constant__ SpMaps maps) {
  using L = Layout<D>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBar);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + L::kAbort);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L::kTmem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < kRing; ++i) {
      tc::mbar_init(bars + kGFull + i, 1);
      tc::mbar_init(bars + kGEmpty + i, 15);
    }
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(bars + kRawFull + s, 1);
      tc::mbar_init(bars + kKReady + s, 4);
      tc::mbar_init(bars + kVReady + s, 4);
      tc::mbar_init(bars + kKFree + s, 2);
      tc::mbar_init(bars + kVFree + s, 1);
    }
    tc::mbar_init(bars + kCvtK, 4);
    tc::mbar_init(bars + kCvtV, 4);
    for (int i = 0; i < kScaleRing; ++i) {
      tc::mbar_init(bars + kScale + i, 4);
      tc::mbar_init(bars + kScaleFree + i, 8);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(bars + kQReady + b, 8);
      tc::mbar_init(bars + kSFull + b, 1);
      tc::mbar_init(bars + kPFull + b, 4);
      tc::mbar_init(bars + kPvDone + b, 1);
    }
    tc::mbar_init(bars + kOEmpty, 4);
    tc::mbar_init(bars + kDrainS0, 1);
    tc::mbar_init(bars + kDrainS1, 1);
    tc::mbar_init(bars + kDrainPv, 1);
    *abort = 0;
    s_tries = p.wait_tries ? p.wait_tries : kTries;
    tc::mbar_init_fence();
  }
  if (warp == 0) {
    tc::tmem_alloc(tslot, 512);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;
  bool bad = false;
  uint32_t issued[kStages] = {};
  // registers: the scheduling and issuing warpgroup (warps 12-15) gives up part of its share
  // to the three data warpgroups; the launch holds 128 per thread
  static_assert(4 * 32 * kRegsIssue + 12 * 32 * kRegsData <= kThreads * 128,
                "register split over the launch's registers");
  if (warp >= 12)
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kRegsIssue) : "memory");
  else
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(kRegsData) : "memory");
  if (warp < 4) {
    softmax_role<D>(p, sm, tmem, bad);
  } else if (warp < 8) {
    store_role<D>(p, sm, tmem);
  } else if (warp < 12) {
    convert_role<D>(p, sm);
  } else if (warp == kSchedWarp) {
    sched_role<D>(p, maps, sm, issued);
    // a wait gave up: the last staging of each stage must land before the CTA leaves
    if (*abort) {
      for (int s = 0; s < kStages; ++s)
        if (issued[s] > 0) tc::mbar_wait(bars + kRawFull + s, (issued[s] - 1) & 1u, s_tries);
    }
  } else if (lane == 0) {
    const int drain = warp == kIssueS0 ? kDrainS0 : warp == kIssueS1 ? kDrainS1 : kDrainPv;
    if (warp == kIssuePv)
      pv_issue_role<D>(p, sm, tmem);
    else
      s_issue_role<D>(p, sm, tmem, warp - kIssueS0);
    // every MMA this thread issued completes before the CTA frees its tensor memory
    tc::commit(bars + drain);
    tc::mbar_wait(bars + drain, 0, s_tries);
  }
  if (bad) flag_status(p.status, PKV_DEV_BAD_EDGE);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (tid == 0 && *abort) flag_status(p.status, PKV_DEV_TIMEOUT);
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

// Q rows split into fp16 (hi, lo) and their shifts; runs before the edge grouping packs the
// shifts into the edge records
cudaError_t launch_qsplit(const SparseParams& p, cudaStream_t s) {
  const int64_t rows = p.Tq * p.hq;
  if (rows <= 0) return cudaSuccess;   // no query rows: no edge is valid
  int dev = -1, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  ProfScope ps("sparse_qsplit", s);
  const int64_t want = (rows + 63) / 64, cap = (int64_t)sms * 8;
  if (p.D == 64)
    qsplit_kernel<64><<<(unsigned)(want < cap ? want : cap), 256, 0, s>>>(p);
  else
    qsplit_kernel<128><<<(unsigned)(want < cap ? want : cap), 256, 0, s>>>(p);
  return cudaGetLastError();
}

bool eligible(const SparseParams& p) {
  return sparse_tc_shape(p.D, p.block_size, p.qhead, p.page_size, p.ppb,
                         p.num_pages * p.hkv * p.page_size, p.Tq * p.hq);
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

// Shapes the tensor-core kernel takes: head size 64/128, blocks of at most 64 keys made of
// whole pages of a multiple of 8 rows (each page's box starts on a 1024-byte boundary)
bool sparse_tc_shape(int D, int block_size, int qhead, int page_size, int ppb,
                     int64_t pool_rows, int64_t q_rows) {
  return (D == 64 || D == 128) && block_size <= tcs::kNK && qhead <= 128 &&
         page_size % 8 == 0 && (int64_t)ppb * page_size <= tcs::kNK && pool_rows <= INT32_MAX &&
         q_rows <= INT32_MAX;
}

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
  if (p.qshift != nullptr) {   // split Q rows (tensor-core path): before the fill reads shifts
    e = tcs::launch_qsplit(p, s);
    if (e != cudaSuccess) return e;
  }
  {
    ProfScope ps("sparse_group", s);
    SparseParams pf = p;
    if (p.f16 || tcs::eligible(p))
      pf.perm = nullptr;
    else
      pf.edge_rec = nullptr;
    sparse_fill_kernel<<<eg, 256, 0, s>>>(pf);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.ngroups == 0) return cudaSuccess;
  if (p.f16) return launch_sparse_tc16(p, s);   // fp16 on the tensor core
  if (tcs::eligible(p)) {   // split fp16 products on the tensor core
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
