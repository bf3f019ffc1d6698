// Paged causal GQA attention: device planner, split-KV decode kernel and tiled
// varlen prefill kernel.
//
// Operator: "com.microsoft.PagedAttention manifest.json" - AttendSplitK (one
// workgroup per (token, kv head, split) covering that kv head's query heads, fp32
// partials) and Attend (one workgroup per (token, kv head), whole causal key range).
// The GB300 form keeps the manifest's sharing of one K/V read across the qPerKv query
// heads of a kv head, but:
//   * a sequence with few new tokens (decode) is one row tile of (new tokens x query
//     heads) per kv head and is split along its keys; each split writes an fp32
//     (o, m, l) partial and a combine pass merges them;
//   * a sequence with many new tokens (prefill) is tiled over its query positions, so
//     K/V is read once per (tile, kv head) instead of once per token;
//   * K/V rows are gathered through block_table with 16-byte cp.async copies into a
//     multi-stage shared-memory ring, and QK^T / PV run on tensor cores
//     (mma.sync m16n8k16, fp16 in, fp32 accumulate) with the score accumulators
//     reused in registers as the A operand of PV.
#include <limits.h>
#include <math.h>

#include "device_common.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr int kThreads = 128;  // 4 warps per CTA for both attention kernels
constexpr int kWarps = 4;

template <int D>
struct Tile {
  static constexpr int CPR = D / 8;  // 16-byte chunks per head row
  // XOR swizzle so that 8 rows read at the same logical chunk hit 8 distinct bank groups
  static __device__ __forceinline__ int chunk(int r, int c) { return r * CPR + (c ^ (r & 7)); }
};

__device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

// Keys the last of N new tokens after P cached ones can see, clamped to what the block
// table addresses (keys past max_blocks * block_size are unmapped: masked, flagged).
__device__ __forceinline__ int seq_keys(const AttnParams& p, int P, int N) {
  return (int)min64((int64_t)P + N, (int64_t)p.MB * p.BS);
}

// Element offset of key j of (sequence b, kv head h) in the cache, or -1 if unmapped.
__device__ __forceinline__ int64_t key_row_offset(const AttnParams& p, int b, int h, int j) {
  int col, off;
  if (p.bs_shift >= 0) {
    col = j >> p.bs_shift;
    off = j & (p.BS - 1);
  } else {
    col = j / p.BS;
    off = j - col * p.BS;
  }
  if (col >= p.MB) return -1;
  const int blk = __ldg(&p.block_table[(int64_t)b * p.MB + col]);
  if (blk < 0 || (int64_t)blk >= p.NB) return -1;
  return (((int64_t)blk * p.BS + off) * p.Hkv + h) * p.D;
}

// Stage keys [k0, k0 + kStageKeys) of (b, h) into shared memory; keys at or past kend
// and unmapped keys are zero-filled and marked invalid.
template <int D>
__device__ __forceinline__ void load_stage(const AttnParams& p, int b, int h, int k0,
                                           int kend, __half* sK, __half* sV,
                                           uint8_t* sValid, bool& bad) {
  constexpr int CPR = D / 8;
  constexpr int TOTAL = kStageKeys * CPR;
  static_assert(TOTAL % kThreads == 0, "stage must split evenly over the CTA");
#pragma unroll
  for (int it = 0; it < TOTAL / kThreads; ++it) {
    const int i = threadIdx.x + it * kThreads;
    const int r = i / CPR;
    const int c = i % CPR;
    const int j = k0 + r;
    int64_t off = -1;
    if (j < kend) {
      off = key_row_offset(p, b, h, j);
      if (off < 0) bad = true;
    }
    const __half* gk = p.kc;
    const __half* gv = p.vc;
    int nbytes = 0;
    if (off >= 0) {
      gk += off + c * 8;
      gv += off + c * 8;
      nbytes = 16;
    }
    const int sidx = Tile<D>::chunk(r, c) * 8;
    cp_async_16(sK + sidx, gk, nbytes);
    cp_async_16(sV + sidx, gv, nbytes);
    if (c == 0) sValid[r] = off >= 0 ? 1 : 0;
  }
}

__device__ __forceinline__ uint32_t ld_half2(const __half* ptr) {
  return __ldg(reinterpret_cast<const unsigned int*>(ptr));
}

// A-operand fragments of 16 query rows (rows g and g+8 of this lane); zero rows
// where ok[] is false.
template <int D>
__device__ __forceinline__ void load_q_frags(uint32_t (&qa)[D / 16][4],
                                             const __half* row0, const __half* row1,
                                             bool ok0, bool ok1, int t4) {
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const int c = ks * 16 + 2 * t4;
    qa[ks][0] = ok0 ? ld_half2(row0 + c) : 0u;
    qa[ks][1] = ok1 ? ld_half2(row1 + c) : 0u;
    qa[ks][2] = ok0 ? ld_half2(row0 + c + 8) : 0u;
    qa[ks][3] = ok1 ? ld_half2(row1 + c + 8) : 0u;
  }
}

// S(16 rows x 16 keys) = Q K^T for keys [kw, kw + 16) of the staged tile.
template <int D>
__device__ __forceinline__ void qk_16(float (&s0)[4], float (&s1)[4],
                                      const uint32_t (&qa)[D / 16][4], const __half* K,
                                      int kw, int lane) {
  const int key = kw + (lane & 7) + ((lane >> 4) << 3);
  const int half = (lane >> 3) & 1;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    uint32_t b0, b1, b2, b3;
    ldsm_x4(b0, b1, b2, b3, K + Tile<D>::chunk(key, 2 * ks + half) * 8);
    mma_16816(s0, qa[ks], b0, b1);
    mma_16816(s1, qa[ks], b2, b3);
  }
}

// O(16 rows x D) += P(16 rows x 16 keys) V for keys [kw, kw + 16) of the staged tile.
template <int D>
__device__ __forceinline__ void pv_16(float (&o)[D / 8][4], const uint32_t (&pa)[4],
                                      const __half* V, int kw, int lane) {
  const int key = kw + (lane & 7) + (((lane >> 3) & 1) << 3);
  const int half = lane >> 4;
#pragma unroll
  for (int j = 0; j < D / 16; ++j) {
    uint32_t b0, b1, b2, b3;
    ldsm_x4_t(b0, b1, b2, b3, V + Tile<D>::chunk(key, 2 * j + half) * 8);
    mma_16816(o[2 * j], pa, b0, b1);
    mma_16816(o[2 * j + 1], pa, b2, b3);
  }
}

// ----------------------------------------------------------------------------------
// Split-KV decode: CTA = one split of one short sequence for one kv head; the 4 warps
// take 16 keys each of every 64-key stage and merge their softmax states at the end.
// ----------------------------------------------------------------------------------
template <int D, int NSTAGE>
__global__ void __launch_bounds__(kThreads) decode_kernel(AttnParams p) {
  constexpr int SK = kStageKeys;
  constexpr int DN = D / 8;
  extern __shared__ __align__(128) unsigned char smem[];
  __half* sK = reinterpret_cast<__half*>(smem);
  __half* sV = sK + NSTAGE * SK * D;
  uint8_t* sValid = reinterpret_cast<uint8_t*>(sV + NSTAGE * SK * D);

  const int h = blockIdx.x % p.Hkv;
  const int64_t item_idx = blockIdx.x / p.Hkv;
  if (item_idx >= p.counts[0]) return;
  const DecodeItem it = p.dec_items[item_idx];
  const int b = it.b;
  const int cu0 = p.cu[b];
  const int P = p.past[b];
  const int n = seq_keys(p, P, it.nq);
  const int kb = it.split * it.chunk;
  const int ke = min(n, kb + it.chunk);
  const int R = it.nq * p.G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;

  int lim[2];
  uint32_t qa[D / 16][4];
  {
    const __half* rows[2];
    bool ok[2];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int r = g + 8 * hr;
      ok[hr] = r < R;
      const int pos = ok[hr] ? r / p.G : 0;
      const int gg = ok[hr] ? r % p.G : 0;
      rows[hr] = p.q + (int64_t)(cu0 + pos) * p.q_stride + (int64_t)(h * p.G + gg) * D;
      lim[hr] = ok[hr] ? (int)min64((int64_t)P + pos, INT32_MAX) : -1;
    }
    load_q_frags<D>(qa, rows[0], rows[1], ok[0], ok[1], t4);
  }

  const int nst = ke > kb ? (ke - kb + SK - 1) / SK : 0;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  float o[DN][4];
#pragma unroll
  for (int i = 0; i < DN; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  bool bad = false;

#pragma unroll
  for (int s = 0; s < NSTAGE - 1; ++s) {
    if (s < nst)
      load_stage<D>(p, b, h, kb + s * SK, ke, sK + s * SK * D, sV + s * SK * D,
                    sValid + s * SK, bad);
    cp_async_commit();
  }
  for (int i = 0; i < nst; ++i) {
    cp_async_wait<NSTAGE - 2>();
    __syncthreads();
    {
      const int nx = i + NSTAGE - 1;
      if (nx < nst) {
        const int bf = nx % NSTAGE;
        load_stage<D>(p, b, h, kb + nx * SK, ke, sK + bf * SK * D, sV + bf * SK * D,
                      sValid + bf * SK, bad);
      }
      cp_async_commit();
    }
    const int bf = i % NSTAGE;
    const __half* K = sK + bf * SK * D;
    const __half* V = sV + bf * SK * D;
    const uint8_t* vld = sValid + bf * SK;
    const int kw = warp * 16;
    const int kstage = kb + i * SK;
    if (kstage + kw < ke) {
      float s[2][4];
#pragma unroll
      for (int e = 0; e < 4; ++e) s[0][e] = s[1][e] = 0.f;
      qk_16<D>(s[0], s[1], qa, K, kw, lane);
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int kk = kw + nt * 8 + 2 * t4 + (e & 1);
          const bool ok = vld[kk] && (kstage + kk <= lim[e >> 1]);
          s[nt][e] = ok ? s[nt][e] * p.scale_log2 : -INFINITY;
        }
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        float mx = fmaxf(fmaxf(s[0][2 * hr], s[0][2 * hr + 1]),
                         fmaxf(s[1][2 * hr], s[1][2 * hr + 1]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float mnew = fmaxf(m_run[hr], mx);
        const float base = mnew == -INFINITY ? 0.f : mnew;
        const float alpha = ex2(m_run[hr] - base);
        m_run[hr] = mnew;
        float sum = 0.f;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            const float pv = ex2(s[nt][2 * hr + x] - base);
            s[nt][2 * hr + x] = pv;
            sum += pv;
          }
        l_run[hr] = l_run[hr] * alpha + sum;
#pragma unroll
        for (int d = 0; d < DN; ++d) {
          o[d][2 * hr] *= alpha;
          o[d][2 * hr + 1] *= alpha;
        }
      }
      uint32_t pa[4] = {pack_half2(s[0][0], s[0][1]), pack_half2(s[0][2], s[0][3]),
                        pack_half2(s[1][0], s[1][1]), pack_half2(s[1][2], s[1][3])};
      pv_16<D>(o, pa, V, kw, lane);
    }
  }
  cp_async_wait<0>();
  __syncthreads();

  // merge the 4 warps' states (stage buffers are free now)
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    l_run[hr] += __shfl_xor_sync(0xffffffffu, l_run[hr], 1);
    l_run[hr] += __shfl_xor_sync(0xffffffffu, l_run[hr], 2);
  }
  float* sO = reinterpret_cast<float*>(smem);  // [kWarps][16][D]
  float* sM = sO + kWarps * 16 * D;            // [kWarps][16]
  float* sL = sM + kWarps * 16;
#pragma unroll
  for (int d = 0; d < DN; ++d) {
    const int c = d * 8 + 2 * t4;
    *reinterpret_cast<float2*>(&sO[(warp * 16 + g) * D + c]) = make_float2(o[d][0], o[d][1]);
    *reinterpret_cast<float2*>(&sO[(warp * 16 + g + 8) * D + c]) =
        make_float2(o[d][2], o[d][3]);
  }
  if (t4 == 0) {
    sM[warp * 16 + g] = m_run[0];
    sM[warp * 16 + g + 8] = m_run[1];
    sL[warp * 16 + g] = l_run[0];
    sL[warp * 16 + g + 8] = l_run[1];
  }
  __syncthreads();
  for (int e = threadIdx.x; e < R * D; e += kThreads) {
    const int r = e / D, d = e % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sM[w * 16 + r]);
    float num = 0.f, L = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float wt = ex2(sM[w * 16 + r] - M);
        num += wt * sO[(w * 16 + r) * D + d];
        L += wt * sL[w * 16 + r];
      }
    }
    const int pos = r / p.G, gg = r % p.G;
    const int64_t prow =
        ((int64_t)(it.slot_base + pos) * p.Hq + h * p.G + gg) * p.max_splits + it.split;
    p.part_o[prow * D + d] = L > 0.f ? num : 0.f;
    if (d == 0) {
      p.part_m[prow] = L > 0.f ? M * kLn2 : kNegLarge;
      p.part_l[prow] = L;
    }
  }
  if (bad) flag_status(p.status, PKV_DEV_BAD_BLOCK);
}

// ----------------------------------------------------------------------------------
// Tiled prefill: CTA = one tile of query positions of one sequence for one kv head;
// warp w owns 16 rows = (16 / G) positions x G query heads; all warps stream the
// same K/V stages up to the tile's causal limit. Output is written directly.
// ----------------------------------------------------------------------------------
template <int D, int NSTAGE>
__global__ void __launch_bounds__(kThreads) prefill_kernel(AttnParams p) {
  constexpr int SK = kStageKeys;
  constexpr int DN = D / 8;
  extern __shared__ __align__(128) unsigned char smem[];
  __half* sK = reinterpret_cast<__half*>(smem);
  __half* sV = sK + NSTAGE * SK * D;
  uint8_t* sValid = reinterpret_cast<uint8_t*>(sV + NSTAGE * SK * D);

  const int h = blockIdx.x % p.Hkv;
  const int64_t item_idx = blockIdx.x / p.Hkv;
  if (item_idx >= p.counts[1]) return;
  const PrefillItem it = p.pre_items[item_idx];
  const int b = it.b;
  const int cu0 = p.cu[b];
  const int P = p.past[b];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int ppw = 16 / p.G;                 // positions per warp
  const int wpos0 = warp * ppw;             // first tile position of this warp
  const int wn = max(0, min(ppw, it.nq - wpos0));  // valid positions of this warp
  const int warp_lim =
      wn > 0 ? (int)min64((int64_t)P + it.q0 + wpos0 + wn - 1, INT32_MAX) : -1;
  const int kend = seq_keys(p, P, it.q0 + it.nq);

  int lim[2];
  bool rok[2];
  int rtok[2], rhq[2];
  uint32_t qa[D / 16][4];
  {
    const __half* rows[2];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int r = g + 8 * hr;
      const int pl = r / p.G;
      rok[hr] = r < ppw * p.G && pl < wn;
      const int pos = rok[hr] ? it.q0 + wpos0 + pl : 0;
      const int gg = rok[hr] ? r % p.G : 0;
      rtok[hr] = cu0 + pos;
      rhq[hr] = h * p.G + gg;
      rows[hr] = p.q + (int64_t)rtok[hr] * p.q_stride + (int64_t)rhq[hr] * D;
      lim[hr] = rok[hr] ? (int)min64((int64_t)P + pos, INT32_MAX) : -1;
    }
    load_q_frags<D>(qa, rows[0], rows[1], rok[0], rok[1], t4);
  }

  const int nst = (kend + SK - 1) / SK;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  float o[DN][4];
#pragma unroll
  for (int i = 0; i < DN; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  bool bad = false;

#pragma unroll
  for (int s = 0; s < NSTAGE - 1; ++s) {
    if (s < nst)
      load_stage<D>(p, b, h, s * SK, kend, sK + s * SK * D, sV + s * SK * D,
                    sValid + s * SK, bad);
    cp_async_commit();
  }
  for (int i = 0; i < nst; ++i) {
    cp_async_wait<NSTAGE - 2>();
    __syncthreads();
    {
      const int nx = i + NSTAGE - 1;
      if (nx < nst) {
        const int bf = nx % NSTAGE;
        load_stage<D>(p, b, h, nx * SK, kend, sK + bf * SK * D, sV + bf * SK * D,
                      sValid + bf * SK, bad);
      }
      cp_async_commit();
    }
    const int bf = i % NSTAGE;
    const __half* K = sK + bf * SK * D;
    const __half* V = sV + bf * SK * D;
    const uint8_t* vld = sValid + bf * SK;
    const int kstage = i * SK;
    if (kstage > warp_lim) continue;   // warp-uniform: everything here is in the future

    float s[8][4];
#pragma unroll
    for (int sub = 0; sub < 4; ++sub) {
#pragma unroll
      for (int e = 0; e < 4; ++e) s[2 * sub][e] = s[2 * sub + 1][e] = 0.f;
      if (kstage + sub * 16 <= warp_lim)
        qk_16<D>(s[2 * sub], s[2 * sub + 1], qa, K, sub * 16, lane);
    }
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int kk = nt * 8 + 2 * t4 + (e & 1);
        const bool ok = vld[kk] && (kstage + kk <= lim[e >> 1]);
        s[nt][e] = ok ? s[nt][e] * p.scale_log2 : -INFINITY;
      }
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      float mx = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) mx = fmaxf(mx, fmaxf(s[nt][2 * hr], s[nt][2 * hr + 1]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float mnew = fmaxf(m_run[hr], mx);
      const float base = mnew == -INFINITY ? 0.f : mnew;
      const float alpha = ex2(m_run[hr] - base);
      m_run[hr] = mnew;
      float sum = 0.f;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          const float pv = ex2(s[nt][2 * hr + x] - base);
          s[nt][2 * hr + x] = pv;
          sum += pv;
        }
      l_run[hr] = l_run[hr] * alpha + sum;
#pragma unroll
      for (int d = 0; d < DN; ++d) {
        o[d][2 * hr] *= alpha;
        o[d][2 * hr + 1] *= alpha;
      }
    }
#pragma unroll
    for (int sub = 0; sub < 4; ++sub) {
      if (kstage + sub * 16 > warp_lim) break;
      uint32_t pa[4] = {pack_half2(s[2 * sub][0], s[2 * sub][1]),
                        pack_half2(s[2 * sub][2], s[2 * sub][3]),
                        pack_half2(s[2 * sub + 1][0], s[2 * sub + 1][1]),
                        pack_half2(s[2 * sub + 1][2], s[2 * sub + 1][3])};
      pv_16<D>(o, pa, V, sub * 16, lane);
    }
  }
  cp_async_wait<0>();

#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    l_run[hr] += __shfl_xor_sync(0xffffffffu, l_run[hr], 1);
    l_run[hr] += __shfl_xor_sync(0xffffffffu, l_run[hr], 2);
  }
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    if (!rok[hr]) continue;
    const float inv = l_run[hr] > 0.f ? 1.f / l_run[hr] : 0.f;
    __half* orow = p.out + (int64_t)rtok[hr] * p.Hq * D + (int64_t)rhq[hr] * D;
#pragma unroll
    for (int d = 0; d < DN; ++d) {
      const __half2 v = __floats2half2_rn(o[d][2 * hr] * inv, o[d][2 * hr + 1] * inv);
      *reinterpret_cast<__half2*>(orow + d * 8 + 2 * t4) = v;
    }
  }
  if (bad) flag_status(p.status, PKV_DEV_BAD_BLOCK);
}

// ----------------------------------------------------------------------------------
// Planner: one CTA. Reads cu / past, decides per sequence between split-KV decode
// (new tokens <= dec_rows) and prefill tiles, and writes the work lists, the partial
// slot map and zero output rows for tokens no valid sequence covers.
// ----------------------------------------------------------------------------------
constexpr int kPlanThreads = 1024;

__device__ __forceinline__ bool seq_valid(const AttnParams& p, int b, int& lo, int& hi,
                                          int& P) {
  lo = p.cu[b];
  hi = p.cu[b + 1];
  P = p.past[b];
  return lo >= 0 && hi >= lo && hi <= p.T && P >= 0;
}

// inclusive block scan of three counters
__device__ void block_scan3(int& a, int& b, int& c, int& ta, int& tb, int& tc) {
  __shared__ int sa[kPlanThreads], sb[kPlanThreads], sc[kPlanThreads];
  const int tid = threadIdx.x;
  sa[tid] = a;
  sb[tid] = b;
  sc[tid] = c;
  __syncthreads();
  for (int off = 1; off < kPlanThreads; off <<= 1) {
    int xa = 0, xb = 0, xc = 0;
    if (tid >= off) {
      xa = sa[tid - off];
      xb = sb[tid - off];
      xc = sc[tid - off];
    }
    __syncthreads();
    sa[tid] += xa;
    sb[tid] += xb;
    sc[tid] += xc;
    __syncthreads();
  }
  a = sa[tid];
  b = sb[tid];
  c = sc[tid];
  ta = sa[kPlanThreads - 1];
  tb = sb[kPlanThreads - 1];
  tc = sc[kPlanThreads - 1];
  __syncthreads();
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(AttnParams p) {
  const int tid = threadIdx.x;
  __shared__ unsigned long long s_keys;
  __shared__ int s_bad, s_bad_block;
  if (tid == 0) {
    s_keys = 0ull;
    s_bad = 0;
    s_bad_block = 0;
  }
  __syncthreads();
  // total keys of the split-KV sequences, for the automatic split size
  unsigned long long keys = 0;
  for (int b = tid; b < p.B; b += kPlanThreads) {
    int lo, hi, P;
    if (seq_valid(p, b, lo, hi, P)) {
      const int N = hi - lo;
      if (N >= 1 && N <= p.dec_rows) keys += (unsigned long long)seq_keys(p, P, N);
      if (N >= 1 && (int64_t)P + N > (int64_t)p.MB * p.BS) s_bad_block = 1;
    } else {
      s_bad = 1;
    }
  }
  atomicAdd(&s_keys, keys);
  __syncthreads();
  int target = p.split_min_keys;
  if (p.split_policy == PKV_SPLIT_AUTO) {
    // aim for ~16 waves of 2 CTAs per SM over all (split, kv head) items
    const unsigned long long denom = (unsigned long long)p.num_sms * 2ull * 16ull;
    const unsigned long long want = (s_keys * (unsigned long long)p.Hkv + denom - 1) / denom;
    if (want > (unsigned long long)target) target = (int)min(want, 1ull << 30);
  }

  int base_dec = 0, base_pre = 0, base_slot = 0;
  for (int c0 = 0; c0 < p.B; c0 += kPlanThreads) {
    const int b = c0 + tid;
    int nd = 0, np = 0, ns = 0, S = 0, chunk = 0, N = 0, lo = 0, hi = 0, P = 0;
    if (b < p.B && seq_valid(p, b, lo, hi, P)) {
      N = hi - lo;
      if (N >= 1 && N <= p.dec_rows) {
        const int n = seq_keys(p, P, N);
        if (p.split_policy == PKV_SPLIT_AUTO)
          S = (n + target - 1) / target;
        else
          S = p.fixed_splits;
        S = max(1, min(S, p.max_splits));
        chunk = (n + S - 1) / S;
        chunk = (chunk + kStageKeys - 1) / kStageKeys * kStageKeys;
        S = (n + chunk - 1) / chunk;
        nd = S;
        ns = N;
      } else if (N > p.dec_rows) {
        np = (N + p.pre_rows - 1) / p.pre_rows;
      }
    }
    int od = nd, op = np, os = ns, td, tp, ts;
    block_scan3(od, op, os, td, tp, ts);
    od -= nd;
    op -= np;
    os -= ns;
    // writes stay inside the host-computed bounds even when overlapping (invalid) cu
    // ranges claim more tokens than exist
    nd = (int)max64(0, min64(nd, p.dec_bound - base_dec - od));
    np = (int)max64(0, min64(np, p.pre_bound - base_pre - op));
    ns = (int)max64(0, min64(ns, p.slot_bound - base_slot - os));
    if (nd > 0 && ns < N) nd = 0;   // a decode item needs all its partial slots
    for (int s = 0; s < nd; ++s) {
      DecodeItem itm;
      itm.b = b;
      itm.nq = N;
      itm.split = s;
      itm.nsplit = S;
      itm.chunk = chunk;
      itm.slot_base = base_slot + os;
      itm.pad0 = itm.pad1 = 0;
      p.dec_items[base_dec + od + s] = itm;
    }
    for (int k = 0; k < np; ++k) {   // the heaviest (latest) tile first
      PrefillItem itm;
      itm.b = b;
      itm.q0 = (np - 1 - k) * p.pre_rows;
      itm.nq = min(p.pre_rows, N - itm.q0);
      itm.pad = 0;
      p.pre_items[base_pre + op + k] = itm;
    }
    for (int t = 0; t < ns; ++t) {
      p.slot_token[base_slot + os + t] = lo + t;
      p.slot_splits[base_slot + os + t] = S;
    }
    base_dec += td;
    base_pre += tp;
    base_slot += ts;
  }
  if (tid == 0) {
    p.counts[0] = (int)min64(base_dec, p.dec_bound);
    p.counts[1] = (int)min64(base_pre, p.pre_bound);
    p.counts[2] = (int)min64(base_slot, p.slot_bound);
    if (s_bad) flag_status(p.status, PKV_DEV_BAD_SEQUENCE);
    if (s_bad_block) flag_status(p.status, PKV_DEV_BAD_BLOCK);
  }
  // tokens that no valid sequence covers get zero output
  for (int i = tid; i < p.T; i += kPlanThreads) {
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
    bool covered = false;
    if (b >= 0) {
      int s0, s1, P;
      covered = seq_valid(p, b, s0, s1, P) && i >= s0 && i < s1;
    }
    if (!covered) {
      uint4* row = reinterpret_cast<uint4*>(p.out + (int64_t)i * p.Hq * p.D);
      for (int c = 0; c < p.Hq * p.D / 8; ++c) row[c] = make_uint4(0, 0, 0, 0);
    }
  }
}

template <int D, int NSTAGE>
cudaError_t launch_attention_d(const AttnParams& p, cudaStream_t s) {
  const size_t smem = (size_t)NSTAGE * kStageKeys * D * 2 * sizeof(__half) +
                      (size_t)NSTAGE * kStageKeys;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, NSTAGE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(prefill_kernel<D, NSTAGE>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  {
    ProfScope ps("plan", s);
    plan_kernel<<<1, kPlanThreads, 0, s>>>(p);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.dec_bound > 0) {
    ProfScope ps("decode", s);
    decode_kernel<D, NSTAGE><<<(unsigned)(p.dec_bound * p.Hkv), kThreads, smem, s>>>(p);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.pre_bound > 0) {
    ProfScope ps("prefill", s);
    prefill_kernel<D, NSTAGE><<<(unsigned)(p.pre_bound * p.Hkv), kThreads, smem, s>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(const AttnParams& p, cudaStream_t s) {
  switch (p.D) {
    case 64:
      return launch_attention_d<64, 4>(p, s);
    case 128:
      return launch_attention_d<128, 3>(p, s);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
