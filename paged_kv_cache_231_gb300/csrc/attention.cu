// Paged causal GQA attention: prologue (device planner + ScatterKV), persistent
// attention kernel (stream-K split-KV decode with a fused LSE combine, then tiled
// varlen prefill), and a per-split decode kernel for fixed split policies.
//
// Operator: "com.microsoft.PagedAttention manifest.json" - ScatterKV, AttendSplitK
// (one workgroup per (token, kv head, split) covering that kv head's query heads, fp32
// partials), AttendSplitKMerge, and Attend (one workgroup per (token, kv head)). The
// GB300 form keeps the manifest's sharing of one K/V read across the qPerKv query heads
// of a kv head, and changes the schedule:
//   * decode (a sequence with few new tokens): the (sequence, kv head) key ranges of
//     the whole batch are cut into 16-key stages and laid end to end; every warp of a
//     persistent grid takes an equal run of stages ("stream-K"), streams them through
//     its own cp.async ring and writes an fp32 (o, m, l) partial wherever its run ends
//     inside a (sequence, kv head) range. The warp that completes a range last (atomic
//     ticket, no waiting) merges its partials into the fp16 output, so the split count
//     adapts per sequence and the load is balanced to one stage;
//   * prefill (many new tokens): tiles of query positions x query heads, taken by the
//     same persistent CTAs from an atomic counter, so K/V is read once per tile. For
//     head size 128 a tile is 128 rows on the 5th-generation tensor core: Q, K and V in
//     128-byte-swizzled shared memory, the S and O accumulators and P in tensor memory,
//     tcgen05.mma issued by two threads (S = Q K^T on one, O += P V on the other) and
//     completed through mbarriers, one softmax thread per row reading its TMEM lane and
//     keeping the row sum in a register;
//   * decode and the head-size-64 tiles run QK^T and PV on mma.sync m16n8k16 (fp16 in,
//     fp32 accumulate) with the score accumulators reused in registers as the A
//     operand of PV. Softmax works in base 2 (scores pre-scaled by log2 e).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <limits.h>
#include <math.h>

#include "device_common.cuh"
#include "internal.h"
#include "scatter_dev.cuh"
#include "tcgen05.cuh"

namespace pkv {
namespace {

// Decode ring depth (16-key stages per warp), warps per CTA and CTAs per SM of the
// persistent kernel; overridable at build time for tuning sweeps.
#ifndef PKV_DEC_STAGES
#define PKV_DEC_STAGES 3
#endif
#ifndef PKV_WARPS
#define PKV_WARPS 4
#endif
#ifndef PKV_CTAS_PER_SM
#define PKV_CTAS_PER_SM 2
#endif
constexpr int kWarps = PKV_WARPS;
constexpr int kThreads = 32 * kWarps;
constexpr int kCtasPerSm = PKV_CTAS_PER_SM;
constexpr int kDecStages = PKV_DEC_STAGES;
constexpr int kTileThreads = 128;   // prefill tiles and split items use 4 warps
constexpr int kTileWarps = kTileThreads / 32;
constexpr int kPrologueThreads = 256;

__device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

// Keys the last of N new tokens after P cached ones can see, clamped to what the block
// table addresses (keys past max_blocks * block_size are unmapped: masked, flagged).
__device__ __forceinline__ int seq_keys(const AttnParams& p, int P, int N) {
  return (int)min64((int64_t)P + N, (int64_t)p.MB * p.BS);
}

template <int D>
struct Tile {
  static constexpr int CPR = D / 8;  // 16-byte chunks per head row
  // XOR swizzle so that 8 rows read at the same logical chunk hit 8 distinct bank groups
  static __device__ __forceinline__ int chunk(int r, int c) { return r * CPR + (c ^ (r & 7)); }
};

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

// CTA-wide: stage keys [k0, k0 + kStageKeys) of (b, h); keys at or past kend and
// unmapped keys are zero-filled and marked invalid.
template <int D>
__device__ __forceinline__ void load_stage(const AttnParams& p, int b, int h, int k0,
                                           int kend, __half* sK, __half* sV,
                                           uint8_t* sValid, bool& bad) {
  constexpr int CPR = D / 8;
  constexpr int TOTAL = kStageKeys * CPR;
  static_assert(TOTAL % kTileThreads == 0, "stage must split evenly over 4 warps");
#pragma unroll
  for (int it = 0; it < TOTAL / kTileThreads; ++it) {
    const int i = threadIdx.x + it * kTileThreads;
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

// Warp-wide block-table lookup for a 16-key stage: lane r < 16 returns the element
// offset of key k0 + r of (b, h), or -1 when the key is past kend or unmapped.
__device__ __forceinline__ int64_t stage_row_offset(const AttnParams& p, int b, int h, int k0,
                                                    int kend, int lane, bool& bad) {
  if (lane >= 16) return -1;
  const int j = k0 + lane;
  if (j >= kend) return -1;
  const int64_t off = key_row_offset(p, b, h, j);
  if (off < 0) bad = true;
  return off;
}

// Warp-wide copy of a 16-key stage whose row offsets lanes 0..15 hold: each
// instruction moves whole 256-byte rows (consecutive lanes, consecutive 16-byte
// chunks), so every 32-byte sector is requested once.
template <int D>
__device__ __forceinline__ void warp_copy16(const AttnParams& p, int64_t my_off, __half* sK,
                                            __half* sV, uint8_t* sValid, int lane) {
  constexpr int CPR = D / 8;        // chunks per row
  constexpr int RPI = 32 / CPR;     // rows per instruction
  const int c = lane % CPR;
#pragma unroll
  for (int i = 0; i < 16 / RPI; ++i) {
    const int r = i * RPI + lane / CPR;
    const long long off = __shfl_sync(0xffffffffu, (long long)my_off, r);
    const int nb = off >= 0 ? 16 : 0;
    const __half* gk = off >= 0 ? p.kc + off + c * 8 : p.kc;
    const __half* gv = off >= 0 ? p.vc + off + c * 8 : p.vc;
    const int sidx = Tile<D>::chunk(r, c) * 8;
    cp_async_16(sK + sidx, gk, nb);
    cp_async_16(sV + sidx, gv, nb);
  }
  if (lane < 16) sValid[lane] = my_off >= 0 ? 1 : 0;
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

// Online-softmax update of the two rows (g, g+8) held by this lane for 16 new scores
// s[2][4] (already scaled to log2 units, -inf where masked); turns s into weights.
template <int DN>
__device__ __forceinline__ void softmax_16(float (&s)[2][4], float (&m_run)[2],
                                           float (&l_run)[2], float (&o)[DN][4]) {
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
}

// ----------------------------------------------------------------------------------
// Stream-K decode (phase 1 of the persistent kernel)
// ----------------------------------------------------------------------------------
__device__ __forceinline__ DecSeq load_seq(const AttnParams& p, int i) {
  const int4* q = reinterpret_cast<const int4*>(p.dec_seqs + i);
  const int4 a = q[0], b = q[1];
  DecSeq d;
  d.b = a.x;
  d.n = a.y;
  d.st = a.z;
  d.base = a.w;
  d.nq = b.x;
  d.cu0 = b.y;
  d.P = b.z;
  d.slot = b.w;
  return d;
}

struct Cursor {
  int i, h, s;  // decode sequence, kv head, stage within the (sequence, kv head) range
  DecSeq d;
};

// cursor at global stage g: the last decode sequence whose range starts at or before g
__device__ __forceinline__ Cursor locate(const AttnParams& p, int g, int ndec) {
  int lo = 0, hi = ndec - 1, i = 0;
  while (lo <= hi) {
    const int mid = (lo + hi) >> 1;
    if (p.dec_seqs[mid].base <= g) {
      i = mid;
      lo = mid + 1;
    } else {
      hi = mid - 1;
    }
  }
  Cursor c;
  c.i = i;
  c.d = load_seq(p, i);
  const int off = g - c.d.base;
  c.h = off / c.d.st;
  c.s = off - c.h * c.d.st;
  return c;
}

__device__ __forceinline__ void advance(const AttnParams& p, Cursor& c, int ndec) {
  if (++c.s < c.d.st) return;
  c.s = 0;
  if (++c.h < p.Hkv) return;
  c.h = 0;
  if (++c.i < ndec) c.d = load_seq(p, c.i);
}

template <int D>
__device__ __forceinline__ void decode_rows(const AttnParams& p, const Cursor& c, int g,
                                            int t4, uint32_t (&qa)[D / 16][4],
                                            int (&lim)[2]) {
  const int R = c.d.nq * p.G;
  const __half* rows[2];
  bool ok[2];
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int r = g + 8 * hr;
    ok[hr] = r < R;
    const int pos = ok[hr] ? r / p.G : 0;
    const int gg = ok[hr] ? r % p.G : 0;
    rows[hr] = p.q + (int64_t)(c.d.cu0 + pos) * p.q_stride + (int64_t)(c.h * p.G + gg) * D;
    lim[hr] = ok[hr] ? (int)min64((int64_t)c.d.P + pos, INT32_MAX) : -1;
  }
  load_q_frags<D>(qa, rows[0], rows[1], ok[0], ok[1], t4);
}

// End of this warp's piece of the (sequence, kv head) range under cursor c: write the
// piece's partial (or the final output if the range is a single piece) and, if this
// warp finished the range last, merge all pieces into the output.
template <int D>
__device__ void flush_piece(const AttnParams& p, const Cursor& c, int gw, int W,
                            float (&m_run)[2], float (&l_run)[2], float (&o)[D / 8][4],
                            int lane) {
  constexpr int DN = D / 8;
  constexpr int V = D / 32;
  const int g = lane >> 2, t4 = lane & 3;
  const int R = c.d.nq * p.G;
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    l_run[hr] += __shfl_xor_sync(0xffffffffu, l_run[hr], 1);
    l_run[hr] += __shfl_xor_sync(0xffffffffu, l_run[hr], 2);
  }
  const int seg0 = c.d.base + c.h * c.d.st;
  const int first_w = seg0 / W;
  const int pieces = (seg0 + c.d.st - 1) / W - first_w + 1;
  if (pieces == 1) {
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int r = g + 8 * hr;
      if (r >= R) continue;
      const float inv = l_run[hr] > 0.f ? 1.f / l_run[hr] : 0.f;
      __half* orow = p.out + ((int64_t)(c.d.cu0 + r / p.G) * p.Hq + c.h * p.G + r % p.G) * D;
#pragma unroll
      for (int d = 0; d < DN; ++d)
        *reinterpret_cast<__half2*>(orow + d * 8 + 2 * t4) =
            __floats2half2_rn(o[d][2 * hr] * inv, o[d][2 * hr + 1] * inv);
    }
    return;
  }
  const int piece = gw - first_w;
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int r = g + 8 * hr;
    if (r >= R) continue;
    const int64_t prow =
        ((int64_t)(c.d.slot + r / p.G) * p.Hq + c.h * p.G + r % p.G) * p.max_splits + piece;
    const bool live = l_run[hr] > 0.f;
#pragma unroll
    for (int d = 0; d < DN; ++d)
      *reinterpret_cast<float2*>(p.part_o + prow * D + d * 8 + 2 * t4) =
          live ? make_float2(o[d][2 * hr], o[d][2 * hr + 1]) : make_float2(0.f, 0.f);
    if (t4 == 0) {
      p.part_m[prow] = live ? m_run[hr] * kLn2 : kNegLarge;
      p.part_l[prow] = l_run[hr];
    }
  }
  __threadfence();
  __syncwarp();
  int done = 0;
  if (lane == 0) done = atomicAdd(&p.seg_done[c.i * p.Hkv + c.h], 1);
  done = __shfl_sync(0xffffffffu, done, 0);
  if (done != pieces - 1) return;
  __threadfence();
  // every (row, piece) m and l in one round when they fit the warp (lane = row * pieces +
  // piece); otherwise row by row
  const bool packed = R * pieces <= 32;
  float lp_all = 0.f, mp_all = -INFINITY;
  if (packed && lane < R * pieces) {
    const int rr = lane / pieces, qq = lane - rr * pieces;
    const int64_t prow =
        ((int64_t)(c.d.slot + rr / p.G) * p.Hq + c.h * p.G + rr % p.G) * p.max_splits + qq;
    lp_all = __ldcg(p.part_l + prow);
    mp_all = __ldcg(p.part_m + prow);
  }
  for (int r = 0; r < R; ++r) {
    const int64_t prow0 =
        ((int64_t)(c.d.slot + r / p.G) * p.Hq + c.h * p.G + r % p.G) * p.max_splits;
    float lp = 0.f, mp = -INFINITY;
    if (packed) {
      const int src = r * pieces + (lane < pieces ? lane : 0);
      lp = __shfl_sync(0xffffffffu, lp_all, src);
      mp = __shfl_sync(0xffffffffu, mp_all, src);
      if (lane >= pieces) lp = 0.f;
      if (!(lp > 0.f)) mp = -INFINITY;
    } else if (lane < pieces) {
      lp = __ldcg(p.part_l + prow0 + lane);
      if (lp > 0.f) mp = __ldcg(p.part_m + prow0 + lane);
    }
    const float M = warp_max(mp);
    const float w = lp > 0.f ? ex2((mp - M) * kLog2e) : 0.f;
    const float L = warp_sum(w * lp);
    float acc[V];
#pragma unroll
    for (int v = 0; v < V; ++v) acc[v] = 0.f;
#pragma unroll 4
    for (int q = 0; q < pieces; ++q) {
      const float wq = __shfl_sync(0xffffffffu, w, q);
      if (wq > 0.f) {
        const float* src = p.part_o + (prow0 + q) * D + lane * V;
        if constexpr (V == 4) {
          const float4 x = __ldcg(reinterpret_cast<const float4*>(src));
          acc[0] += wq * x.x;
          acc[1] += wq * x.y;
          acc[2] += wq * x.z;
          acc[3] += wq * x.w;
        } else {
          const float2 x = __ldcg(reinterpret_cast<const float2*>(src));
          acc[0] += wq * x.x;
          acc[1] += wq * x.y;
        }
      }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    __half* orow = p.out + ((int64_t)(c.d.cu0 + r / p.G) * p.Hq + c.h * p.G + r % p.G) * D +
                   lane * V;
#pragma unroll
    for (int v = 0; v < V; v += 2)
      *reinterpret_cast<__half2*>(orow + v) = __floats2half2_rn(acc[v] * inv, acc[v + 1] * inv);
  }
}

template <int D, int NS>
__device__ void decode_phase(const AttnParams& p, unsigned char* wsm, int gw, int lane,
                             bool& bad) {
  constexpr int DN = D / 8;
  const int ndec = p.counts[kCntDecSeqs];
  const int total = p.counts[kCntStages];
  const int W = p.counts[kCntW];
  if (ndec == 0 || W <= 0) return;
  const int64_t g0 = (int64_t)gw * W;
  if (g0 >= total) return;
  const int nst = (int)(min64(total, g0 + W) - g0);
  __half* rK = reinterpret_cast<__half*>(wsm);
  __half* rV = rK + NS * 16 * D;
  uint8_t* rValid = reinterpret_cast<uint8_t*>(rV + NS * 16 * D);

  // pc: the next stage to issue; la_off: its row offsets, looked up one iteration
  // ahead so the block-table latency hides behind the current stage
  Cursor pc = locate(p, (int)g0, ndec);
  Cursor cc = pc;
  int64_t la_off = stage_row_offset(p, pc.d.b, pc.h, pc.s * 16, pc.d.n, lane, bad);
#pragma unroll
  for (int k = 0; k < NS - 1; ++k) {
    if (k < nst) {
      warp_copy16<D>(p, la_off, rK + k * 16 * D, rV + k * 16 * D, rValid + k * 16, lane);
      advance(p, pc, ndec);
      if (k + 1 < nst)
        la_off = stage_row_offset(p, pc.d.b, pc.h, pc.s * 16, pc.d.n, lane, bad);
    }
    cp_async_commit();
  }
  const int g = lane >> 2, t4 = lane & 3;
  uint32_t qa[D / 16][4];
  int lim[2];
  decode_rows<D>(p, cc, g, t4, qa, lim);
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  float o[DN][4];
#pragma unroll
  for (int i = 0; i < DN; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  for (int k = 0; k < nst; ++k) {
    cp_async_wait<NS - 2>();
    __syncwarp();
    if (k + NS - 1 < nst) {
      const int bf = (k + NS - 1) % NS;
      warp_copy16<D>(p, la_off, rK + bf * 16 * D, rV + bf * 16 * D, rValid + bf * 16, lane);
      advance(p, pc, ndec);
      if (k + NS < nst)
        la_off = stage_row_offset(p, pc.d.b, pc.h, pc.s * 16, pc.d.n, lane, bad);
    }
    cp_async_commit();
    const int bf = k % NS;
    const uint8_t* vld = rValid + bf * 16;
    const int kstage = cc.s * 16;
    float s[2][4];
#pragma unroll
    for (int e = 0; e < 4; ++e) s[0][e] = s[1][e] = 0.f;
    qk_16<D>(s[0], s[1], qa, rK + bf * 16 * D, 0, lane);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int kk = nt * 8 + 2 * t4 + (e & 1);
        const bool ok = vld[kk] && (kstage + kk <= lim[e >> 1]);
        s[nt][e] = ok ? s[nt][e] * p.scale_log2 : -INFINITY;
      }
    softmax_16<DN>(s, m_run, l_run, o);
    uint32_t pa[4] = {pack_half2(s[0][0], s[0][1]), pack_half2(s[0][2], s[0][3]),
                      pack_half2(s[1][0], s[1][1]), pack_half2(s[1][2], s[1][3])};
    pv_16<D>(o, pa, rV + bf * 16 * D, 0, lane);

    const bool seg_last = cc.s == cc.d.st - 1;
    if (seg_last || k == nst - 1) {
      flush_piece<D>(p, cc, gw, W, m_run, l_run, o, lane);
      m_run[0] = m_run[1] = -INFINITY;
      l_run[0] = l_run[1] = 0.f;
#pragma unroll
      for (int i = 0; i < DN; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    }
    advance(p, cc, ndec);
    if (seg_last && k < nst - 1) decode_rows<D>(p, cc, g, t4, qa, lim);
  }
  cp_async_wait<0>();
  __syncwarp();
}

// barrier of the 4 warps that work on a prefill tile (named barrier 1, 128 threads)
__device__ __forceinline__ void tile_sync() {
  asm volatile("bar.sync 1, 128;\n" ::: "memory");
}

// ----------------------------------------------------------------------------------
// Prefill tile (phase 2 of the persistent kernel): one tile of query positions of one
// sequence for one kv head; warp w owns 16 rows = (16 / G) positions x G query heads;
// all warps stream the same 64-key stages up to the tile's causal limit.
// ----------------------------------------------------------------------------------
template <int D, int NSTAGE>
__device__ void prefill_tile(const AttnParams& p, unsigned char* smem, int item_idx, int h,
                             bool& bad) {
  constexpr int SK = kStageKeys;
  constexpr int DN = D / 8;
  __half* sK = reinterpret_cast<__half*>(smem);
  __half* sV = sK + NSTAGE * SK * D;
  uint8_t* sValid = reinterpret_cast<uint8_t*>(sV + NSTAGE * SK * D);

  const PrefillItem it = p.pre_items[item_idx];
  const int b = it.b;
  const int cu0 = p.cu[b];
  const int P = p.past[b];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int ppw = 16 / p.G;
  const int wpos0 = warp * ppw;
  const int wn = (int)max64(0, min64(ppw, it.nq - wpos0));
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

#pragma unroll
  for (int s = 0; s < NSTAGE - 1; ++s) {
    if (s < nst)
      load_stage<D>(p, b, h, s * SK, kend, sK + s * SK * D, sV + s * SK * D, sValid + s * SK,
                    bad);
    cp_async_commit();
  }
  for (int i = 0; i < nst; ++i) {
    cp_async_wait<NSTAGE - 2>();
    tile_sync();
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
    const __half* Vt = sV + bf * SK * D;
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
      pv_16<D>(o, pa, Vt, sub * 16, lane);
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
}


// ----------------------------------------------------------------------------------
// Tensor-core prefill (head size 128), warp-specialised. A tile is 128 rows =
// (128 / G) query positions x G query heads of one sequence and kv head, streamed
// against 128-key blocks:
//   warps 5 and 6 (loaders): the Q tile and the K boxes (warp 5) and the V boxes
//            (warp 6) of each block by TMA, straight from the paged cache into
//            128-byte-swizzled shared memory. A box is R consecutive keys of one cache
//            block (R = the largest power of two <= 128 dividing the block size) and is
//            issued by one lane. Value rows of keys that are unmapped or past the tile's
//            last visible key are zero-filled with cp.async instead, so that masked
//            columns meet zeros in P V. K (2 stages) and V (3 stages) are released
//            separately: K_{j+2} streams in once S_j is computed, V_{j+3} once
//            O += P_j V_j is. Warp 5 also claims the tiles from the planner's counter and
//            publishes them in a 4-entry ring that every other role reads in order; there
//            is no block-wide barrier between tiles, so a tile's epilogue overlaps the next
//            tile's loads and S = Q K^T (the Q buffer is released by a commit after the
//            last S of a tile).
//   warp 4 (lane 0) and warp 7 (lane 0): the two tcgen05.mma issuers, S_j = Q K_j^T into
//            TMEM buffer G % 2 (G counts blocks across tiles) and O += P_j V_j, each
//            issued as soon as its operands are ready.
//   warps 0-3 (softmax): thread r reads row r of S_j from TMEM, masks it by key
//            validity (block table entries looked up by the warp itself) and causality,
//            keeps a running max that is raised only when exceeded by more than 2^8
//            (then O and l are rescaled), writes P_j (fp16) to TMEM, and finally
//            normalises O.
// TMEM: S0 columns 0..127, S1 128..255, O 256..383, P 448..511. Each role waits every
// phase of the barriers it consumes in order, and no producer can run two phases ahead of
// a consumer, so parity waits never alias.
// ----------------------------------------------------------------------------------
struct TcMaps {     // TMA descriptors (kernel parameters)
  CUtensorMap q;    // query [tokens][Hq][128], box 64 x G x 128/G
  CUtensorMap k;    // key cache [blocks * block_size][Hkv][128], box 64 x 1 x R
  CUtensorMap v;    // value cache, same geometry
};
struct TcLayout {  // byte offsets from a 1024-byte-aligned base
  static constexpr uint32_t kQ = 0;               // 2 x [128][64] fp16 sub-tiles
  static constexpr uint32_t kK = 32768;           // kKStages x 32 KB
  static constexpr uint32_t kV = kK + 65536;      // kVStages x 32 KB
  static constexpr uint32_t kBars = kV + 98304;   // mbarriers (see TcBar)
  static constexpr uint32_t kTmem = kBars + 256;  // TMEM base address
  static constexpr uint32_t kTile = kTmem + 4;    // ring of claimed tile indices (4)
  static constexpr uint32_t kAbort = kTile + 16;  // set when a bounded wait gives up
  static constexpr uint32_t kEnd = kAbort + 8;
};
enum TcBar {  // mbarrier slots
  kBarQFull = 0,     // count 1 + tx: Q boxes landed
  kBarKFull0 = 1,    // + stage (2), count 1 + tx: K boxes landed
  kBarVFull0 = 3,    // + stage (3), count 32 + tx: V boxes and zero-filled rows landed
  kBarKEmpty0 = 6,   // + stage (2), count 1: the S = Q K^T that read the stage completed
  kBarVEmpty0 = 8,   // + stage (3), count 1: the O += P V that read the stage completed
  kBarSFull0 = 11,   // + buffer, count 1: S_j in TMEM
  kBarPFull = 13,    // count 4 (one per softmax warp): softmax wrote P_j to TMEM
  kBarODone = 14,    // count 1: O += P_j V_j completed
  kBarDrain = 15,    // count 1: S = Q K^T MMAs in flight when a wait gave up
  kBarSEmpty0 = 16,  // + buffer, count 4: softmax has read S_j out of the buffer
  kBarDrainPv = 18,  // count 1: O += P V MMAs in flight when a wait gave up
  kBarQEmpty = 19,   // count 1: every S = Q K^T of a tile completed (Q buffer free)
  kBarTileFull0 = 20,   // + slot (4), count 1: tile ring entry published (key loader)
  kBarTileEmpty0 = 24,  // + slot (4), count 7: entry read by the other roles
  kNumBars = 28
};
static_assert(kNumBars * 8 <= 256, "mbarrier slots");
// TMEM columns: S_j in buffer j % 2, the O accumulator, and P_j as fp16 pairs (two keys
// per 32-bit column); the row sums l stay in the softmax threads' registers
constexpr uint32_t kTmS = 0, kTmO = 256, kTmP = 448;
constexpr int kKStages = 2;        // K ring depth
constexpr int kVStages = 3;        // V ring depth: V_j streams in once O += P_{j-3} V_{j-3} is done
constexpr uint32_t kTcWaitTries = 1u << 22;   // default bound of each wait (polls)
constexpr int kTcThreads = 256;
constexpr int kMmaThread = 128;    // lane 0 of warp 4: S = Q K^T
constexpr int kPvThread = 224;     // lane 0 of warp 7: O += P V
constexpr int kKLoaderWarp = 5;
constexpr int kVLoaderWarp = 6;
constexpr float kTcRescale = 8.f;  // log2 of the largest weight a stale max may give

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
// arrive when every cp.async this thread issued so far has landed (count not raised)
__device__ __forceinline__ void mbar_arrive_cp_async(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(smem_u32(bar))
               : "memory");
}
// polls a wait of this kernel may take before it gives up
__device__ __forceinline__ uint32_t tc_tries(const AttnParams& p) {
  return p.wait_tries ? p.wait_tries : kTcWaitTries;
}
// bounded wait that also gives up when another thread of the CTA already did
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                        uint32_t tries) {
  const uint32_t addr = smem_u32(bar);
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

struct TcTile {
  int b, h, q0, nq, cu0, P, kend, nblk, PT;
};

__device__ __forceinline__ TcTile tc_tile(const AttnParams& p, int t) {
  const PrefillItem it = p.pre_items[t / p.Hkv];
  TcTile d;
  d.b = it.b;
  d.h = t % p.Hkv;
  d.q0 = it.q0;
  d.nq = it.nq;
  d.cu0 = p.cu[it.b];
  d.P = p.past[it.b];
  d.kend = seq_keys(p, d.P, it.q0 + it.nq);
  d.nblk = (d.kend + 127) / 128;
  d.PT = 128 / p.G;
  return d;
}

// Box `lane` of key block j: keys [key0, key0 + R) of one cache block, with its first
// row in the cache when the block-table entry is valid.
struct TcBox {
  int key0, row;
  bool mapped;
};
__device__ __forceinline__ TcBox tc_box(const AttnParams& p, const TcTile& t, int j, int lane,
                                        bool& unmapped) {
  const int R = p.tc_rows;
  TcBox x;
  x.key0 = j * 128 + lane * R;
  x.row = 0;
  x.mapped = false;
  if (lane < 128 / R && x.key0 < t.kend) {
    const int col = p.bs_shift >= 0 ? x.key0 >> p.bs_shift : x.key0 / p.BS;
    const int blk = __ldg(&p.block_table[(int64_t)t.b * p.MB + col]);
    if (blk >= 0 && (int64_t)blk < p.NB) {
      x.mapped = true;
      x.row = blk * p.BS + (x.key0 - col * p.BS);
    } else {
      unmapped = true;
    }
  }
  return x;
}

// Key loader warp: Q tile, then the K boxes of every block (keys past the visible range
// and unmapped boxes are left as they are: the softmax masks them).
__device__ void tc_load_k(const AttnParams& p, const TcMaps& maps, unsigned char* sm,
                          const TcTile& t, uint32_t q_n, uint32_t (&k_use)[kKStages], bool& bad) {
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + TcLayout::kBars);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + TcLayout::kAbort);
  const int lane = threadIdx.x & 31;
  const int R = p.tc_rows;
  // testing hook: the CTA's first K box is announced but never copied, so the MMA's wait
  // for it gives up (no copy or MMA of that block is in flight when it does)
  const bool withhold = p.withhold_copy && k_use[0] == 0;
  if (q_n > 0 && !__all_sync(0xffffffffu, tc_wait(bars + kBarQEmpty, (q_n - 1) & 1u, abort,
                                                     tc_tries(p))))
    return;
  if (lane == 0) {
    // rows past the tile's positions hold other tokens (or zeros past the last token)
    // and are never written out
    unsigned char* Qs = sm + TcLayout::kQ;
    tc::mbar_arrive_expect_tx(bars + kBarQFull, (uint32_t)(t.PT * p.G) * 256u);
    tc::tma_load_3d(Qs, &maps.q, 0, t.h * p.G, t.cu0 + t.q0, bars + kBarQFull);
    tc::tma_load_3d(Qs + 16384, &maps.q, 64, t.h * p.G, t.cu0 + t.q0, bars + kBarQFull);
  }
  for (int j = 0, s = 0; j < t.nblk; ++j, s = s + 1 == kKStages ? 0 : s + 1) {
    const TcBox x = tc_box(p, t, j, lane, bad);
    const bool ok = k_use[s] == 0 || tc_wait(bars + kBarKEmpty0 + s, (k_use[s] - 1) & 1u, abort, tc_tries(p));
    if (!__all_sync(0xffffffffu, ok)) return;
    ++k_use[s];
    const uint32_t bits = __ballot_sync(0xffffffffu, x.mapped);
    if (lane == 0)
      tc::mbar_arrive_expect_tx(bars + kBarKFull0 + s, (uint32_t)__popc(bits) * R * 256u);
    __syncwarp();
    unsigned char* Ks = sm + TcLayout::kK + s * 32768;
    if (x.mapped && !(withhold && j == 0)) {
      tc::tma_load_3d(Ks + lane * R * 128, &maps.k, 0, t.h, x.row, bars + kBarKFull0 + s);
      tc::tma_load_3d(Ks + 16384 + lane * R * 128, &maps.k, 64, t.h, x.row,
                      bars + kBarKFull0 + s);
    }
  }
}

// Value loader warp: whole boxes by TMA, the rest of the rows through zero-filling cp.async
// (rows of unmapped or not-yet-visible keys must be zeros for P V).
__device__ void tc_load_v(const AttnParams& p, const TcMaps& maps, unsigned char* sm,
                          const TcTile& t, uint32_t (&v_use)[kVStages]) {
  constexpr int D = 128;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + TcLayout::kBars);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + TcLayout::kAbort);
  const int lane = threadIdx.x & 31;
  const int R = p.tc_rows;
  bool unmapped = false;   // reported by the key loader
  for (int j = 0, s = 0; j < t.nblk; ++j, s = s + 1 == kVStages ? 0 : s + 1) {
    const TcBox x = tc_box(p, t, j, lane, unmapped);
    const bool whole = x.mapped && x.key0 + R <= t.kend;
    const bool ok = v_use[s] == 0 || tc_wait(bars + kBarVEmpty0 + s, (v_use[s] - 1) & 1u, abort, tc_tries(p));
    if (!__all_sync(0xffffffffu, ok)) return;
    ++v_use[s];
    const uint32_t bits = __ballot_sync(0xffffffffu, whole);
    if (lane == 0)
      tc::mbar_expect_tx(bars + kBarVFull0 + s, (uint32_t)__popc(bits) * R * 256u);
    __syncwarp();
    unsigned char* Vs = sm + TcLayout::kV + s * 32768;
    if (whole) {
      tc::tma_load_3d(Vs + lane * R * 128, &maps.v, 0, t.h, x.row, bars + kBarVFull0 + s);
      tc::tma_load_3d(Vs + 16384 + lane * R * 128, &maps.v, 64, t.h, x.row,
                      bars + kBarVFull0 + s);
    }
    uint32_t rest = __ballot_sync(0xffffffffu, lane < 128 / R && !whole);
    while (rest) {
      const int i = __ffs(rest) - 1;
      rest &= rest - 1;
      const int rowi = __shfl_sync(0xffffffffu, x.row, i);
      const int mi = __shfl_sync(0xffffffffu, x.mapped ? 1 : 0, i);
      const int k0 = j * 128 + i * R;
      for (int idx = lane; idx < R * 16; idx += 32) {
        const int rr = idx >> 4, c = idx & 15;
        const bool live = mi && k0 + rr < t.kend;
        const __half* src =
            live ? p.vc + (((int64_t)(rowi + rr) * p.Hkv + t.h) * D + c * 8) : p.vc;
        cp_async_16(Vs + (c >> 3) * 16384 + tc::sw128(i * R + rr, c & 7), src, live ? 16 : 0);
      }
    }
    mbar_arrive_cp_async(bars + kBarVFull0 + s);
  }
}

// O += P V with the A operand (P) read from TMEM
__device__ __forceinline__ void mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
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

// Two MMA issuers, each a thread that does nothing else: the cost of a tcgen05.mma is
// paid by the issuing thread, so S = Q K^T and O += P V issued from separate threads
// overlap on the tensor pipe.
//
// Warp 4, lane 0: S_jq = Q K_jq^T once K_jq landed and the softmax has read S_{jq-2} out
// of buffer jq % 2 (SEmpty phases are counted per block, across tiles, because the last
// two of a tile are never waited for).
__device__ void tc_mma_s(const AttnParams& p, unsigned char* sm, const TcTile& t,
                         uint32_t tmem, uint32_t q_use, uint32_t (&k_use)[kKStages],
                         uint32_t& g_blk) {
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + TcLayout::kBars);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + TcLayout::kAbort);
  const uint32_t idesc_qk = tc::idesc_f16(128, 128, false, false);
  const uint32_t qa = smem_u32(sm + TcLayout::kQ);
  if (!tc_wait(bars + kBarQFull, q_use & 1u, abort, tc_tries(p))) return;
  uint32_t idle = 0;
  for (int jq = 0, kq = 0; jq < t.nblk;) {
    // block G = g_blk + jq (counted across tiles) fills buffer G % 2, last filled by
    // block G - 2: phase (G - 2) / 2 of SEmpty_s
    const uint32_t G = g_blk + (uint32_t)jq;
    const int s = (int)(G & 1u);
    if ((G < 2 || tc::mbar_test(bars + kBarSEmpty0 + s, ((G >> 1) - 1u) & 1u)) &&
        tc::mbar_test(bars + kBarKFull0 + kq, k_use[kq] & 1u)) {
      ++k_use[kq];
      tc::fence_after_sync();
      const uint32_t ka = smem_u32(sm + TcLayout::kK + kq * 32768);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t koff = (uint32_t)(ks >> 2) * 16384u + (uint32_t)(ks & 3) * 32u;
        tc::mma_f16(tmem + kTmS + s * 128, tc::smem_desc(qa + koff, 16, 1024),
                    tc::smem_desc(ka + koff, 16, 1024), idesc_qk, ks > 0 ? 1u : 0u);
      }
      tc::commit(bars + kBarSFull0 + s);
      tc::commit(bars + kBarKEmpty0 + kq);
      ++jq;
      kq = kq + 1 == kKStages ? 0 : kq + 1;
      idle = 0;
    } else if (++idle >= tc_tries(p) || ((idle & 255u) == 0 && *abort)) {
      *abort = 1;
      return;
    }
  }
  g_blk += (uint32_t)t.nblk;
  // the next tile's Q may land once every S of this one has completed
  tc::commit(bars + kBarQEmpty);
}

// Warp 7, lane 0: O += P_jp V_jp once the softmax has written P_jp to TMEM and V_jp landed.
__device__ void tc_mma_pv(const AttnParams& p, unsigned char* sm, const TcTile& t,
                          uint32_t tmem, uint32_t (&v_use)[kVStages], uint32_t& blk_use) {
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + TcLayout::kBars);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + TcLayout::kAbort);
  const uint32_t idesc_pv = tc::idesc_f16(128, 128, false, true);
  uint32_t idle = 0;
  for (int jp = 0, vq = 0; jp < t.nblk;) {
    const int s = vq;
    if (tc::mbar_test(bars + kBarPFull, (blk_use + jp) & 1u) &&
        tc::mbar_test(bars + kBarVFull0 + s, v_use[s] & 1u)) {
      ++v_use[s];
      tc::fence_async_shared();   // zero-filled value rows were written by cp.async
      tc::fence_after_sync();
      const uint32_t va = smem_u32(sm + TcLayout::kV + s * 32768);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t acc = (jp > 0 || ks > 0) ? 1u : 0u;
        mma_f16_tmem_a(tmem + kTmO, tmem + kTmP + (uint32_t)ks * 8u,
                       tc::smem_desc(va + (uint32_t)ks * 2048u, 16384, 1024), idesc_pv, acc);
      }
      tc::commit(bars + kBarODone);
      tc::commit(bars + kBarVEmpty0 + s);
      ++jp;
      vq = vq + 1 == kVStages ? 0 : vq + 1;
      idle = 0;
    } else if (++idle >= tc_tries(p) || ((idle & 255u) == 0 && *abort)) {
      *abort = 1;
      return;
    }
  }
  blk_use += t.nblk;
}

__device__ __forceinline__ float fmax3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float fmin3f(float a, float b, float c) {
  float r;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Warps 0-3: softmax of row threadIdx.x and its normalised output. The row max is taken
// over the raw scores (the minimum when the scale is negative), so that each weight is
// one fused multiply-add and an exp2: p = 2^(s * scale * log2 e - m).
__device__ void tc_softmax(const AttnParams& p, unsigned char* sm, const TcTile& t,
                           uint32_t tmem, uint32_t (&s_use)[2], uint32_t& blk_use) {
  constexpr int D = 128;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + TcLayout::kBars);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + TcLayout::kAbort);
  const int r = threadIdx.x, lane = r & 31;
  const int pl = r / p.G;
  const bool rvalid = r < t.PT * p.G && pl < t.nq;
  const int lim = rvalid ? (int)min64((int64_t)t.P + t.q0 + pl, INT32_MAX) : -1;
  const uint32_t lane_taddr = tmem + ((uint32_t)(r & ~31) << 16);
  const float sl2 = p.scale_log2;
  const bool pos_scale = sl2 >= 0.f;
  const float hide = pos_scale ? -INFINITY : INFINITY;   // masked raw score
  float m_used = -INFINITY;
  float l_run = 0.f;   // row sum of the weights, relative to m_used like O
  bool ok = true;
  // block-table entry of the cache block holding keys [kbase + 4 lane, + 4) of block j
  auto lookup = [&](int j) -> int {
    const int key0 = j * 128 + 4 * lane;
    if (key0 >= t.kend) return -1;
    const int col = p.bs_shift >= 0 ? key0 >> p.bs_shift : key0 / p.BS;
    return __ldg(&p.block_table[(int64_t)t.b * p.MB + col]);
  };
  int blk_next = lookup(0);
  for (int j = 0; j < t.nblk && ok; ++j) {
    const int s = (int)((blk_use + (uint32_t)j) & 1u);
    const int kbase = j * 128;
    // key validity of block j: lane covers keys [kbase + 4 lane, + 4), which lie in one
    // cache block because the block size is a multiple of 8; key c of the block is bit
    // c / 4 of words[c % 4]
    const int key0 = kbase + 4 * lane;
    const bool page = blk_next >= 0 && (int64_t)blk_next < p.NB;
    if (j + 1 < t.nblk) blk_next = lookup(j + 1);
    uint32_t words[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) words[i] = __ballot_sync(0xffffffffu, page && key0 + i < t.kend);
    ok = tc_wait(bars + kBarSFull0 + s, s_use[s] & 1u, abort, tc_tries(p));
    ++s_use[s];
    ok = __all_sync(0xffffffffu, ok);   // TMEM loads below are warp-collective
    if (!ok) break;
    tc::fence_after_sync();
    const int cut = lim - kbase + 1;  // columns below cut are causally visible to this row
    const bool full = (words[0] & words[1] & words[2] & words[3]) == 0xffffffffu && cut >= 128;
    // the whole row of S_j in one TMEM round trip; the buffer is then free for S_{j+2}
    float v[128];
    {
      float (*v32)[32] = reinterpret_cast<float (*)[32]>(v);
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) tc::tmem_ld32(lane_taddr + kTmS + s * 128 + ch * 32, v32[ch]);
      tc::tmem_wait_ld();
    }
    tc::fence_before_sync();
    __syncwarp();   // one arrival per warp: 128 arrivals on one word would serialise
    if (lane == 0) mbar_arrive(bars + kBarSEmpty0 + s);
    if (!__all_sync(0xffffffffu, full)) {
#pragma unroll
      for (int c = 0; c < 128; ++c) {
        const bool vis = c < cut && ((words[c & 3] >> (c >> 2)) & 1u);
        v[c] = vis ? v[c] : hide;
      }
    }
    float e4[4];
    if (pos_scale) {
      e4[0] = fmaxf(v[0], v[1]); e4[1] = fmaxf(v[2], v[3]);
      e4[2] = fmaxf(v[4], v[5]); e4[3] = fmaxf(v[6], v[7]);
#pragma unroll
      for (int c = 8; c < 128; c += 8) {
        e4[0] = fmax3f(e4[0], v[c], v[c + 1]); e4[1] = fmax3f(e4[1], v[c + 2], v[c + 3]);
        e4[2] = fmax3f(e4[2], v[c + 4], v[c + 5]); e4[3] = fmax3f(e4[3], v[c + 6], v[c + 7]);
      }
      e4[0] = fmax3f(e4[0], e4[1], fmaxf(e4[2], e4[3]));
    } else {
      e4[0] = fminf(v[0], v[1]); e4[1] = fminf(v[2], v[3]);
      e4[2] = fminf(v[4], v[5]); e4[3] = fminf(v[6], v[7]);
#pragma unroll
      for (int c = 8; c < 128; c += 8) {
        e4[0] = fmin3f(e4[0], v[c], v[c + 1]); e4[1] = fmin3f(e4[1], v[c + 2], v[c + 3]);
        e4[2] = fmin3f(e4[2], v[c + 4], v[c + 5]); e4[3] = fmin3f(e4[3], v[c + 6], v[c + 7]);
      }
      e4[0] = fmin3f(e4[0], e4[1], fminf(e4[2], e4[3]));
    }
    const float mx = e4[0] * sl2;   // -inf when nothing in the block is visible
    const bool first = m_used == -INFINITY;
    const bool raise = (first && mx != -INFINITY) || (!first && mx > m_used + kTcRescale);
    const float alpha = raise && !first ? ex2(m_used - mx) : 1.f;
    if (raise) m_used = mx;
    const float nbase = m_used == -INFINITY ? 0.f : -m_used;
    float pw[64];   // P_j row as fp16 pairs (bit patterns)
    // l sums the fp32 weights: four pairs of accumulators, each pair one f32x2 add
    float la[4] = {0.f, 0.f, 0.f, 0.f}, lb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c = 0; c < 128; c += 2) {
      float e0, e1;
      fma2(e0, e1, v[c], v[c + 1], sl2, nbase);
      const float p0 = ex2(e0), p1 = ex2(e1);
      add2(la[(c >> 1) & 3], lb[(c >> 1) & 3], p0, p1);
      pw[c / 2] = __uint_as_float(pack_half2(p0, p1));
    }
    l_run = l_run * alpha + (((la[0] + lb[0]) + (la[1] + lb[1])) + ((la[2] + lb[2]) + (la[3] + lb[3])));
    // O and the P columns are free once O += P_{j-1} V_{j-1} has completed
    if (j > 0) {
      ok = __all_sync(0xffffffffu, tc_wait(bars + kBarODone, (blk_use + j - 1) & 1u, abort, tc_tries(p)));
      if (!ok) break;
      tc::fence_after_sync();
      if (__any_sync(0xffffffffu, alpha != 1.f)) {   // warp-collective TMEM rescale of O
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          float o[32];
          tc::tmem_ld32(lane_taddr + kTmO + ch * 32, o);
          tc::tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] *= alpha;
          tc::tmem_st32(lane_taddr + kTmO + ch * 32, o);
        }
      }
    }
    {
      float (*p32)[32] = reinterpret_cast<float (*)[32]>(pw);
      tc::tmem_st32(lane_taddr + kTmP, p32[0]);
      tc::tmem_st32(lane_taddr + kTmP + 32, p32[1]);
    }
    tc::tmem_wait_st();
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + kBarPFull);
  }
  if (ok) {
    ok = __all_sync(0xffffffffu,
                    tc_wait(bars + kBarODone, (blk_use + t.nblk - 1) & 1u, abort, tc_tries(p)));
    if (ok) {
      tc::fence_after_sync();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      __half* orow = p.out + (int64_t)(t.cu0 + t.q0 + pl) * p.Hq * D +
                     (int64_t)(t.h * p.G + r % p.G) * D;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        float o[32];
        tc::tmem_ld32(lane_taddr + kTmO + ch * 32, o);
        tc::tmem_wait_ld();
        if (rvalid) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<uint4*>(orow + ch * 32 + q * 8) =
                make_uint4(pack_half2(o[q * 8 + 0] * inv, o[q * 8 + 1] * inv),
                           pack_half2(o[q * 8 + 2] * inv, o[q * 8 + 3] * inv),
                           pack_half2(o[q * 8 + 4] * inv, o[q * 8 + 5] * inv),
                           pack_half2(o[q * 8 + 6] * inv, o[q * 8 + 7] * inv));
        }
      }
    }
  }
  blk_use += t.nblk;
}

// Tiles from the planner's counter through the tile ring; barriers and 512 TMEM columns
// held throughout.
__device__ void prefill_phase_tc(const AttnParams& p, const TcMaps& maps, unsigned char* sm,
                                 bool& bad) {
  const int ntiles = p.counts[kCntTiles];
  if (ntiles == 0) return;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + TcLayout::kBars);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + TcLayout::kTmem);
  volatile int* tile = reinterpret_cast<volatile int*>(sm + TcLayout::kTile);   // [4]
  volatile int* abort = reinterpret_cast<volatile int*>(sm + TcLayout::kAbort);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    tc::mbar_init(bars + kBarQFull, 1);
    for (int s = 0; s < kKStages; ++s) {
      tc::mbar_init(bars + kBarKFull0 + s, 1);
      tc::mbar_init(bars + kBarKEmpty0 + s, 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      tc::mbar_init(bars + kBarVFull0 + s, 32);
      tc::mbar_init(bars + kBarVEmpty0 + s, 1);
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(bars + kBarSFull0 + s, 1);
      tc::mbar_init(bars + kBarSEmpty0 + s, 4);
    }
    tc::mbar_init(bars + kBarPFull, 4);
    tc::mbar_init(bars + kBarODone, 1);
    tc::mbar_init(bars + kBarDrain, 1);
    tc::mbar_init(bars + kBarDrainPv, 1);
    tc::mbar_init(bars + kBarQEmpty, 1);
    for (int i = 0; i < 4; ++i) {
      tc::mbar_init(bars + kBarTileFull0 + i, 1);
      tc::mbar_init(bars + kBarTileEmpty0 + i, 7);
    }
    tc::mbar_init_fence();
    *abort = 0;
  }
  if (warp == kKLoaderWarp && lane == 0) {
    tc::tma_prefetch_desc(&maps.q);
    tc::tma_prefetch_desc(&maps.k);
  }
  if (warp == kVLoaderWarp && lane == 0) tc::tma_prefetch_desc(&maps.v);
  if (warp == 0) {
    tc::tmem_alloc(tslot, 512);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;
  // per-role phase counters (each role waits every phase it depends on, in order)
  uint32_t k_use[kKStages] = {}, v_use[kVStages] = {}, s_use[2] = {0u, 0u};
  uint32_t g_blk = 0u;   // S issuer: blocks of earlier tiles
  uint32_t q_use = 0u, blk_use = 0u;
  bool mma_aborted = false;
  // Tiles flow through a 4-entry ring: the key loader claims each from the planner's
  // counter and publishes it (-1 = no more); every other role reads the entries in order
  // and releases each at once. No block-wide barrier between tiles: a tile's epilogue and
  // the next tile's loads and S = Q K^T overlap.
  const bool producer = warp == kKLoaderWarp;
  const bool consumer = tid < 128 || tid == kMmaThread || tid == kPvThread || warp == kVLoaderWarp;
  for (uint32_t n = 0; producer || consumer; ++n) {
    const uint32_t slot = n & 3u, ph = (n >> 2) & 1u;
    int ti = -1;
    if (producer) {
      if (lane == 0) ti = atomicAdd(&p.counts[kCntTileNext], 1);
      ti = __shfl_sync(0xffffffffu, ti, 0);
      if (ti >= ntiles || *abort) ti = -1;
      if (n >= 4 && !__all_sync(0xffffffffu, tc_wait(bars + kBarTileEmpty0 + slot, ph ^ 1u, abort,
                                                       tc_tries(p))))
        break;
      if (lane == 0) {
        tile[slot] = ti;
        mbar_arrive(bars + kBarTileFull0 + slot);
      }
    } else {
      const bool whole_warp = tid < 128 || warp == kVLoaderWarp;
      bool ok = tc_wait(bars + kBarTileFull0 + slot, ph, abort, tc_tries(p));
      if (whole_warp) ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ti = tile[slot];
      if (whole_warp) {
        __syncwarp();
        if (lane == 0) mbar_arrive(bars + kBarTileEmpty0 + slot);
      } else {
        mbar_arrive(bars + kBarTileEmpty0 + slot);
      }
    }
    if (ti < 0) break;
    const TcTile t = tc_tile(p, ti);
    if (tid < 128) {
      tc_softmax(p, sm, t, tmem, s_use, blk_use);
    } else if (tid == kMmaThread) {
      tc_mma_s(p, sm, t, tmem, q_use, k_use, g_blk);
      mma_aborted = *abort != 0;
    } else if (tid == kPvThread) {
      tc_mma_pv(p, sm, t, tmem, v_use, blk_use);
      mma_aborted = *abort != 0;
    } else if (warp == kKLoaderWarp) {
      tc_load_k(p, maps, sm, t, q_use, k_use, bad);
    } else if (warp == kVLoaderWarp) {
      tc_load_v(p, maps, sm, t, v_use);
    }
    ++q_use;
    if (*abort) break;
  }
  if (*abort) {
    // a wait gave up: let the copies and MMAs this CTA issued land before it exits
    if (tid == 0) flag_status(p.status, PKV_DEV_TIMEOUT);
    if ((tid == kMmaThread || tid == kPvThread) && mma_aborted) {
      // each issuer drains its own MMAs (a commit tracks the issuing thread's MMAs)
      uint64_t* drain = bars + (tid == kMmaThread ? kBarDrain : kBarDrainPv);
      tc::commit(drain);
      tc::mbar_wait(drain, 0, tc_tries(p));
    }
    if (warp == kKLoaderWarp && lane == 0) {
      if (q_use > 0) tc::mbar_wait(bars + kBarQFull, (q_use - 1) & 1u, tc_tries(p));
      for (int s = 0; s < kKStages; ++s)
        if (k_use[s] > 0) tc::mbar_wait(bars + kBarKFull0 + s, (k_use[s] - 1) & 1u, tc_tries(p));
    }
    if (warp == kVLoaderWarp && lane == 0) {
      for (int s = 0; s < kVStages; ++s)
        if (v_use[s] > 0) tc::mbar_wait(bars + kBarVFull0 + s, (v_use[s] - 1) & 1u, tc_tries(p));
    }
  }
  cp_async_wait<0>();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

// Persistent tensor-core prefill kernel: one CTA of 8 warps per SM, tiles from the
// planner's counter.
__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_tc_kernel(AttnParams p, const __grid_constant__ TcMaps maps) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  bool bad = false;
  prefill_phase_tc(p, maps, smem, bad);
  if (bad) flag_status(p.status, PKV_DEV_BAD_BLOCK);
}
constexpr size_t kTcSmem = TcLayout::kEnd + 1024;   // + slack for the 1024-byte alignment
static_assert(kTcSmem <= 232448, "tensor-core prefill shared memory over the limit");

// ring sizes (bytes) of the two phases; the dynamic shared memory is their maximum
template <int D, int NS>
struct DecodeRing {
  static constexpr size_t kWarpBytes =
      ((size_t)NS * 16 * D * 2 * 2 + NS * 16 + 127) / 128 * 128;
  static constexpr size_t kBytes = kWarpBytes * kWarps;
};
template <int D, int NSTAGE>
struct TileRing {
  static constexpr size_t kBytes =
      (size_t)NSTAGE * kStageKeys * D * 2 * 2 + NSTAGE * kStageKeys;
};

static_assert(kWarps >= 4, "prefill tiles need at least 4 warps");

template <int D, int NS, int NSTAGE>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) attention_kernel(AttnParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int s_tile;
  // the tensor-core prefill kernel behind this one may start as SMs free up; it reads
  // only what the prologue wrote and writes disjoint output rows
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  bool bad = false;
  decode_phase<D, NS>(p, smem + warp * DecodeRing<D, NS>::kWarpBytes,
                      blockIdx.x * kWarps + warp, lane, bad);
  __syncthreads();
  // with tensor-core prefill the tiles (and their counter) belong to prefill_tc_kernel
  const int ntiles = p.tc_prefill ? 0 : p.counts[kCntTiles];
  while (ntiles > 0) {
    if (threadIdx.x == 0) s_tile = atomicAdd(&p.counts[kCntTileNext], 1);
    __syncthreads();
    const int t = s_tile;
    __syncthreads();
    if (t >= ntiles) break;
    if (warp < 4) prefill_tile<D, NSTAGE>(p, smem, t / p.Hkv, t % p.Hkv, bad);
  }
  if (bad) flag_status(p.status, PKV_DEV_BAD_BLOCK);
}

// ----------------------------------------------------------------------------------
// Rows of one (sequence, kv head) over one key range, by a CTA of 4 warps: each warp
// takes 16 keys of every 64-key stage and the four warps' (o, m, l) are merged through
// shared memory. Serves the split mode (one split of a short sequence per CTA, partials
// for the combine kernel, or the output itself when every sequence has one split) and the
// single-pass path (whole sequences, output written directly).
// ----------------------------------------------------------------------------------
// Rows [row0, min(row0 + 16, R)) of (sequence b, kv head h): row r is query head
// h*G + r % G of token cu0 + r / G at position P + r / G, over keys [kb, ke). kDirect:
// the normalised fp16 output; else unnormalised partials of split `split` at slot
// slot_base + r / G.
template <int D, int NSTAGE, bool kDirect>
__device__ void split_rows(const AttnParams& p, unsigned char* smem, int b, int h, int cu0,
                           int P, int row0, int R, int kb, int ke, int slot_base, int split,
                           bool& bad) {
  constexpr int SK = kStageKeys;
  constexpr int DN = D / 8;
  __half* sK = reinterpret_cast<__half*>(smem);
  __half* sV = sK + NSTAGE * SK * D;
  uint8_t* sValid = reinterpret_cast<uint8_t*>(sV + NSTAGE * SK * D);
  const int nr = min(16, R - row0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;

  int lim[2];
  uint32_t qa[D / 16][4];
  {
    const __half* rows[2];
    bool ok[2];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int rl = g + 8 * hr;
      ok[hr] = rl < nr;
      const int r = row0 + rl;
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
    const int kw = warp * 16;
    const int kstage = kb + i * SK;
    if (kstage + kw < ke) {
      const uint8_t* vld = sValid + bf * SK;
      float s[2][4];
#pragma unroll
      for (int e = 0; e < 4; ++e) s[0][e] = s[1][e] = 0.f;
      qk_16<D>(s[0], s[1], qa, sK + bf * SK * D, kw, lane);
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int kk = kw + nt * 8 + 2 * t4 + (e & 1);
          const bool ok = vld[kk] && (kstage + kk <= lim[e >> 1]);
          s[nt][e] = ok ? s[nt][e] * p.scale_log2 : -INFINITY;
        }
      softmax_16<DN>(s, m_run, l_run, o);
      uint32_t pa[4] = {pack_half2(s[0][0], s[0][1]), pack_half2(s[0][2], s[0][3]),
                        pack_half2(s[1][0], s[1][1]), pack_half2(s[1][2], s[1][3])};
      pv_16<D>(o, pa, sV + bf * SK * D, kw, lane);
    }
  }
  cp_async_wait<0>();
  __syncthreads();

#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    l_run[hr] += __shfl_xor_sync(0xffffffffu, l_run[hr], 1);
    l_run[hr] += __shfl_xor_sync(0xffffffffu, l_run[hr], 2);
  }
  float* sO = reinterpret_cast<float*>(smem);  // [kTileWarps][16][D]
  float* sM = sO + kTileWarps * 16 * D;            // [kTileWarps][16]
  float* sL = sM + kTileWarps * 16;
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
  // two adjacent columns per thread
  for (int e = threadIdx.x; e < nr * D / 2; e += kTileThreads) {
    const int rl = e / (D / 2), d = 2 * (e % (D / 2));
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kTileWarps; ++w) M = fmaxf(M, sM[w * 16 + rl]);
    float num0 = 0.f, num1 = 0.f, L = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kTileWarps; ++w) {
        const float wt = ex2(sM[w * 16 + rl] - M);
        num0 += wt * sO[(w * 16 + rl) * D + d];
        num1 += wt * sO[(w * 16 + rl) * D + d + 1];
        L += wt * sL[w * 16 + rl];
      }
    }
    const int r = row0 + rl;
    const int pos = r / p.G, gg = r % p.G;
    if constexpr (kDirect) {
      const float inv = L > 0.f ? 1.f / L : 0.f;
      *reinterpret_cast<__half2*>(p.out + ((int64_t)(cu0 + pos) * p.Hq + h * p.G + gg) * D + d) =
          __floats2half2_rn(num0 * inv, num1 * inv);
    } else {
      const int64_t prow =
          ((int64_t)(slot_base + pos) * p.Hq + h * p.G + gg) * p.max_splits + split;
      *reinterpret_cast<float2*>(p.part_o + prow * D + d) =
          L > 0.f ? make_float2(num0, num1) : make_float2(0.f, 0.f);
      if (d == 0) {
        p.part_m[prow] = L > 0.f ? M * kLn2 : kNegLarge;
        p.part_l[prow] = L;
      }
    }
  }
}

// Split mode (fixed split counts): CTA = one split of one short sequence for one kv head.
// With one split per sequence the output is written here and no combine runs; otherwise
// the combine kernel merges the partials.
template <int D, int NSTAGE>
__global__ void __launch_bounds__(kTileThreads) decode_split_kernel(AttnParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int h = blockIdx.x % p.Hkv;
  const int64_t item_idx = blockIdx.x / p.Hkv;
  if (item_idx >= p.counts[kCntSplitItems]) return;
  const DecodeItem it = p.dec_items[item_idx];
  const int b = it.b;
  const int cu0 = p.cu[b];
  const int P = p.past[b];
  const int n = seq_keys(p, P, it.nq);
  const int kb = it.split * it.chunk;
  const int ke = (int)min64(n, (int64_t)kb + it.chunk);
  const int R = it.nq * p.G;
  bool bad = false;
  if (p.max_splits == 1)
    split_rows<D, NSTAGE, true>(p, smem, b, h, cu0, P, 0, R, kb, ke, 0, 0, bad);
  else
    split_rows<D, NSTAGE, false>(p, smem, b, h, cu0, P, 0, R, kb, ke, it.slot_base, it.split,
                                 bad);
  if (bad) flag_status(p.status, PKV_DEV_BAD_BLOCK);
}

// ----------------------------------------------------------------------------------
// Prologue: block 0 plans (one pass over the sequences), the other blocks run the
// ScatterKV pass. The attention kernels run after it on the same stream.
// ----------------------------------------------------------------------------------
__device__ __forceinline__ bool seq_valid(const AttnParams& p, int b, int& lo, int& hi,
                                          int& P) {
  lo = p.cu[b];
  hi = p.cu[b + 1];
  P = p.past[b];
  return lo >= 0 && hi >= lo && hi <= p.T && P >= 0;
}

// exclusive scan over the 256 threads of the block; *total gets the block sum
__device__ int block_scan(int v, int* total) {
  __shared__ int warp_tot[kPrologueThreads / 32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[w] = x;
  __syncthreads();
  if (w == 0) {
    int t = lane < kPrologueThreads / 32 ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < kPrologueThreads / 32) warp_tot[lane] = t;
  }
  __syncthreads();
  const int base = w > 0 ? warp_tot[w - 1] : 0;
  *total = warp_tot[kPrologueThreads / 32 - 1];
  __syncthreads();
  return base + x - v;
}

// Zero output rows of tokens that no valid sequence covers (nothing to do when
// all_covered); threads tid, tid + nthr, ... of the caller take the tokens.
__device__ void zero_uncovered(const AttnParams& p, bool all_covered, int tid, int nthr) {
  for (int i = tid; !all_covered && i < p.T; i += nthr) {
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

__device__ void plan_block(const AttnParams& p) {
  const int tid = threadIdx.x;
  // s_w*: extent of what was actually written. Every write condition below is monotone
  // in the scan offsets, so the written entries form a prefix of each array.
  __shared__ int s_maxst, s_bad, s_badblk, s_wdec, s_wst, s_witems, s_wslot, s_wpre;
  if (tid == 0) {
    s_maxst = 0;
    s_bad = 0;
    s_badblk = 0;
    s_wdec = s_wst = s_witems = s_wslot = s_wpre = 0;
  }
  __syncthreads();
  const bool sk = p.streamk != 0;
  int run_dec = 0, run_st = 0, run_slot = 0, run_pre = 0, run_items = 0;
  for (int c0 = 0; c0 < p.B; c0 += kPrologueThreads) {
    const int b = c0 + tid;
    int lo = 0, hi = 0, P = 0, N = 0;
    int is_dec = 0, st = 0, nslot = 0, tiles = 0, S = 0, chunk = 0, n = 0;
    if (b < p.B) {
      if (seq_valid(p, b, lo, hi, P)) {
        N = hi - lo;
        if (N >= 1 && (int64_t)P + N > (int64_t)p.MB * p.BS) s_badblk = 1;
        if (N >= 1 && N <= p.dec_rows) {
          is_dec = 1;
          n = seq_keys(p, P, N);
          nslot = N;
          if (sk) {
            st = (n + 15) / 16;
          } else {
            S = max(1, min(p.fixed_splits, p.max_splits));
            chunk = (n + S - 1) / S;
            chunk = (chunk + kStageKeys - 1) / kStageKeys * kStageKeys;
            S = (n + chunk - 1) / chunk;
          }
        } else if (N > p.dec_rows) {
          tiles = (N + p.pre_rows - 1) / p.pre_rows;
        }
      } else {
        s_bad = 1;
      }
    }
    int t_dec, t_st, t_slot, t_pre, t_items;
    const int o_dec = block_scan(is_dec, &t_dec);
    const int o_st = block_scan(st, &t_st);
    const int o_slot = block_scan(nslot, &t_slot);
    const int o_pre = block_scan(tiles, &t_pre);
    const int o_items = block_scan(S, &t_items);
    // every index below stays inside its host-computed bound, even when overlapping
    // (invalid) cu ranges claim more tokens than exist
    const bool slot_ok = (int64_t)run_slot + o_slot + nslot <= p.slot_bound;
    const bool dec_ok =
        is_dec && slot_ok &&
        (sk ? run_dec + o_dec < p.B : (int64_t)run_items + o_items + S <= p.dec_bound);
    if (dec_ok) {
      atomicMax(&s_wslot, run_slot + o_slot + nslot);
      if (sk) {
        atomicMax(&s_wdec, run_dec + o_dec + 1);
        atomicMax(&s_wst, run_st + o_st + st);
      } else {
        atomicMax(&s_witems, run_items + o_items + S);
      }
    }
    if (dec_ok && sk) {
      DecSeq d;
      d.b = b;
      d.n = n;
      d.st = st;
      d.base = p.Hkv * (run_st + o_st);
      d.nq = N;
      d.cu0 = lo;
      d.P = P;
      d.slot = run_slot + o_slot;
      p.dec_seqs[run_dec + o_dec] = d;
      atomicMax(&s_maxst, st);
    }
    if (dec_ok && !sk) {
      for (int s = 0; s < S; ++s) {
        DecodeItem itm;
        itm.b = b;
        itm.nq = N;
        itm.split = s;
        itm.nsplit = S;
        itm.chunk = chunk;
        itm.slot_base = run_slot + o_slot;
        itm.pad0 = itm.pad1 = 0;
        p.dec_items[run_items + o_items + s] = itm;
      }
      for (int t = 0; t < N; ++t) {
        p.slot_token[run_slot + o_slot + t] = lo + t;
        p.slot_splits[run_slot + o_slot + t] = S;
      }
    }
    if (tiles > 0 && (int64_t)run_pre + o_pre + tiles <= p.pre_bound) {
      atomicMax(&s_wpre, run_pre + o_pre + tiles);
      for (int k = 0; k < tiles; ++k) {   // the heaviest (latest) tile first
        PrefillItem itm;
        itm.b = b;
        itm.q0 = (tiles - 1 - k) * p.pre_rows;
        itm.nq = min(p.pre_rows, N - itm.q0);
        itm.pad = 0;
        p.pre_items[run_pre + o_pre + k] = itm;
      }
    }
    run_dec += t_dec;
    run_st += t_st;
    run_slot += t_slot;
    run_pre += t_pre;
    run_items += t_items;
  }
  __syncthreads();
  const int ndec = sk ? s_wdec : 0;
  if (tid == 0) {
    const int64_t total = (int64_t)p.Hkv * s_wst;
    int64_t W = (total + p.total_warps - 1) / max(1, p.total_warps);
    W = max64(W, kSplitMinKeysDefault / 16);
    if (p.max_splits >= 2) W = max64(W, (s_maxst + p.max_splits - 2) / (p.max_splits - 1));
    p.counts[kCntDecSeqs] = ndec;
    p.counts[kCntTiles] = s_wpre * p.Hkv;
    p.counts[kCntStages] = sk ? (int)total : 0;
    p.counts[kCntTileNext] = 0;
    p.counts[kCntW] = (int)W;
    p.counts[kCntSplitItems] = sk ? 0 : s_witems;
    p.counts[kCntSlots] = s_wslot;
    if (s_bad) flag_status(p.status, PKV_DEV_BAD_SEQUENCE);
    if (s_badblk) flag_status(p.status, PKV_DEV_BAD_BLOCK);
  }
  for (int i = tid; i < ndec * p.Hkv; i += kPrologueThreads) p.seg_done[i] = 0;
  // tokens that no valid sequence covers get zero output; when every sequence is
  // valid and cu runs from 0 to T, cu is monotone and covers every token
  zero_uncovered(p, s_bad == 0 && p.cu[0] == 0 && p.cu[p.B] == p.T, tid, kPrologueThreads);
}

// kQ: the scatter blocks also rotate the query heads into the workspace (the kernel
// without kQ carries none of that code)
template <bool kQ>
__global__ void __launch_bounds__(kPrologueThreads) prologue_kernel(AttnParams p,
                                                                    ScatterParams sp) {
  if (blockIdx.x == 0) {
    plan_block(p);
    return;
  }
  const int64_t gid = (int64_t)(blockIdx.x - 1) * kPrologueThreads + threadIdx.x;
  if (sp.row_path)
    paged_scatter_row<kQ>(sp, gid >> 4, threadIdx.x & 31);
  else
    paged_scatter_thread<kQ>(sp, gid);
}

// ----------------------------------------------------------------------------------
// Single-pass path (the manifest's non-split variants, ScatterKV then Attend, here in one
// launch): CTA (b, h) writes the new K/V rows of sequence b for kv head h into the cache
// (rotated when asked, and with kQ the token's query heads of that kv head into the
// workspace), then attends every query row of (b, h) over all the keys it sees and writes
// the fp16 output. Only this CTA reads what it scattered, so no plan, partials, combine or
// second launch are needed. The last CTA zeroes tokens that no valid sequence covers.
// Taken when every sequence has one split and the call is small (host-side bound).
// ----------------------------------------------------------------------------------
template <int D, int NSTAGE, bool kQ>
__global__ void __launch_bounds__(kTileThreads) single_pass_kernel(AttnParams p,
                                                                   ScatterParams sp) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int64_t nseq = (int64_t)p.B * p.Hkv;
  if ((int64_t)blockIdx.x >= nseq) {
    int any_bad = 0;
    for (int b = threadIdx.x; b < p.B; b += kTileThreads) {
      int lo, hi, P;
      if (!seq_valid(p, b, lo, hi, P)) any_bad = 1;
    }
    any_bad = __syncthreads_or(any_bad);
    zero_uncovered(p, !any_bad && p.cu[0] == 0 && p.cu[p.B] == p.T, threadIdx.x, kTileThreads);
    return;
  }
  const int b = (int)(blockIdx.x / p.Hkv), h = (int)(blockIdx.x % p.Hkv);
  int lo, hi, P;
  if (!seq_valid(p, b, lo, hi, P)) {
    if (h == 0 && threadIdx.x == 0) flag_status(p.status, PKV_DEV_BAD_SEQUENCE);
    return;
  }
  const int N = hi - lo;
  if (N == 0) return;
  if (h == 0 && threadIdx.x == 0 && (int64_t)P + N > (int64_t)p.MB * p.BS)
    flag_status(p.status, PKV_DEV_BAD_BLOCK);
  if (sp.row_path) {   // half a warp per (token, kv head) row pair
    for (int t0 = 0; t0 < N; t0 += kTileThreads / 16) {
      const int t = t0 + (threadIdx.x >> 4);
      if (t < N) paged_scatter_row<kQ>(sp, (int64_t)(lo + t) * p.Hkv + h, threadIdx.x & 31);
    }
  } else {             // one thread per 16-byte chunk
    const int cpr = p.D / 8;
    for (int k = threadIdx.x; k < N * cpr; k += kTileThreads)
      paged_scatter_thread<kQ>(sp, ((int64_t)(lo + k / cpr) * p.Hkv + h) * cpr + k % cpr);
  }
  __threadfence_block();
  __syncthreads();   // the rows written above are read back below by this CTA alone
  const int n = seq_keys(p, P, N);
  const int R = N * p.G;
  bool bad = false;
  for (int row0 = 0; row0 < R; row0 += 16) {
    // keys up to the last row's position (causal)
    const int last_pos = (min(R, row0 + 16) - 1) / p.G;
    const int ke = (int)min64(n, (int64_t)P + last_pos + 1);
    split_rows<D, NSTAGE, true>(p, smem, b, h, lo, P, row0, R, 0, ke, 0, 0, bad);
    __syncthreads();   // the merge buffers alias the next row tile's key stages
  }
  if (bad) flag_status(p.status, PKV_DEV_BAD_BLOCK);
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

// fp16 tensor of dims (d0, d1, d2), innermost first, byte strides s1 and s2 of dims 1 and
// 2, boxes of b0 x b1 x b2 elements in the 128-byte swizzle; reads past the end give 0
bool encode_f16_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                   uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2) {
  const PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
  if (!fn) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {s1, s2};
  const cuuint32_t box[3] = {b0, b1, b2};
  const cuuint32_t unit[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            unit, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// Descriptors of the tensor-core prefill: query tile boxes of 64 columns x G heads x
// 128/G positions, and cache boxes of 64 columns x 1 kv head x tc_rows keys.
bool make_tc_maps(const AttnParams& p, TcMaps* m) {
  const uint64_t row_bytes = 128 * 2;
  return encode_f16_3d(&m->q, p.q, 128, (uint64_t)p.Hq, (uint64_t)p.T, row_bytes,
                       (uint64_t)p.q_stride * 2, 64, (uint32_t)p.G, (uint32_t)(128 / p.G)) &&
         encode_f16_3d(&m->k, p.kc, 128, (uint64_t)p.Hkv, (uint64_t)p.NB * p.BS, row_bytes,
                       (uint64_t)p.Hkv * row_bytes, 64, 1, (uint32_t)p.tc_rows) &&
         encode_f16_3d(&m->v, p.vc, 128, (uint64_t)p.Hkv, (uint64_t)p.NB * p.BS, row_bytes,
                       (uint64_t)p.Hkv * row_bytes, 64, 1, (uint32_t)p.tc_rows);
}

template <int D, int NS, int NSTAGE>
cudaError_t launch_attention_d(const AttnParams& p, const ScatterParams& sp, cudaStream_t s) {
  constexpr size_t smem = DecodeRing<D, NS>::kBytes > TileRing<D, NSTAGE>::kBytes
                              ? DecodeRing<D, NS>::kBytes
                              : TileRing<D, NSTAGE>::kBytes;
  static_assert(smem <= 232448, "dynamic shared memory over the per-block limit");
  constexpr size_t split_smem = TileRing<D, NSTAGE>::kBytes;
  static std::atomic<uint64_t> configured{0};
  int dev = -1;
  if (needs_configure(configured, &dev)) {
    cudaError_t e = cudaFuncSetAttribute(attention_kernel<D, NS, NSTAGE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(decode_split_kernel<D, NSTAGE>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)split_smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(single_pass_kernel<D, NSTAGE, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)split_smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(single_pass_kernel<D, NSTAGE, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)split_smem);
    if (e != cudaSuccess) return e;
    if (D == 128) {
      e = cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kTcSmem);
      if (e != cudaSuccess) return e;
    }
    mark_configured(configured, dev);
  }
  if (p.single_pass) {   // one launch: scatter and attention per (sequence, kv head)
    ProfScope ps("single_pass", s);
    const unsigned grid = (unsigned)((int64_t)p.B * p.Hkv + 1);
    if (sp.q_dst)
      single_pass_kernel<D, NSTAGE, true><<<grid, kTileThreads, split_smem, s>>>(p, sp);
    else
      single_pass_kernel<D, NSTAGE, false><<<grid, kTileThreads, split_smem, s>>>(p, sp);
    return cudaGetLastError();
  }
  const int64_t scatter_threads = pkv::scatter_threads(sp);
  {
    ProfScope ps("prologue", s);
    const unsigned pgrid =
        (unsigned)(1 + (scatter_threads + kPrologueThreads - 1) / kPrologueThreads);
    if (sp.q_dst)
      prologue_kernel<true><<<pgrid, kPrologueThreads, 0, s>>>(p, sp);
    else
      prologue_kernel<false><<<pgrid, kPrologueThreads, 0, s>>>(p, sp);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (!p.streamk && p.dec_bound > 0) {
    ProfScope ps("decode_split", s);
    decode_split_kernel<D, NSTAGE>
        <<<(unsigned)(p.dec_bound * p.Hkv), kTileThreads, split_smem, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  {
    ProfScope ps("attention", s);
    attention_kernel<D, NS, NSTAGE>
        <<<(unsigned)(p.total_warps / kWarps), kThreads, smem, s>>>(p);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess || !p.tc_prefill) return e;
  TcMaps maps;
  if (!make_tc_maps(p, &maps)) return cudaErrorInvalidValue;
  // programmatic dependent launch: prefill CTAs take SMs as decode CTAs retire
  ProfScope ps("prefill_tc", s);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.total_warps / (kWarps * kCtasPerSm)));
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = kTcSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_tc_kernel, p, maps);
}

}  // namespace

int attention_ctas_per_sm() { return kCtasPerSm; }
int attention_warps_per_cta() { return kWarps; }

cudaError_t launch_attention(const AttnParams& p, const ScatterParams& sp, cudaStream_t s) {
  switch (p.D) {
    case 64:
      return launch_attention_d<64, 2 * kDecStages, 4>(p, sp, s);
    case 128:
      return launch_attention_d<128, kDecStages, 3>(p, sp, s);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
