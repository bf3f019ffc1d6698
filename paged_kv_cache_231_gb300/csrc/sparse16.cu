// Block-sparse attention partials over fp16 queries and pages, on the 5th-generation
// tensor core.
//
// "alice-llm src/shaders/sparse_attention_forward.wgsl", sparse_forward and its layout
// comment: one partial (o, m, l) per (edge, query lane), edge = (q_idx, kv head, block,
// batch, block_len); key t < block_len of the block lives in page slot
// blk * pages_per_block + t / page_size of the sequence's table row, row t % page_size;
// an unmapped page gives score -1e30 and weight 0; s = scale * <q, k>, m = max s,
// weights exp(s - m), l = their sum, o = the weighted sum of value rows (unnormalised).
// The page computes in fp32; this variant takes fp16 q and pages (the partials stay
// fp32, so the combine is unchanged). Scores are fp16 products summed in fp32; the
// weights are computed in fp32, summed into l, and rounded once to fp16 for O = P V.
//
// GB300 form (edges grouped by (batch, block, kv head) by the grouping kernels of the
// fp32 path): a persistent CTA per SM, warp-specialised, every hand-off on an mbarrier.
//   warp 8 (scheduler): takes groups from a counter, publishes them in an 8-entry ring and
//     stages each group's K and V pages by TMA (one box per page and 64-column slice,
//     128-byte swizzle) straight in the operand layouts - K is the K-major B operand of
//     S = Q K^T, V the MN-major B operand of O = P V - in one of three stages. Its global
//     round trips are pipelined: the counter claim for the next group goes out an
//     iteration early, the claimed group's offsets and this group's block-table entries
//     are requested together, and the next group's entry is published before this
//     group's staging (the gather warps read edge records from it at group boundaries).
//   warps 10-13 (gather, 32 rows each): for each tile of 128 query rows (edges x query
//     lanes) read the rows' edge records (one 16-byte load per row, issued a tile ahead),
//     publish (partial index, block_len) per row in an 8-tile ring, and gather the Q rows
//     with cp.async into one of two K-major swizzled Q buffers.
//   warp 9, lane 0 (MMA): S(t) = Q(t) K^T into one of two TMEM S buffers, then
//     O(t-1) = P(t-1) V into one of two TMEM O buffers (tcgen05.mma kind::f16, P read
//     from TMEM), so the tensor core works on tile t while the softmax finishes t-1.
//   warps 0-3 (softmax, one thread per row): m, the weights (rounded to fp16, into one of
//     four TMEM P buffers) and l of tile t; (m, l) go to an 8-tile shared ring. The
//     softmax issues no global store, so its barrier arrivals never wait for one.
//   warps 4-7 (store): the O rows of tile t, through a per-warp shared-memory transpose
//     (whole 128-byte row segments, 32-byte stores: eight rows per store instruction), and
//     the rows' m and l.
// TMEM: S 0 / 64, O 128 / 128 + D, P 384 + 32 k (k < 4). Every wait is bounded; a wait that
// gives up raises a shared abort flag that ends every role, and the CTA drains what it
// issued.
#include <atomic>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "device_common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace pkv {
namespace {

constexpr int kThreads = 448;
constexpr int kNK = 64;                 // keys per block tile
constexpr uint32_t kTries = 1u << 22;   // default bound of each wait (polls)
// bound of this CTA's waits (kTries unless a test lowered it), set before the first barrier
__shared__ uint32_t s_tries;
constexpr uint32_t kTmS = 0, kTmO = 128, kTmP = 384;
constexpr int kSchedWarp = 8, kMmaWarp = 9, kGatherWarp0 = 10;   // gather: warps 10-13
constexpr int kRing = 8;                // group ring entries
constexpr uint32_t kStages = 3;         // K/V stages
constexpr uint32_t kQBufs = 2;          // Q buffers
constexpr uint32_t kRows = 8;           // row-info ring (tiles)

// mbarriers (index into the barrier array)
enum : int {
  kKVFull = 0,                   // [kStages] K/V stage landed (1 arrive + tx)
  kKVEmpty = kKVFull + kStages,  // [kStages] every MMA reading the stage done (commit)
  kQFull = kKVEmpty + kStages,   // [kQBufs] Q buffer gathered (4 x 32 cp.async arrivals)
  kQEmpty = kQFull + kQBufs,     // [kQBufs] S = Q K^T done with the buffer (commit)
  kSFull = kQEmpty + kQBufs,     // [2] S in TMEM (commit)
  kSEmpty = kSFull + 2,          // [2] softmax read S (4 warps)
  kPFull = kSEmpty + 2,          // [4] P in TMEM (4 warps)
  kPEmpty = kPFull + 4,          // [4] O = P V done with the P buffer (commit)
  kODone = kPEmpty + 4,          // [2] O = P V done (commit)
  kOEmpty = kODone + 2,          // [2] store warps read O (4 warps)
  kGFull = kOEmpty + 2,          // [kRing] ring entry published (scheduler)
  kGEmpty = kGFull + kRing,      // [kRing] ring entry released (softmax, store, gather, MMA)
  kRowFull = kGEmpty + kRing,    // [kRows] row info of a tile published (4 gather warps)
  kMLFull = kRowFull + kRows,    // [kRows] (m, l) of a tile published (4 softmax warps)
  kDrain = kMLFull + kRows,
  kNumBars = kDrain + 1
};

struct GroupEntry {   // a ring entry: group id (ngroups = no more groups) and its edges
  long long g;
  int e0, e1;
};

template <int D>
struct Layout {   // byte offsets from a 1024-byte-aligned base
  static constexpr uint32_t kSub = kNK * 128;           // [64 keys][64 columns] fp16, 8 KB
  static constexpr uint32_t kKV = (D / 64) * kSub;      // one K or V stage
  static constexpr uint32_t kQBuf = (D / 64) * 16384;   // D/64 x [128 rows][128 B]
  static constexpr uint32_t kK = 0;                     // K stages
  static constexpr uint32_t kV = kStages * kKV;         // V stages
  static constexpr uint32_t kQ = 2 * kStages * kKV;     // Q buffers
  static constexpr uint32_t kXfer = kQ + kQBufs * kQBuf;   // 4 store warps x [32][32] fp32
  static constexpr uint32_t kRowInfo = kXfer + 4 * 4096;   // [8][128] (partial, block_len)
  static constexpr uint32_t kML = kRowInfo + kRows * 128 * 8;      // [8][128] (m, l)
  static constexpr uint32_t kMasks = kML + kRows * 128 * 8;        // [3][2] key masks
  static constexpr uint32_t kRingOff = kMasks + kStages * 16;
  static constexpr uint32_t kBar = kRingOff + kRing * sizeof(GroupEntry);
  static constexpr uint32_t kAbort = kBar + kNumBars * 8;
  static constexpr uint32_t kTmem = kAbort + 4;
  static constexpr uint32_t kEnd = kTmem + 4;
};

struct Maps {     // TMA descriptors of the fp16 K and V pages (kernel parameters)
  CUtensorMap k;  // [pages * hkv * page_size rows][D] fp16, box 64 x page_size
  CUtensorMap v;
};

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

__device__ __forceinline__ void bar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
// arrive when every cp.async this thread issued so far has landed (count not raised)
__device__ __forceinline__ void bar_arrive_cp_async(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(smem_u32(bar))
               : "memory");
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

// Q rows are re-read by every edge that names their query: keep them in L2
__device__ __forceinline__ uint64_t l2_policy_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;\n" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void cp_async_16_hint(void* smem, const void* gmem, int src_bytes,
                                                 uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;\n" ::"r"(
                   smem_u32(smem)),
               "l"(gmem), "r"(src_bytes), "l"(pol)
               : "memory");
}

// The staging of one group, worked out by one warp from the block table: the key states
// {bit t set: key t mapped, bit t set: key t an invalid table reference} (keys past the
// block and keys of unmapped pages in neither), two ballots per mask; for lane j < pages
// per block the first row of page j in the page tensors (-1: unmapped, no copy), and the
// ballot of the lanes with a copy.
struct StagePlan {
  uint64_t vmask, imask;
  int row0;
  uint32_t bits;
};
// The staging of group g (block-table reads only: no shared memory is touched).
__device__ __forceinline__ StagePlan plan_group(const SparseParams& p, int64_t g) {
  const int lane = threadIdx.x & 31;
  const int h = (int)(g % p.hkv);
  const int64_t bb = g / p.hkv;
  const int blk = (int)(bb % p.nblk);
  const int batch = (int)(bb / p.nblk);
  uint64_t vmask = 0, imask = 0;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int t = lane + 32 * k;
    int state = 0;
    if (t < p.block_size) {
      const int64_t slot = (int64_t)blk * p.ppb + t / p.page_size;
      if (slot < p.max_pages) {
        const int64_t page = p.bt[(int64_t)batch * p.max_pages + slot];
        state = page >= p.num_pages ? 2 : page >= 0 ? 1 : 0;
      } else {
        state = 2;
      }
    }
    vmask |= (uint64_t)__ballot_sync(0xffffffffu, state == 1) << (32 * k);
    imask |= (uint64_t)__ballot_sync(0xffffffffu, state == 2) << (32 * k);
  }
  int row0 = -1;   // first row of page `lane` of the block in the page tensors
  if (lane < p.ppb) {
    const int64_t slot = (int64_t)blk * p.ppb + lane;
    if (slot < p.max_pages) {
      const int64_t page = p.bt[(int64_t)batch * p.max_pages + slot];
      if (page >= 0 && page < p.num_pages) row0 = (int)((page * p.hkv + h) * p.page_size);
    }
  }
  StagePlan sp;
  sp.vmask = vmask;
  sp.imask = imask;
  sp.row0 = row0;
  sp.bits = __ballot_sync(0xffffffffu, row0 >= 0);
  return sp;
}
// Stage `st` (free): the key masks of the plan into masks[st], then its K and V pages by
// TMA onto sbar. Unmapped pages get no copy: their rows keep earlier (finite) contents or
// the zeros the kernel starts with, and their weights are exactly 0.
template <int D>
__device__ void issue_group(const SparseParams& p, const Maps& maps, unsigned char* sm,
                            const StagePlan& sp, uint32_t st, uint64_t* sbar, bool withhold) {
  using L = Layout<D>;
  const int lane = threadIdx.x & 31;
  uint64_t* masks = reinterpret_cast<uint64_t*>(sm + L::kMasks) + 2 * st;
  if (lane == 0) {
    masks[0] = sp.vmask;
    masks[1] = sp.imask;
  }
  const int row0 = sp.row0;
  const uint32_t bits = sp.bits;
  __syncwarp();   // the key states are published by lane 0's arrive
  if (lane == 0)
    tc::mbar_arrive_expect_tx(sbar, (uint32_t)__popc(bits) * (uint32_t)p.page_size * D * 2u * 2u);
  __syncwarp();
  // one box per lane, all issued together: lane = (page j, 64-column slice q, K or V)
  constexpr int kBoxes = 2 * (D / 64);   // boxes per page
  const int j = lane / kBoxes, q = (lane % kBoxes) >> 1, isv = lane & 1;
  const int rj = __shfl_sync(0xffffffffu, row0, j & 31);
  if (j < p.ppb && rj >= 0 && !withhold) {
    unsigned char* dst = sm + (isv ? L::kV : L::kK) + st * L::kKV;
    const uint32_t off = (uint32_t)q * L::kSub + (uint32_t)(j * p.page_size) * 128u;
    tc::tma_load_2d(dst + off, isv ? &maps.v : &maps.k, q * 64, rj, sbar);
  }
}

// Reads ring entry gi (waiting for it); false at the end of the work or on abort.
__device__ __forceinline__ bool read_entry(const SparseParams& p, uint64_t* bars,
                                           const volatile GroupEntry* ring, uint32_t gi,
                                           volatile int* abort, bool whole_warp, long long& g,
                                           int& e0, int& e1) {
  const int slot = (int)(gi % kRing);
  const bool ok = whole_warp ? warp_wait(bars + kGFull + slot, (gi / kRing) & 1u, abort)
                             : wait_bar(bars + kGFull + slot, (gi / kRing) & 1u, abort);
  if (!ok) return false;
  g = ring[slot].g;
  e0 = ring[slot].e0;
  e1 = ring[slot].e1;
  return g < p.ngroups;
}

// Warps 0-3: per tile, m, the fp16 weights (into TMEM P) and l of row r.
template <int D>
__device__ void softmax_role(const SparseParams& p, unsigned char* sm, uint32_t tmem,
                             bool& bad) {
  using L = Layout<D>;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBar);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + L::kAbort);
  const volatile GroupEntry* ring = reinterpret_cast<const volatile GroupEntry*>(sm + L::kRingOff);
  const int2* rowinfo = reinterpret_cast<const int2*>(sm + L::kRowInfo);
  float2* mlinfo = reinterpret_cast<float2*>(sm + L::kML);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = warp * 32 + lane;
  const uint32_t lane_tm = tmem + ((uint32_t)(warp * 32) << 16);
  const int epc = 128 / p.qhead;
  uint32_t t = 0;
  for (uint32_t gi = 0;; ++gi) {
    long long g;
    int e0, e1;
    if (!read_entry(p, bars, ring, gi, abort, true, g, e0, e1)) return;
    const uint32_t st = gi % kStages;
    if (!warp_wait(bars + kKVFull + st, (gi / kStages) & 1u, abort)) return;
    // key masks of the group: bit t of vmask = mapped, of imask = invalid reference
    const uint64_t* masks = reinterpret_cast<const uint64_t*>(sm + L::kMasks) + 2 * st;
    const uint64_t vmask = masks[0], imask = masks[1];
    for (int c0 = e0; c0 < e1; c0 += epc, ++t) {
      if (!warp_wait(bars + kRowFull + (t % kRows), (t / kRows) & 1u, abort)) return;
      const int2 ri = rowinfo[(t % kRows) * 128 + r];   // (partial index or -1, block_len)
      const int b = (int)(t & 1u);
      if (!warp_wait(bars + kSFull + b, (t >> 1) & 1u, abort)) return;
      tc::fence_after_sync();
      float s[64];
      float (*s32)[32] = reinterpret_cast<float (*)[32]>(s);
      tc::tmem_ld32(lane_tm + kTmS + b * 64, s32[0]);
      tc::tmem_ld32(lane_tm + kTmS + b * 64 + 32, s32[1]);
      tc::tmem_wait_ld();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) bar_arrive(bars + kSEmpty + b);
      const int bl = ri.y;
      const uint64_t inblk = bl >= 64 ? ~0ull : ((1ull << bl) - 1ull);
      if (imask & inblk) bad = true;
      // keys that take part: mapped and inside the block (the rest score -1e30, and keys
      // past the block never raise m above that sentinel either)
      const uint64_t live = vmask & inblk;
      const uint32_t live_lo = (uint32_t)live, live_hi = (uint32_t)(live >> 32);
      // scores in base-2 units (scale * log2(e) * <q, k>): the weights are 2^(s - max);
      // four partial maxima and sums keep the dependency chains short
      // (pairs of keys go through one f32x2 instruction; each result is rounded as the
      // scalar operation)
      const float sl2 = p.scale * kLog2e;
      float mp[4] = {kNegLarge, kNegLarge, kNegLarge, kNegLarge};
#pragma unroll
      for (int k = 0; k < 64; k += 2) {
        const uint32_t word = k < 32 ? live_lo : live_hi;
        float x0, x1;
        fma2(x0, x1, s[k], s[k + 1], sl2, 0.f);
        const float sv0 = ((word >> (k & 31)) & 1u) ? x0 : kNegLarge;
        const float sv1 = ((word >> ((k + 1) & 31)) & 1u) ? x1 : kNegLarge;
        s[k] = sv0;
        s[k + 1] = sv1;
        mp[k & 3] = fmaxf(mp[k & 3], sv0);
        mp[(k + 1) & 3] = fmaxf(mp[(k + 1) & 3], sv1);
      }
      const float m2 = fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3]));
      // 2^(-1e30 - m) is exactly 0 for every finite m; with no key taking part m is the
      // sentinel itself, and subtracting 0 instead keeps every weight 0
      const float msub = m2 > 0.5f * kNegLarge ? m2 : 0.f;
      float pw[32];   // weights as fp16 pairs; l sums the fp32 weights
      float la[4] = {0.f, 0.f, 0.f, 0.f}, lb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int k = 0; k < 64; k += 2) {
        float d0, d1;
        fma2(d0, d1, s[k], s[k + 1], 1.f, -msub);   // s - m, exactly as a subtraction
        const float w0 = ex2(d0), w1 = ex2(d1);
        add2(la[(k >> 1) & 3], lb[(k >> 1) & 3], w0, w1);
        pw[k / 2] = __uint_as_float(pack_half2(w0, w1));
      }
      const float lrow =
          ((la[0] + lb[0]) + (la[1] + lb[1])) + ((la[2] + lb[2]) + (la[3] + lb[3]));
      // m in natural-log units (the -1e30 sentinel as is when no key takes part)
      const float mrow = m2 > 0.5f * kNegLarge ? m2 * 0.6931471805599453f : kNegLarge;
      // P buffer t % 4 is free once O(t-4) = P(t-4) V has completed
      const uint32_t pb = t & 3u;
      if (t >= 4 && !warp_wait(bars + kPEmpty + pb, ((t >> 2) - 1) & 1u, abort)) return;
      tc::fence_after_sync();
      tc::tmem_st32(lane_tm + kTmP + pb * 32, pw);
      tc::tmem_wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) bar_arrive(bars + kPFull + pb);
      // (m, l) for the store warps. The slot was last read for tile t - 8, whose stores are
      // done: S(t) followed O(t-2) = P V in the MMA order, which waited for the stores of
      // tile t-4 to read out their O buffer, and the stores of a tile read (m, l) first.
      mlinfo[(t % kRows) * 128 + r] = make_float2(mrow, lrow);
      __syncwarp();
      if (lane == 0) bar_arrive(bars + kMLFull + (t % kRows));
    }
    __syncwarp();
    if (lane == 0) bar_arrive(bars + kGEmpty + (gi % kRing));
  }
}

// 32-byte global store (the 256-bit st.global of sm_100 and later) with the streaming hint:
// half the store instructions of two 16-byte stores. dst must be 32-byte aligned.
__device__ __forceinline__ void st_cs_v8(float* dst, const float4& a, const float4& b) {
  asm volatile("st.global.cs.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};\n" ::"l"(dst),
               "f"(a.x), "f"(a.y), "f"(a.z), "f"(a.w), "f"(b.x), "f"(b.y), "f"(b.z), "f"(b.w)
               : "memory");
}

// Warps 4-7: per tile, the O rows of this warp's 32 TMEM lanes to memory.
template <int D>
__device__ void store_role(const SparseParams& p, unsigned char* sm, uint32_t tmem) {
  using L = Layout<D>;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBar);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + L::kAbort);
  const volatile GroupEntry* ring = reinterpret_cast<const volatile GroupEntry*>(sm + L::kRingOff);
  const int2* rowinfo = reinterpret_cast<const int2*>(sm + L::kRowInfo);
  const float2* mlinfo = reinterpret_cast<const float2*>(sm + L::kML);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;
  const int r = quarter * 32 + lane;
  const uint32_t lane_tm = tmem + ((uint32_t)(quarter * 32) << 16);
  float* xf = reinterpret_cast<float*>(sm + L::kXfer) + quarter * 1024;
  const int epc = 128 / p.qhead;
  const int q4 = lane & 7;
  // o_partial need only be 16-byte aligned; 32-byte stores when it is 32-byte aligned
  const bool o32 = (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0;
  uint32_t t = 0;
  for (uint32_t gi = 0;; ++gi) {
    long long g;
    int e0, e1;
    if (!read_entry(p, bars, ring, gi, abort, true, g, e0, e1)) return;
    for (int c0 = e0; c0 < e1; c0 += epc, ++t) {
      if (!warp_wait(bars + kRowFull + (t % kRows), (t / kRows) & 1u, abort)) return;
      const int pi = rowinfo[(t % kRows) * 128 + r].x;
      if (!warp_wait(bars + kMLFull + (t % kRows), (t / kRows) & 1u, abort)) return;
      const float2 ml = mlinfo[(t % kRows) * 128 + r];
      const int b = (int)(t & 1u);
      if (!warp_wait(bars + kODone + b, (t >> 1) & 1u, abort)) return;
      tc::fence_after_sync();
#pragma unroll 1
      for (int ch = 0; ch < D / 32; ++ch) {
        float o[32];
        tc::tmem_ld32(lane_tm + kTmO + b * D + ch * 32, o);
        tc::tmem_wait_ld();
        if (ch == D / 32 - 1) {   // O buffer b is read out
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) bar_arrive(bars + kOEmpty + b);
        }
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<float4*>(xf + lane * 32 + ((q ^ (lane & 7)) << 2)) =
              make_float4(o[q * 4], o[q * 4 + 1], o[q * 4 + 2], o[q * 4 + 3]);
        __syncwarp();
        if (o32) {   // four lanes per 128-byte row segment, eight rows per instruction
          const int j = lane & 3;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int rr = i * 8 + (lane >> 2);
            const int rpi = __shfl_sync(0xffffffffu, pi, rr);
            const float* row = xf + rr * 32;
            const float4 v0 = *reinterpret_cast<const float4*>(row + (((2 * j) ^ (rr & 7)) << 2));
            const float4 v1 =
                *reinterpret_cast<const float4*>(row + (((2 * j + 1) ^ (rr & 7)) << 2));
            if (rpi >= 0) st_cs_v8(p.o + (int64_t)rpi * D + ch * 32 + j * 8, v0, v1);
          }
        } else {   // eight lanes per row segment, four rows per instruction
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rr = i * 4 + (lane >> 3);
            const int rpi = __shfl_sync(0xffffffffu, pi, rr);
            const float4 v =
                *reinterpret_cast<const float4*>(xf + rr * 32 + ((q4 ^ (rr & 7)) << 2));
            if (rpi >= 0)
              __stcs(reinterpret_cast<float4*>(p.o + (int64_t)rpi * D + ch * 32 + q4 * 4), v);
          }
        }
        __syncwarp();
      }
      if (pi >= 0) {
        __stcs(p.m + pi, ml.x);
        __stcs(p.l + pi, ml.y);
      }
    }
    __syncwarp();
    if (lane == 0) bar_arrive(bars + kGEmpty + (gi % kRing));
  }
}

// Warp 8: group scheduling and K/V staging. Returns after publishing the end-of-work
// entry (or on abort); `issued[st]` counts the stagings of each stage.
template <int D>
__device__ void sched_role(const SparseParams& p, const Maps& maps, unsigned char* sm,
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
  int* counter = p.group_count + p.ngroups;
  // the first group in counter order at or after claimed counter value c that has edges
  auto resolve = [&](int c) -> long long {
    long long g = p.ngroups;
    if (lane == 0) {
      while (c < p.ngroups && p.group_off[c + 1] <= p.group_off[c]) c = atomicAdd(counter, 1);
      g = c < p.ngroups ? c : p.ngroups;
    }
    return __shfl_sync(0xffffffffu, g, 0);
  };
  // ring entry gi <- group g (a group past the last one ends the work)
  auto publish = [&](uint32_t gi, long long g, int e0, int e1) -> bool {
    const int slot = (int)(gi % kRing);
    if (gi >= kRing && !warp_wait(bars + kGEmpty + slot, ((gi / kRing) - 1) & 1u, abort))
      return false;
    if (lane == 0) {
      if (g >= p.ngroups) e0 = e1 = 0;
      ring[slot].g = g;
      ring[slot].e0 = e0;
      ring[slot].e1 = e1;
      bar_arrive(bars + kGFull + slot);   // release: the entry is visible to the waiters
    }
    return true;
  };
  int c0 = 0;
  if (lane == 0) c0 = atomicAdd(counter, 1);
  long long g = resolve(c0);
  if (!publish(0, g, g < p.ngroups ? p.group_off[g] : 0, g < p.ngroups ? p.group_off[g + 1] : 0))
    return;
  // lane 0: the counter value claimed for the next entry, one iteration ahead
  int cn = 0;
  if (lane == 0) cn = atomicAdd(counter, 1);
  for (uint32_t gi = 0; g < p.ngroups; ++gi) {
    // the claimed group's offsets are requested before this group's block-table reads, so
    // the two round trips overlap; the claim for the entry after it goes out next
    int o0 = 0, o1 = 0;
    if (lane == 0 && cn < p.ngroups) {
      o0 = p.group_off[cn];
      o1 = p.group_off[cn + 1];
    }
    const StagePlan sp = plan_group(p, g);
    long long gn = p.ngroups;
    if (lane == 0) {
      int c = cn;
      if (c < p.ngroups && o1 <= o0) {   // empty: the first non-empty group after it
        c = atomicAdd(counter, 1);
        while (c < p.ngroups && p.group_off[c + 1] <= p.group_off[c]) c = atomicAdd(counter, 1);
        if (c < p.ngroups) {
          o0 = p.group_off[c];
          o1 = p.group_off[c + 1];
        }
      }
      gn = c < p.ngroups ? c : p.ngroups;
      cn = gn < p.ngroups ? atomicAdd(counter, 1) : p.ngroups;
    }
    gn = __shfl_sync(0xffffffffu, gn, 0);
    if (!publish(gi + 1, gn, o0, o1)) return;
    const uint32_t st = gi % kStages;
    // the stage is free once every MMA of the group kStages back has completed
    if (gi >= kStages &&
        !warp_wait(bars + kKVEmpty + st, ((gi / kStages) - 1) & 1u, abort))
      return;
    // testing hook: the CTA's first staging is announced but never copied, so the waits
    // for it give up with nothing in flight
    issue_group<D>(p, maps, sm, sp, st, bars + kKVFull + st, p.withhold_copy && gi == 0);
    ++issued[st];
    g = gn;
  }
}

// Warps 10-13: per tile, rows 32 gw .. 32 gw + 31 (gw = warp - 10): their row info and Q
// rows by cp.async. The edge record of the next tile is loaded before this tile's copies
// are issued, so its latency overlaps them.
template <int D>
__device__ void gather_role(const SparseParams& p, unsigned char* sm) {
  using L = Layout<D>;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBar);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + L::kAbort);
  const volatile GroupEntry* ring = reinterpret_cast<const volatile GroupEntry*>(sm + L::kRingOff);
  int2* rowinfo = reinterpret_cast<int2*>(sm + L::kRowInfo);
  const int lane = threadIdx.x & 31;
  const int gw = (threadIdx.x >> 5) - kGatherWarp0;
  const int r = gw * 32 + lane;   // tile row of this lane
  const int epc = 128 / p.qhead;
  const int er = r / p.qhead, qh = r - er * p.qhead;
  constexpr int cpr = D / 8;        // 16-byte chunks per Q row
  constexpr int rpi = 32 / cpr;     // rows per warp instruction
  const uint64_t keep = l2_policy_last();
  // the tile in hand: ring entry gi, edges [c0, e1), kv head h
  uint32_t gi = 0;
  long long g;
  int c0, e1;
  if (!read_entry(p, bars, ring, 0, abort, true, g, c0, e1)) return;
  int h = (int)(g % p.hkv);
  auto lookup = [&](int cc, int ee) {
    return er < epc && cc + er < ee ? p.edge_rec[cc + er] : make_int4(-1, 0, 0, 0);
  };
  int4 rec = lookup(c0, e1);
  for (uint32_t t = 0;; ++t) {
    // the next tile (possibly the first of the next group), its record loaded ahead
    uint32_t ngi = gi;
    int nc0 = c0 + epc, ne1 = e1, nh = h;
    bool more = nc0 < e1;
    if (!more) {
      long long ng;
      more = read_entry(p, bars, ring, gi + 1, abort, true, ng, nc0, ne1);
      if (!more && *abort) return;
      ngi = gi + 1;
      nh = more ? (int)(ng % p.hkv) : 0;
    }
    const int4 nrec = more ? lookup(nc0, ne1) : make_int4(-1, 0, 0, 0);
    // row info of this tile. The slot was last read for tile t - 8, whose softmax and
    // stores are done: this point follows the gather of Q(t-1), which waited for S(t-3)
    // to finish; the MMA issued S(t-3) after O(t-5) = P V, which waited for the stores of
    // tile t-7 to read out their O buffer (the stores run in tile order) and for P(t-5),
    // which came after the softmax of t-5.
    const bool live = rec.x >= 0;
    rowinfo[(t % kRows) * 128 + r] =
        live ? make_int2(rec.x * p.qhead + qh, rec.z) : make_int2(-1, 0);
    __syncwarp();
    if (lane == 0) bar_arrive(bars + kRowFull + (t % kRows));
    const __half* src = live ? p.q16 + ((int64_t)rec.y * p.hq + h * p.qhead + qh) * D : nullptr;
    const uint32_t qb = t % kQBufs;
    if (t >= kQBufs && !warp_wait(bars + kQEmpty + qb, ((t / kQBufs) - 1) & 1u, abort)) return;
    unsigned char* qbuf = sm + L::kQ + qb * L::kQBuf;
    const int ch = lane % cpr;
#pragma unroll 4
    for (int i = 0; i < 32 / rpi; ++i) {
      const int rr = i * rpi + lane / cpr;   // row within this warp's 32 rows
      const __half* s = reinterpret_cast<const __half*>(
          __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(src), rr));
      unsigned char* dst = qbuf + (uint32_t)(ch >> 3) * 16384u +
                           tc::sw128((uint32_t)(gw * 32 + rr), (uint32_t)(ch & 7));
      cp_async_16_hint(dst, s ? s + ch * 8 : p.q16, s ? 16 : 0, keep);
    }
    bar_arrive_cp_async(bars + kQFull + qb);
    if (ngi != gi) {   // every tile of ring entry gi is gathered
      __syncwarp();
      if (lane == 0) bar_arrive(bars + kGEmpty + (gi % kRing));
    }
    if (!more) return;
    gi = ngi;
    c0 = nc0;
    e1 = ne1;
    h = nh;
    rec = nrec;
  }
}

// Warp 9, lane 0: S(t) = Q(t) K^T, then O(t-1) = P(t-1) V.
template <int D>
__device__ void mma_role(const SparseParams& p, unsigned char* sm, uint32_t tmem) {
  using L = Layout<D>;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBar);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + L::kAbort);
  const volatile GroupEntry* ring = reinterpret_cast<const volatile GroupEntry*>(sm + L::kRingOff);
  const int epc = 128 / p.qhead;
  const uint32_t idesc_s = tc::idesc_f16(128, kNK, false, false);
  const uint32_t idesc_o = tc::idesc_f16(128, D, false, true);
  const uint32_t kbase = smem_u32(sm + L::kK), vbase = smem_u32(sm + L::kV);
  const uint32_t qbase = smem_u32(sm + L::kQ);
  bool pend = false, pend_last = false;
  uint32_t pend_t = 0, pend_st = 0;
  auto issue_pv = [&]() -> bool {
    const uint32_t b = pend_t & 1u, pb = pend_t & 3u;
    if (!wait_bar(bars + kPFull + pb, (pend_t >> 2) & 1u, abort)) return false;
    if (pend_t >= 2 && !wait_bar(bars + kOEmpty + b, ((pend_t >> 1) - 1) & 1u, abort))
      return false;
    tc::fence_after_sync();
    const uint32_t va = vbase + pend_st * L::kKV;
#pragma unroll
    for (int ks = 0; ks < kNK / 16; ++ks)
      mma_tmem_a(tmem + kTmO + b * D, tmem + kTmP + pb * 32 + (uint32_t)ks * 8u,
                 tc::smem_desc(va + (uint32_t)ks * 2048u, L::kSub, 1024), idesc_o,
                 ks > 0 ? 1u : 0u);
    tc::commit(bars + kODone + b);
    tc::commit(bars + kPEmpty + pb);
    if (pend_last) tc::commit(bars + kKVEmpty + pend_st);
    pend = false;
    return true;
  };
  uint32_t t = 0;
  for (uint32_t gi = 0;; ++gi) {
    long long g;
    int e0, e1;
    if (!read_entry(p, bars, ring, gi, abort, false, g, e0, e1)) {
      if (!*abort && pend) issue_pv();
      return;
    }
    bar_arrive(bars + kGEmpty + (gi % kRing));
    const uint32_t st = gi % kStages;
    if (!wait_bar(bars + kKVFull + st, (gi / kStages) & 1u, abort)) return;
    const uint32_t ka = kbase + st * L::kKV;
    for (int c0 = e0; c0 < e1; c0 += epc, ++t) {
      const uint32_t qb = t % kQBufs, b = t & 1u;
      if (!wait_bar(bars + kQFull + qb, (t / kQBufs) & 1u, abort)) return;
      if (t >= 2 && !wait_bar(bars + kSEmpty + b, ((t >> 1) - 1) & 1u, abort)) return;
      tc::fence_async_shared();   // the Q rows were written by cp.async
      tc::fence_after_sync();
      const uint32_t qa = qbase + qb * L::kQBuf;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t qoff = (uint32_t)(ks >> 2) * 16384u + (uint32_t)(ks & 3) * 32u;
        const uint32_t koff = (uint32_t)(ks >> 2) * L::kSub + (uint32_t)(ks & 3) * 32u;
        tc::mma_f16(tmem + kTmS + b * 64, tc::smem_desc(qa + qoff, 16, 1024),
                    tc::smem_desc(ka + koff, 16, 1024), idesc_s, ks > 0 ? 1u : 0u);
      }
      tc::commit(bars + kSFull + b);
      tc::commit(bars + kQEmpty + qb);
      if (pend && !issue_pv()) return;
      pend = true;
      pend_t = t;
      pend_st = st;
      pend_last = c0 + epc >= e1;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    sparse_tc16_kernel(SparseParams p, const __grid_constant__ Maps maps) {
  using L = Layout<D>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBar);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + L::kAbort);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L::kTmem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the K/V stages start as zeros: rows no page fills must hold finite values
  for (uint32_t i = tid * 16; i < 2 * kStages * L::kKV; i += kThreads * 16)
    *reinterpret_cast<uint4*>(sm + i) = make_uint4(0u, 0u, 0u, 0u);
  tc::fence_async_shared();
  if (tid == 0) {
    for (uint32_t i = 0; i < kStages; ++i) {
      tc::mbar_init(bars + kKVFull + i, 1);
      tc::mbar_init(bars + kKVEmpty + i, 1);
    }
    for (uint32_t i = 0; i < kQBufs; ++i) {
      tc::mbar_init(bars + kQFull + i, 128);
      tc::mbar_init(bars + kQEmpty + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(bars + kSFull + i, 1);
      tc::mbar_init(bars + kSEmpty + i, 4);
      tc::mbar_init(bars + kODone + i, 1);
      tc::mbar_init(bars + kOEmpty + i, 4);
    }
    for (int i = 0; i < 4; ++i) {
      tc::mbar_init(bars + kPFull + i, 4);
      tc::mbar_init(bars + kPEmpty + i, 1);
    }
    for (int i = 0; i < kRing; ++i) {
      tc::mbar_init(bars + kGFull + i, 1);
      tc::mbar_init(bars + kGEmpty + i, 13);
    }
    for (uint32_t i = 0; i < kRows; ++i) {
      tc::mbar_init(bars + kRowFull + i, 4);
      tc::mbar_init(bars + kMLFull + i, 4);
    }
    tc::mbar_init(bars + kDrain, 1);
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
  if (warp < 4) {
    softmax_role<D>(p, sm, tmem, bad);
  } else if (warp < 8) {
    store_role<D>(p, sm, tmem);
  } else if (warp == kSchedWarp) {
    sched_role<D>(p, maps, sm, issued);
  } else if (warp >= kGatherWarp0) {
    gather_role<D>(p, sm);
    cp_async_wait<0>();
  } else if (warp == kMmaWarp && lane == 0) {
    mma_role<D>(p, sm, tmem);
    // let every MMA this thread issued finish before the CTA leaves
    tc::commit(bars + kDrain);
    tc::mbar_wait(bars + kDrain, 0, s_tries);
  }
  if (warp == kSchedWarp && *abort) {
    // a wait gave up: the last staging of each stage must land before the CTA leaves
    for (uint32_t st = 0; st < kStages; ++st)
      if (issued[st] > 0) tc::mbar_wait(bars + kKVFull + st, (issued[st] - 1) & 1u, s_tries);
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

// [pages * hkv * page_size rows][D] fp16 pages, boxes of 64 columns (128 bytes) x
// page_size rows in the 128-byte swizzle
bool encode_pages(CUtensorMap* m, const void* base, const SparseParams& p) {
  const PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)p.D, (cuuint64_t)(p.num_pages * p.hkv * p.page_size)};
  const cuuint64_t strides[1] = {(cuuint64_t)p.D * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)p.page_size};
  const cuuint32_t unit[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            unit, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_d(const SparseParams& p, cudaStream_t s) {
  constexpr size_t smem = Layout<D>::kEnd + 1024;
  static_assert(smem <= 232448, "shared memory over the per-block limit");
  static std::atomic<uint64_t> configured{0};
  int dev = -1;
  if (needs_configure(configured, &dev)) {
    cudaError_t e = cudaFuncSetAttribute(sparse_tc16_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    mark_configured(configured, dev);
  }
  int sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  Maps maps;
  if (!encode_pages(&maps.k, p.kp16, p) || !encode_pages(&maps.v, p.vp16, p))
    return cudaErrorInvalidValue;
  const int64_t grid = p.ngroups < sms ? p.ngroups : sms;
  ProfScope ps("sparse_partials", s);
  sparse_tc16_kernel<D><<<(unsigned)grid, kThreads, smem, s>>>(p, maps);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_sparse_tc16(const SparseParams& p, cudaStream_t s) {
  if (p.D == 64) return launch_d<64>(p, s);
  if (p.D == 128) return launch_d<128>(p, s);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
