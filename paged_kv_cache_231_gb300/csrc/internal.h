// Internal host/device declarations shared by the library's translation units.
#pragma once

#include <atomic>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedkv.h"

namespace pkv {

constexpr int kMaxSplitsDefault = 16;    // manifest tunable MAX_SPLITS
constexpr int kSplitMinKeysDefault = 128;  // manifest tunable SPLIT_MIN_KEYS
constexpr int kSplitTargetWorkgroups = 1024;  // manifest tunable SPLIT_TARGET_WORKGROUPS
constexpr int kStageKeys = 64;           // keys per shared-memory stage (attention)
// Single-pass path bound: row tiles of 16 (if every token were in one sequence) x key
// ceiling of a sequence, i.e. the most key rows one CTA of that path may have to read.
constexpr int64_t kSinglePassWork = int64_t(1) << 18;

// ---- paged scatter (ScatterKV) ----------------------------------------------------
struct ScatterParams {
  const __half* k_src;     // first K element of token 0, kv head 0
  const __half* v_src;
  int64_t src_stride;      // elements between consecutive token rows
  __half* kc;
  __half* vc;
  const int32_t* cu;
  const int32_t* past;
  const int32_t* block_table;
  const int32_t* slot_mapping;
  const __half* cos;
  const __half* sin;
  int32_t* status;
  int T, B, Hkv, D, BS, MB;
  int64_t NB;
  int rotary_dim, rotary_positions, interleaved;
  int row_path;            // 1: half a warp per (token, kv head) row pair (scatter_dev.cuh)
  // query rotation (q_dst NULL: none): head hq of token i read at q_src + i*q_stride +
  // hq*D, written rotated at q_dst + (i*Hq + hq)*D
  const __half* q_src;
  __half* q_dst;
  int64_t q_stride;
  int Hq;
};

// ---- BNSH append (SparseAttention append) -----------------------------------------
struct AppendParams {
  const __half* k_src;
  const __half* v_src;
  int64_t src_stride;
  const int32_t* total_seq;
  const int32_t* key_totals;
  const __half* cos;
  const __half* sin;
  __half* pk;
  __half* pv;
  int32_t* status;
  int B, S, Hkv, D;
  int64_t MCS;
  int rotary_dim, rotary_positions, interleaved;
  int row_path;            // 1: half a warp per (token, kv head) row pair
  // query rotation (q_dst NULL: none): head hq of source row r read at q_src +
  // r*q_stride + hq*D, written at q_dst + (r*Hq + hq)*D
  const __half* q_src;
  __half* q_dst;
  int64_t q_stride;
  int Hq;
};

// Whether a row pair can move as half a warp: head rows of at most 16 chunks and, with a
// rotation, pairs that stay inside 8-element chunks (NeoX halves of a multiple of 8
// elements, interleaved rotary_dim a multiple of 8) and 16-byte aligned cos/sin rows.
inline bool row_path_ok(int D, int R, int interleaved, const void* cos_t, const void* sin_t) {
  if (D > 128 || D % 8 != 0) return false;
  if (R == 0) return true;
  const bool pairs = interleaved ? R % 8 == 0 : (R / 2) % 8 == 0;
  return pairs && (reinterpret_cast<uintptr_t>(cos_t) & 15u) == 0 &&
         (reinterpret_cast<uintptr_t>(sin_t) & 15u) == 0;
}

// ---- attention (AttendSplitK / Attend) ----------------------------------------------
struct DecodeItem {   // split mode: one split of one short (decoding) sequence
  int b, nq, split, nsplit, chunk, slot_base, pad0, pad1;
};
struct PrefillItem {  // one query tile of one multi-token sequence
  int b, q0, nq, pad;
};
struct DecSeq {       // stream-K mode: one short (decoding) sequence
  int b;              // batch row
  int n;              // keys its last new token sees (clamped to the block table)
  int st;             // 16-key stages per kv head = ceil(n / 16)
  int base;           // first global stage of (this sequence, kv head 0)
  int nq;             // new tokens
  int cu0;            // first token row
  int P;              // past length
  int slot;           // first partial slot
};

// counts[] words written by the planner
constexpr int kCntDecSeqs = 0;    // stream-K decode sequences
constexpr int kCntTiles = 1;      // prefill tiles = prefill items x kv heads
constexpr int kCntStages = 2;     // total 16-key stages of the stream-K decode
constexpr int kCntTileNext = 3;   // tile counter of the persistent kernel (zeroed)
constexpr int kCntW = 4;          // stages per warp
constexpr int kCntSplitItems = 5; // split mode: decode items
constexpr int kCntSlots = 6;      // split mode: partial slots
constexpr int kCntWords = 8;

struct AttnParams {
  const __half* q;         // query head row of (token, hq) at q + token*q_stride + hq*D
  int64_t q_stride;
  const __half* kc;
  const __half* vc;
  const int32_t* cu;
  const int32_t* past;
  const int32_t* block_table;
  __half* out;
  int32_t* status;
  int T, B, Hq, Hkv, G, D, BS, MB;
  int64_t NB;
  int bs_shift;            // log2(BS) when BS is a power of two, else -1
  float scale_log2;        // softmax scale * log2(e)
  // planning
  int streamk;             // 1: stream-K decode with fused combine; 0: split items
  int split_policy, fixed_splits, max_splits, split_min_keys;
  int dec_rows;            // max new tokens of a sequence handled as decode
  int pre_rows;            // query positions per prefill tile
  int total_warps;         // warps of the persistent kernel
  int tc_prefill;          // 1: prefill tiles of 128 rows on tcgen05 (head size 128)
  int tc_rows;             // keys per TMA box of the tcgen05 prefill (power of two, >= 8)
  int single_pass;         // 1: one launch, scatter + attention per (sequence, kv head)
  // testing hook (pkv_testing_wait_limit): poll bound of the tensor-core kernel's waits
  // (0 = its default) and 1 = each CTA withholds its first bulk copy
  uint32_t wait_tries;
  int withhold_copy;
  // workspace
  int32_t* counts;         // kCnt* words
  DecSeq* dec_seqs;        // stream-K
  int32_t* seg_done;       // stream-K: finished pieces per (decode sequence, kv head)
  DecodeItem* dec_items;   // split mode
  PrefillItem* pre_items;
  int32_t* slot_token;     // split mode: partial slot -> token
  int32_t* slot_splits;    // split mode: partial slot -> split count
  float* part_o;           // [(slot*Hq + hq)*max_splits + piece][D]
  float* part_m;
  float* part_l;
  int64_t dec_bound, pre_bound, slot_bound;
};

// ---- combine ------------------------------------------------------------------------
struct CombineParams {
  const float* o;
  const float* m;
  const float* l;
  const int32_t* seg_off;   // CSR or nullptr
  int64_t uniform;          // groups per segment when seg_off == nullptr
  void* out;
  float* lse;
  int64_t num_segments, lanes;
  int D;
  int out_f16;
  // paged-internal mode (seg_off == nullptr and slot_token != nullptr): segment =
  // slot*Hq + hq, groups [segment*uniform, segment*uniform + slot_splits[slot]),
  // output row slot_token[slot]*Hq + hq.
  const int32_t* slot_token;
  const int32_t* slot_splits;
  const int32_t* slot_count;
  int Hq;
};

// ---- block-sparse -------------------------------------------------------------------
struct SparseParams {
  const float* q;
  const float* kp;
  const float* vp;
  const int32_t* meta;
  const int32_t* bt;
  float* o;
  float* m;
  float* l;
  int32_t* status;
  int64_t Tq, E, nseq, max_pages, num_pages;
  int qhead, hq, hkv, D, block_size, page_size, ppb;
  float scale;
  const int32_t* qpos;     // [Tq] query positions (right-aligned causal) or NULL
  // fp16 inputs (f16 = 1): the same tensors as q / kp / vp, as halves
  int f16;
  const __half* q16;
  const __half* kp16;
  const __half* vp16;
  // grouping workspace
  int64_t nblk;            // blocks per sequence row of the table
  int64_t ngroups;         // nseq * nblk * hkv
  int32_t* group_count;    // [ngroups + 1]
  int32_t* group_off;      // [ngroups + 1]
  int32_t* group_cursor;   // [ngroups]
  int32_t* perm;           // [E]
  int4* edge_rec;          // [E] (edge, q_idx, block_len clipped to block_size, Q shifts of
                           // the edge's query heads as signed bytes when qshift is set and
                           // qhead <= 4, else 0), grouped order
  // fp32 tensor-core path: Q rows [Tq * hq] split into fp16 (hi, lo) scaled by 2^qshift, each
  // array chunk-major: [D / 8][Tq * hq][8]
  __half* qhi;
  __half* qlo;
  int32_t* qshift;
  // testing hook (pkv_testing_wait_limit), as in AttnParams
  uint32_t wait_tries;
  int withhold_copy;
};

// Kernel attributes (the dynamic shared memory limit) belong to a device's context: each
// launcher sets them once per device. Returns true when the current device still needs
// them; mark_configured records that they were set.
inline bool needs_configure(const std::atomic<uint64_t>& done, int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess) *dev = -1;
  return *dev < 0 || *dev >= 64 || !(done.load() & (1ull << *dev));
}
inline void mark_configured(std::atomic<uint64_t>& done, int dev) {
  if (dev >= 0 && dev < 64) done.fetch_or(1ull << dev);
}

// threads of the ScatterKV pass: 16 per row pair on the row path, else one per chunk
inline int64_t scatter_threads(const ScatterParams& p) {
  const int64_t rows = (int64_t)p.T * p.Hkv;
  return p.row_path ? rows * 16 : rows * (p.D / 8);
}

// launchers (return cudaSuccess or the launch error)
cudaError_t launch_paged_scatter(const ScatterParams& p, cudaStream_t s);
cudaError_t launch_append(const AppendParams& p, cudaStream_t s);
cudaError_t launch_attention(const AttnParams& p, const ScatterParams& sp, cudaStream_t s);
int attention_ctas_per_sm();
int attention_warps_per_cta();
cudaError_t launch_combine(const CombineParams& p, cudaStream_t s);
cudaError_t launch_sparse(const SparseParams& p, cudaStream_t s);

// Keys of an edge that take part: block_len clipped to the block and, with query
// positions, to the keys at or before the query's position (right-aligned causal).
__device__ __forceinline__ int edge_keys(const SparseParams& p, int q_idx, int blk, int bl) {
  int n = bl < p.block_size ? bl : p.block_size;
  if (p.qpos) {
    const int64_t lim = (int64_t)p.qpos[q_idx] - (int64_t)blk * p.block_size + 1;
    if (lim < n) n = (int)(lim < 0 ? 0 : lim);
  }
  return n;
}
// fp16 partials (sparse16.cu); the runtime has checked the shapes it takes
cudaError_t launch_sparse_tc16(const SparseParams& p, cudaStream_t s);
// Whether fp32 partials of this shape run on the tensor core (sparse.cu); such calls need
// the split Q rows in their workspace. pool_rows = num_pages * hkv * page_size and
// q_rows = num_queries * hq (callers pass INT64_MAX when a product would overflow).
bool sparse_tc_shape(int D, int block_size, int qhead, int page_size, int ppb,
                     int64_t pool_rows, int64_t q_rows);

// testing hook of the bounded waits (runtime.cpp): current poll bound (0 = default) and
// whether tensor-core kernels withhold their first bulk copy
uint32_t testing_wait_tries();
int testing_withhold_copy();

// profiler hooks (runtime.cpp)
void prof_begin(const char* name, cudaStream_t s);
void prof_end(const char* name, cudaStream_t s);
void count_launch();

struct ProfScope {
  const char* name;
  cudaStream_t stream;
  ProfScope(const char* n, cudaStream_t s) : name(n), stream(s) { prof_begin(n, s); }
  ~ProfScope() { prof_end(name, stream); count_launch(); }
};

}  // namespace pkv
