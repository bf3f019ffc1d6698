// Internal host/device declarations shared by the library's translation units.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedkv.h"

namespace pkv {

constexpr int kMaxSplitsDefault = 16;    // manifest tunable MAX_SPLITS
constexpr int kSplitMinKeysDefault = 128;  // manifest tunable SPLIT_MIN_KEYS
constexpr int kSplitTargetWorkgroups = 1024;  // manifest tunable SPLIT_TARGET_WORKGROUPS
constexpr int kStageKeys = 64;           // keys per shared-memory stage (attention)

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
};

// ---- attention (AttendSplitK / Attend) ----------------------------------------------
struct DecodeItem {   // one split of one short (decoding) sequence
  int b, nq, split, nsplit, chunk, slot_base, pad0, pad1;
};
struct PrefillItem {  // one query tile of one multi-token sequence
  int b, q0, nq, pad;
};

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
  int split_policy, fixed_splits, max_splits, split_min_keys, num_sms;
  int dec_rows;            // max new tokens of a sequence handled as split-KV decode
  int pre_rows;            // query positions per prefill tile
  // workspace
  int32_t* counts;         // [0] decode items, [1] prefill items, [2] partial slots
  DecodeItem* dec_items;
  PrefillItem* pre_items;
  int32_t* slot_token;     // partial slot -> token
  int32_t* slot_splits;    // partial slot -> split count
  float* part_o;           // [(slot*Hq + hq)*max_splits + s][D]
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
  // grouping workspace
  int64_t nblk;            // blocks per sequence row of the table
  int64_t ngroups;         // nseq * nblk * hkv
  int32_t* group_count;    // [ngroups + 1]
  int32_t* group_off;      // [ngroups + 1]
  int32_t* group_cursor;   // [ngroups]
  int32_t* perm;           // [E]
};

// launchers (return cudaSuccess or the launch error)
cudaError_t launch_paged_scatter(const ScatterParams& p, cudaStream_t s);
cudaError_t launch_append(const AppendParams& p, cudaStream_t s);
cudaError_t launch_attention(const AttnParams& p, cudaStream_t s);
cudaError_t launch_combine(const CombineParams& p, cudaStream_t s);
cudaError_t launch_sparse(const SparseParams& p, cudaStream_t s);

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
