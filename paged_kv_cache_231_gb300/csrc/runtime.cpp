// Host side of the C ABI: argument validation (the PagedAttention manifest's contract
// predicates), planning (split bounds, the manifest's numSplits, workspace layout),
// launches, and a small per-kernel CUDA-event profiler.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstring>
#include <map>
#include <string>
#include <utility>
#include <vector>

#include "internal.h"

namespace pkv {

// ---------------------------------------------------------------- profiler / counters
namespace {
std::atomic<int64_t> g_launches{0};
// read by every launch on any thread; the event records themselves are single-threaded
// (the profiler is documented as not thread-safe)
std::atomic<bool> g_prof{false};
struct Rec {
  cudaEvent_t a, b;
};
std::map<std::string, std::vector<Rec>> g_recs;
std::vector<cudaEvent_t> g_pool;
std::vector<std::pair<std::string, cudaEvent_t>> g_open;

cudaEvent_t pooled_event() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}
}  // namespace

void prof_begin(const char* name, cudaStream_t s) {
  if (!g_prof.load(std::memory_order_relaxed)) return;
  cudaEvent_t e = pooled_event();
  cudaEventRecord(e, s);
  g_open.emplace_back(name, e);
}

void prof_end(const char* name, cudaStream_t s) {
  if (!g_prof.load(std::memory_order_relaxed) || g_open.empty()) return;
  cudaEvent_t e = pooled_event();
  cudaEventRecord(e, s);
  auto top = g_open.back();
  g_open.pop_back();
  g_recs[top.first].push_back({top.second, e});
  (void)name;
}

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

namespace {
std::atomic<uint32_t> g_wait_tries{0};
std::atomic<int> g_withhold{0};
}  // namespace
uint32_t testing_wait_tries() { return g_wait_tries.load(std::memory_order_relaxed); }
int testing_withhold_copy() { return g_withhold.load(std::memory_order_relaxed); }

// ---------------------------------------------------------------- helpers
namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// SM count of the current device, cached per device (safe to call from several host
// threads: each slot is written with the same value by whichever thread gets there first)
int num_sms_current() {
  constexpr int kFallback = 152;   // a GB300; used only if the runtime cannot be queried
  constexpr int kMaxDevices = 64;
  static std::atomic<int> cache[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return kFallback;
  if (dev >= 0 && dev < kMaxDevices) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return kFallback;
  if (dev >= 0 && dev < kMaxDevices) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

struct PagedLayout {
  int mode = 0;
  int G = 1;
  int dec_rows = 1, pre_rows = 4;
  int max_splits = 1;
  int fixed_splits = 1;
  int streamk = 0;
  int tc_rows = 0;   // > 0: prefill tiles on the tensor core, TMA boxes of tc_rows keys
  int single_pass = 0;   // 1: one launch of the single-pass kernel does the whole call
  int64_t dec_bound = 0, pre_bound = 0, slot_bound = 0;
  size_t off_counts = 0, off_seqs = 0, off_done = 0, off_dec = 0, off_pre = 0,
         off_slot_tok = 0, off_slot_spl = 0, off_po = 0, off_pm = 0, off_pl = 0,
         off_qrot = 0, total = 0;
  bool rotate_query = false;
  int pages_splits = 1;
};

// The manifest's numSplits (derive table).
int pages_num_splits(int64_t tokens, int64_t kv_heads, int64_t max_blocks,
                     int64_t block_size) {
  const int64_t base = tokens * kv_heads;
  const int64_t key_ceiling = max_blocks * block_size;
  const int64_t cap = std::max<int64_t>(
      1, std::min<int64_t>(kMaxSplitsDefault, key_ceiling / kSplitMinKeysDefault));
  const int64_t want = ceil_div(kSplitTargetWorkgroups, std::max<int64_t>(1, base));
  return (int)std::max<int64_t>(1, std::min(cap, want));
}

int check_paged(const pkv_paged_attention_args* a, bool attention, PagedLayout* L) {
  if (!a) return PKV_ERR_NULL;
  if (a->dtype != PKV_F16) return PKV_ERR_DTYPE;
  if (a->is_causal != 1) return PKV_ERR_CAUSAL;
  if (a->num_heads <= 0 || a->kv_num_heads <= 0 || a->num_heads % a->kv_num_heads != 0)
    return PKV_ERR_HEADS;
  if (a->head_size <= 0 || a->block_size <= 0 || a->num_blocks <= 0 || a->batch < 1 ||
      a->max_blocks < 1 || a->num_tokens < 0)
    return PKV_ERR_SHAPE;
  // every size below is formed from these as int64 products: bound the factors first
  if (a->num_heads > INT32_MAX || a->head_size > INT32_MAX || a->block_size > INT32_MAX ||
      a->max_blocks > INT32_MAX || a->num_blocks > INT32_MAX)
    return PKV_ERR_UNSUPPORTED;
  if (a->num_tokens == 0) {   // nothing is read or written; empty tensors may be NULL
    if (L) {
      L->mode = 0;
      L->G = (int)(a->num_heads / a->kv_num_heads);
      L->pages_splits = pages_num_splits(0, a->kv_num_heads, a->max_blocks, a->block_size);
      L->total = kAlign;
    }
    return PKV_OK;
  }
  const bool hk = a->key != nullptr, hv = a->value != nullptr;
  if (hk != hv) return PKV_ERR_KV_MODE;
  const int64_t qh = a->num_heads * a->head_size, kvh = a->kv_num_heads * a->head_size;
  const int mode = hk ? 1 : 2;
  if (mode == 1 && a->query_hidden != qh) return PKV_ERR_SHAPE;
  if (mode == 2 && a->query_hidden != qh + 2 * kvh) return PKV_ERR_SHAPE;
  if (a->rotary_dim < 0 || a->rotary_dim % 2 != 0 || a->rotary_dim > a->head_size)
    return PKV_ERR_SHAPE;
  if (a->rotary_dim > 0 && (!a->cos_cache || !a->sin_cache)) return PKV_ERR_NULL;
  if (a->rotary_dim > 0 && a->rotary_positions <= 0) return PKV_ERR_SHAPE;
  if (!a->query || !a->key_cache || !a->value_cache || !a->cumulative_sequence_length ||
      !a->past_seqlens || !a->block_table)
    return PKV_ERR_NULL;
  if (attention && !a->output) return PKV_ERR_NULL;
  if (a->head_size % 8 != 0) return PKV_ERR_UNSUPPORTED;
  if (!aligned16(a->query) || (hk && (!aligned16(a->key) || !aligned16(a->value))) ||
      !aligned16(a->key_cache) || !aligned16(a->value_cache) ||
      (attention && !aligned16(a->output)))
    return PKV_ERR_ALIGN;
  if (a->num_tokens > INT32_MAX / 2 || a->batch > INT32_MAX / 2 ||
      a->max_blocks * a->block_size > INT32_MAX / 2 || a->num_blocks > INT32_MAX)
    return PKV_ERR_UNSUPPORTED;
  const int64_t G = a->num_heads / a->kv_num_heads;
  if (attention) {
    if (a->head_size != 64 && a->head_size != 128) return PKV_ERR_UNSUPPORTED;
    if (G > 16) return PKV_ERR_UNSUPPORTED;
    if (a->split_policy == PKV_SPLIT_FIXED && a->fixed_splits < 1) return PKV_ERR_SHAPE;
    if (a->split_policy < PKV_SPLIT_AUTO || a->split_policy > PKV_SPLIT_FIXED)
      return PKV_ERR_SHAPE;
    if (a->max_splits < 0 || a->split_min_keys < 0) return PKV_ERR_SHAPE;
  }
  if (!L) return PKV_OK;
  L->mode = mode;
  L->G = (int)G;
  L->pages_splits =
      pages_num_splits(a->num_tokens, a->kv_num_heads, a->max_blocks, a->block_size);
  if (!attention) return PKV_OK;
  const int min_keys = a->split_min_keys > 0 ? a->split_min_keys : kSplitMinKeysDefault;
  const int cap = a->max_splits > 0 ? a->max_splits : kMaxSplitsDefault;
  if (a->split_policy == PKV_SPLIT_AUTO) {
    L->max_splits = (int)std::max<int64_t>(
        1, std::min<int64_t>(cap, ceil_div(a->max_blocks * a->block_size, min_keys)));
    L->fixed_splits = 1;
    // stream-K decode needs room for at least two pieces per (sequence, kv head)
    L->streamk = L->max_splits >= 2 ? 1 : 0;
  } else if (a->split_policy == PKV_SPLIT_PAGES) {
    L->max_splits = L->pages_splits;
    L->fixed_splits = L->pages_splits;
  } else {
    L->max_splits = a->fixed_splits;
    L->fixed_splits = a->fixed_splits;
  }
  L->dec_rows = (int)(16 / G);
  // prefill tiles: 128 rows on the 5th-generation tensor core (head size 128, cache
  // blocks of a multiple of 8 keys, loaded as TMA boxes of up to 128 keys), else 64 rows
  // of mma.sync tiles
  if (a->head_size == 128 && a->block_size % 8 == 0 &&
      a->num_blocks * a->block_size <= INT32_MAX) {
    int r = 8;
    while (r < 128 && a->block_size % (2 * r) == 0) r *= 2;
    L->tc_rows = r;
  }
  L->pre_rows = L->tc_rows > 0 ? (int)(128 / G) : 4 * L->dec_rows;
  const int64_t T = a->num_tokens, B = a->batch;
  // every sequence has one split (no partials, no combine) and the call is small: one
  // CTA per (sequence, kv head) scatters and attends in a single launch
  L->single_pass = L->max_splits == 1 && B * a->kv_num_heads < INT32_MAX / 2 &&
                   ceil_div(T * G, 16) * (a->max_blocks * a->block_size) <= kSinglePassWork;
  L->dec_bound = L->streamk ? 0 : B * L->max_splits;
  L->pre_bound = ceil_div(T, L->pre_rows) + std::min<int64_t>(B, T / (L->dec_rows + 1));
  L->slot_bound = std::min<int64_t>(T, B * L->dec_rows);
  // stage indices and grid sizes must fit in int32
  if (a->kv_num_heads * B * ceil_div(a->max_blocks * a->block_size, 16) > INT32_MAX / 2 ||
      L->dec_bound * a->kv_num_heads > INT32_MAX || L->pre_bound * a->kv_num_heads > INT32_MAX)
    return PKV_ERR_UNSUPPORTED;
  const int64_t prow = L->slot_bound * a->num_heads * L->max_splits;
  size_t off = 0;
  L->off_counts = off;
  off += align_up(4 * kCntWords);
  L->off_seqs = off;
  off += align_up(L->streamk ? sizeof(DecSeq) * (size_t)B : 0);
  L->off_done = off;
  off += align_up(L->streamk ? 4 * (size_t)B * a->kv_num_heads : 0);
  L->off_dec = off;
  off += align_up(sizeof(DecodeItem) * (size_t)L->dec_bound);
  L->off_pre = off;
  off += align_up(sizeof(PrefillItem) * (size_t)L->pre_bound);
  L->off_slot_tok = off;
  off += align_up(L->streamk ? 0 : 4 * (size_t)L->slot_bound);
  L->off_slot_spl = off;
  off += align_up(L->streamk ? 0 : 4 * (size_t)L->slot_bound);
  L->off_po = off;
  off += align_up(4 * (size_t)prow * a->head_size);
  L->off_pm = off;
  off += align_up(4 * (size_t)prow);
  L->off_pl = off;
  off += align_up(4 * (size_t)prow);
  L->rotate_query = a->rotary_query != 0 && a->rotary_dim > 0;
  L->off_qrot = off;
  off += align_up(L->rotate_query ? 2 * (size_t)T * a->num_heads * a->head_size : 0);
  L->total = off;
  return PKV_OK;
}

void fill_scatter(const pkv_paged_attention_args* a, int mode, ScatterParams& sp) {
  const int64_t D = a->head_size;
  const __half* q = static_cast<const __half*>(a->query);
  if (mode == 1) {
    sp.k_src = static_cast<const __half*>(a->key);
    sp.v_src = static_cast<const __half*>(a->value);
    sp.src_stride = a->kv_num_heads * D;
  } else {
    sp.k_src = q + a->num_heads * D;
    sp.v_src = q + (a->num_heads + a->kv_num_heads) * D;
    sp.src_stride = a->query_hidden;
  }
  sp.kc = static_cast<__half*>(a->key_cache);
  sp.vc = static_cast<__half*>(a->value_cache);
  sp.cu = a->cumulative_sequence_length;
  sp.past = a->past_seqlens;
  sp.block_table = a->block_table;
  sp.slot_mapping = a->slot_mapping;
  sp.cos = static_cast<const __half*>(a->cos_cache);
  sp.sin = static_cast<const __half*>(a->sin_cache);
  sp.status = a->device_status;
  sp.T = (int)a->num_tokens;
  sp.B = (int)a->batch;
  sp.Hkv = (int)a->kv_num_heads;
  sp.D = (int)D;
  sp.BS = (int)a->block_size;
  sp.MB = (int)a->max_blocks;
  sp.NB = a->num_blocks;
  sp.rotary_dim = (int)a->rotary_dim;
  sp.rotary_positions = (int)std::min<int64_t>(a->rotary_positions, INT32_MAX);
  sp.interleaved = a->rotary_interleaved ? 1 : 0;
  sp.row_path = row_path_ok(sp.D, sp.rotary_dim, sp.interleaved, sp.cos, sp.sin) ? 1 : 0;
}

int launch_status(cudaError_t e) { return e == cudaSuccess ? PKV_OK : PKV_ERR_LAUNCH; }

bool is_pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }
int log2i(int64_t x) {
  int s = 0;
  while ((int64_t(1) << s) < x) ++s;
  return s;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" {

int pkv_abi_version(void) { return PKV_ABI_VERSION; }

const char* pkv_status_string(int status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_NULL: return "a required pointer is NULL";
    case PKV_ERR_SHAPE: return "a size breaks the operator contract";
    case PKV_ERR_HEADS: return "num_heads / kv_num_heads must be positive and divisible";
    case PKV_ERR_DTYPE: return "unsupported dtype (the contract admits float16)";
    case PKV_ERR_KV_MODE: return "key and value must both be given or both be NULL";
    case PKV_ERR_CAUSAL: return "is_causal must be 1";
    case PKV_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case PKV_ERR_ALIGN: return "tensor pointer not 16-byte aligned";
    case PKV_ERR_UNSUPPORTED: return "size outside the compiled kernel variants";
    case PKV_ERR_LAUNCH: return "CUDA launch failed";
    default: return "unknown status";
  }
}

size_t pkv_sizeof_struct(const char* name) {
  if (!name) return 0;
  const std::string n(name);
  if (n == "pkv_paged_attention_args") return sizeof(pkv_paged_attention_args);
  if (n == "pkv_paged_plan") return sizeof(pkv_paged_plan);
  if (n == "pkv_tensor_desc") return sizeof(pkv_tensor_desc);
  if (n == "pkv_paged_shapes") return sizeof(pkv_paged_shapes);
  if (n == "pkv_kv_append_args") return sizeof(pkv_kv_append_args);
  if (n == "pkv_sparse_args") return sizeof(pkv_sparse_args);
  if (n == "pkv_combine_args") return sizeof(pkv_combine_args);
  return 0;
}

int64_t pkv_launch_count(void) { return g_launches.load(); }

int pkv_testing_wait_limit(uint32_t max_polls, int32_t withhold_first_copy) {
  if (withhold_first_copy && max_polls == 0) return PKV_ERR_SHAPE;
  g_wait_tries.store(max_polls, std::memory_order_relaxed);
  g_withhold.store(withhold_first_copy ? 1 : 0, std::memory_order_relaxed);
  return PKV_OK;
}

void pkv_profiler_enable(int on) { g_prof.store(on != 0, std::memory_order_relaxed); }

void pkv_profiler_reset(void) {
  for (auto& kv : g_recs)
    for (auto& r : kv.second) {
      g_pool.push_back(r.a);
      g_pool.push_back(r.b);
    }
  g_recs.clear();
  for (auto& o : g_open) g_pool.push_back(o.second);
  g_open.clear();
}

int pkv_profiler_query(const char* kernel, double* total_ms, int64_t* launches) {
  if (!kernel || !total_ms || !launches) return PKV_ERR_NULL;
  *total_ms = 0.0;
  *launches = 0;
  auto it = g_recs.find(kernel);
  if (it == g_recs.end()) return PKV_OK;
  for (auto& r : it->second) {
    if (cudaEventSynchronize(r.b) != cudaSuccess) return PKV_ERR_LAUNCH;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) return PKV_ERR_LAUNCH;
    *total_ms += ms;
    *launches += 1;
  }
  return PKV_OK;
}

// ---------------------------------------------------------------- paged attention
int pkv_paged_attention_plan(const pkv_paged_attention_args* args, pkv_paged_plan* plan) {
  if (!plan) return PKV_ERR_NULL;
  std::memset(plan, 0, sizeof(*plan));
  PagedLayout L;
  const int st = check_paged(args, true, &L);
  if (st != PKV_OK) return st;
  plan->mode = L.mode;
  plan->group_size = L.G;
  plan->pages_num_splits = L.pages_splits;
  plan->max_splits = L.max_splits;
  plan->pages_partial_bytes =
      args->num_tokens * args->num_heads * L.pages_splits * args->head_size * 4;
  plan->pages_stats_bytes = 2 * args->num_tokens * args->num_heads * L.pages_splits * 4;
  plan->workspace_bytes = (int64_t)L.total;
  plan->decode_item_bound = L.dec_bound;
  plan->prefill_item_bound = L.pre_bound;
  plan->partial_slot_bound = L.slot_bound;
  return PKV_OK;
}

int pkv_paged_attention_workspace_size(const pkv_paged_attention_args* args,
                                       size_t* bytes) {
  if (!bytes) return PKV_ERR_NULL;
  PagedLayout L;
  const int st = check_paged(args, true, &L);
  if (st != PKV_OK) return st;
  *bytes = L.total;
  return PKV_OK;
}

int pkv_paged_scatter_kv(const pkv_paged_attention_args* args, void* stream) {
  PagedLayout L;
  const int st = check_paged(args, false, &L);
  if (st != PKV_OK) return st;
  if (args->num_tokens == 0) return PKV_OK;
  ScatterParams sp{};
  fill_scatter(args, L.mode, sp);
  return launch_status(launch_paged_scatter(sp, static_cast<cudaStream_t>(stream)));
}

int pkv_paged_attention(const pkv_paged_attention_args* args, void* workspace,
                        size_t workspace_bytes, void* stream) {
  PagedLayout L;
  int st = check_paged(args, true, &L);
  if (st != PKV_OK) return st;
  if (args->num_tokens == 0) return PKV_OK;
  if (!workspace || workspace_bytes < L.total ||
      (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0)
    return PKV_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);

  ScatterParams sp{};
  fill_scatter(args, L.mode, sp);

  AttnParams ap{};
  ap.q = static_cast<const __half*>(args->query);
  ap.q_stride = args->query_hidden;
  ap.kc = static_cast<const __half*>(args->key_cache);
  ap.vc = static_cast<const __half*>(args->value_cache);
  ap.cu = args->cumulative_sequence_length;
  ap.past = args->past_seqlens;
  ap.block_table = args->block_table;
  ap.out = static_cast<__half*>(args->output);
  ap.status = args->device_status;
  ap.T = (int)args->num_tokens;
  ap.B = (int)args->batch;
  ap.Hq = (int)args->num_heads;
  ap.Hkv = (int)args->kv_num_heads;
  ap.G = L.G;
  ap.D = (int)args->head_size;
  ap.BS = (int)args->block_size;
  ap.MB = (int)args->max_blocks;
  ap.NB = args->num_blocks;
  ap.bs_shift = is_pow2(args->block_size) ? log2i(args->block_size) : -1;
  const double scale = args->scale != 0.f ? (double)args->scale
                                          : 1.0 / std::sqrt((double)args->head_size);
  ap.scale_log2 = (float)(scale * 1.4426950408889634);
  ap.streamk = L.streamk;
  ap.split_policy = args->split_policy;
  ap.fixed_splits = L.fixed_splits;
  ap.max_splits = L.max_splits;
  ap.split_min_keys = args->split_min_keys > 0 ? args->split_min_keys : kSplitMinKeysDefault;
  ap.dec_rows = L.dec_rows;
  ap.pre_rows = L.pre_rows;
  ap.total_warps = num_sms_current() * attention_ctas_per_sm() * attention_warps_per_cta();
  ap.tc_prefill = L.tc_rows > 0 ? 1 : 0;
  ap.tc_rows = L.tc_rows;
  ap.single_pass = L.single_pass;
  ap.wait_tries = testing_wait_tries();
  ap.withhold_copy = testing_withhold_copy();
  ap.counts = reinterpret_cast<int32_t*>(ws + L.off_counts);
  ap.dec_seqs = reinterpret_cast<DecSeq*>(ws + L.off_seqs);
  ap.seg_done = reinterpret_cast<int32_t*>(ws + L.off_done);
  ap.dec_items = reinterpret_cast<DecodeItem*>(ws + L.off_dec);
  ap.pre_items = reinterpret_cast<PrefillItem*>(ws + L.off_pre);
  ap.slot_token = reinterpret_cast<int32_t*>(ws + L.off_slot_tok);
  ap.slot_splits = reinterpret_cast<int32_t*>(ws + L.off_slot_spl);
  ap.part_o = reinterpret_cast<float*>(ws + L.off_po);
  ap.part_m = reinterpret_cast<float*>(ws + L.off_pm);
  ap.part_l = reinterpret_cast<float*>(ws + L.off_pl);
  if (L.rotate_query) {   // the prologue writes the rotated query; the attention reads it
    sp.q_src = static_cast<const __half*>(args->query);
    sp.q_stride = args->query_hidden;
    sp.q_dst = reinterpret_cast<__half*>(ws + L.off_qrot);
    sp.Hq = (int)args->num_heads;
    ap.q = sp.q_dst;
    ap.q_stride = args->num_heads * args->head_size;
  }
  ap.dec_bound = L.dec_bound;
  ap.pre_bound = L.pre_bound;
  ap.slot_bound = L.slot_bound;
  cudaError_t e = launch_attention(ap, sp, s);
  if (e != cudaSuccess) return PKV_ERR_LAUNCH;

  // one split per sequence: the split kernel (or the single-pass one) wrote the output
  if (!L.streamk && L.slot_bound > 0 && L.max_splits > 1 && !L.single_pass) {
    CombineParams cp{};
    cp.o = ap.part_o;
    cp.m = ap.part_m;
    cp.l = ap.part_l;
    cp.seg_off = nullptr;
    cp.uniform = L.max_splits;
    cp.out = args->output;
    cp.lse = nullptr;
    cp.num_segments = L.slot_bound;
    cp.lanes = 1;
    cp.D = (int)args->head_size;
    cp.out_f16 = 1;
    cp.slot_token = ap.slot_token;
    cp.slot_splits = ap.slot_splits;
    cp.slot_count = ap.counts + kCntSlots;
    cp.Hq = ap.Hq;
    e = launch_combine(cp, s);
    if (e != cudaSuccess) return PKV_ERR_LAUNCH;
  }
  return PKV_OK;
}

// ---------------------------------------------------------------- contract check
int pkv_paged_contract_check(const pkv_paged_shapes* sh, uint32_t* failed, int32_t* mode) {
  if (!sh || !failed || !mode) return PKV_ERR_NULL;
  *failed = 0;
  *mode = 0;
  const pkv_tensor_desc &q = sh->query, &k = sh->key, &v = sh->value, &kc = sh->key_cache,
                        &vc = sh->value_cache, &cu = sh->cumulative_sequence_length,
                        &past = sh->past_seqlens, &bt = sh->block_table,
                        &sm = sh->slot_mapping, &out = sh->output;
  if (!q.present || !kc.present || !vc.present || !cu.present || !past.present ||
      !bt.present || !out.present)
    return PKV_ERR_NULL;
  const int64_t Hq = sh->num_heads, Hkv = sh->kv_num_heads;
  const int64_t head = kc.rank == 4 ? kc.dims[3] : 0;
  const int64_t bsz = kc.rank == 4 ? kc.dims[1] : 0;
  const int64_t qhid = Hq * head, kvhid = Hkv * head, pstride = qhid + 2 * kvhid;
  const int64_t tokens = q.rank >= 1 ? q.dims[0] : -1;
  bool same = kc.rank == vc.rank;
  for (int i = 0; same && i < kc.rank && i < 4; ++i) same = kc.dims[i] == vc.dims[i];
  const bool cache_ok = kc.rank == 4 && vc.rank == 4 && same && kc.dims[2] == Hkv &&
                        bsz > 0 && head > 0 && kc.dtype == q.dtype && vc.dtype == q.dtype;
  const bool heads_ok = Hq > 0 && Hkv > 0 && Hq % Hkv == 0;
  const int64_t batch = cu.rank == 1 ? cu.dims[0] - 1 : -1;
  const int64_t mblocks = bt.rank == 2 ? bt.dims[1] : 0;
  const bool sched_ok = cu.rank == 1 && past.rank == 1 && bt.rank == 2 && batch >= 1 &&
                        past.dims[0] == batch && bt.dims[0] == batch && mblocks >= 1;
  const bool io_ok = q.rank == 2 && out.rank == 2 && out.dims[0] == tokens &&
                     out.dims[1] == qhid && out.dtype == q.dtype && q.dtype == PKV_F16;
  const bool sep = k.present && v.present && k.rank == 2 && v.rank == 2 &&
                   k.dims[0] == tokens && v.dims[0] == tokens && k.dims[1] == kvhid &&
                   v.dims[1] == kvhid && k.dtype == q.dtype && v.dtype == q.dtype &&
                   q.rank == 2 && q.dims[1] == qhid;
  const bool packed = !k.present && !v.present && q.rank == 2 && q.dims[1] == pstride;
  const bool slot_ok = sm.present ? (sm.rank == 1 && sm.dims[0] == tokens) : true;
  uint32_t f = 0;
  if (!cache_ok) f |= PKV_PRED_CACHE_SHAPE;
  if (!heads_ok) f |= PKV_PRED_HEAD_LAYOUT;
  if (!sched_ok) f |= PKV_PRED_SCHEDULE_SHAPE;
  if (!io_ok) f |= PKV_PRED_IO_SHAPE;
  if (!sep) f |= PKV_PRED_SEPARATE_KV;
  if (!packed) f |= PKV_PRED_PACKED_KV;
  if (!slot_ok) f |= PKV_PRED_SLOT_SHAPE;
  *failed = f;
  *mode = sep ? 1 : (packed ? 2 : 0);
  // status of the first failure
  const bool int_ok = (cu.dtype == PKV_I32 && past.dtype == PKV_I32 && bt.dtype == PKV_I32 &&
                       (!sm.present || sm.dtype == PKV_I32));
  if (q.dtype != PKV_F16 || kc.dtype != q.dtype || vc.dtype != q.dtype ||
      out.dtype != q.dtype || !int_ok)
    return PKV_ERR_DTYPE;
  if (!heads_ok) return PKV_ERR_HEADS;
  if (!cache_ok || !sched_ok || !io_ok || !slot_ok) return PKV_ERR_SHAPE;
  if (*mode == 0) return k.present != v.present ? PKV_ERR_KV_MODE : PKV_ERR_SHAPE;
  if (sh->is_causal != 1) return PKV_ERR_CAUSAL;
  return PKV_OK;
}

// ---------------------------------------------------------------- KV append
int pkv_kv_append_rotary(const pkv_kv_append_args* a, void* stream) {
  if (!a) return PKV_ERR_NULL;
  if (a->dtype != PKV_F16) return PKV_ERR_DTYPE;
  if (a->num_heads <= 0 || a->kv_num_heads <= 0 || a->num_heads % a->kv_num_heads != 0)
    return PKV_ERR_HEADS;
  if (a->batch < 0 || a->seq_len < 0 || a->head_size <= 0 || a->max_cache_seq <= 0)
    return PKV_ERR_SHAPE;
  // offsets below are int64 products of these: bound the factors first
  if (a->num_heads > INT32_MAX || a->head_size > INT32_MAX || a->max_cache_seq > INT32_MAX ||
      a->batch > INT32_MAX / 2 || a->seq_len > INT32_MAX / 2)
    return PKV_ERR_UNSUPPORTED;
  if (a->rotary_dim < 0 || a->rotary_dim % 2 != 0 || a->rotary_dim > a->head_size)
    return PKV_ERR_SHAPE;
  if (!a->source || !a->present_key || !a->present_value || !a->total_sequence_length ||
      !a->key_total_sequence_lengths)
    return PKV_ERR_NULL;
  if (!a->packed && !a->value) return PKV_ERR_KV_MODE;
  if (a->rotary_dim > 0 && (!a->cos_cache || !a->sin_cache)) return PKV_ERR_NULL;
  if (a->rotary_dim > 0 && a->rotary_positions <= 0) return PKV_ERR_SHAPE;
  if (a->head_size % 8 != 0) return PKV_ERR_UNSUPPORTED;
  if (!aligned16(a->source) || (!a->packed && !aligned16(a->value)) ||
      !aligned16(a->present_key) || !aligned16(a->present_value))
    return PKV_ERR_ALIGN;
  if (a->query_out && !a->packed && !a->query) return PKV_ERR_NULL;
  if (a->query_out && (!aligned16(a->query_out) || (!a->packed && !aligned16(a->query))))
    return PKV_ERR_ALIGN;
  if (a->batch * a->seq_len > INT32_MAX / 2 || a->batch > INT32_MAX / 2)
    return PKV_ERR_UNSUPPORTED;
  if (a->batch == 0 || a->seq_len == 0) return PKV_OK;
  AppendParams p{};
  const int64_t D = a->head_size;
  const __half* src = static_cast<const __half*>(a->source);
  if (a->packed) {
    p.k_src = src + a->num_heads * D;
    p.v_src = src + (a->num_heads + a->kv_num_heads) * D;
    p.src_stride = (a->num_heads + 2 * a->kv_num_heads) * D;
  } else {
    p.k_src = src;
    p.v_src = static_cast<const __half*>(a->value);
    p.src_stride = a->kv_num_heads * D;
  }
  p.total_seq = a->total_sequence_length;
  p.key_totals = a->key_total_sequence_lengths;
  p.cos = static_cast<const __half*>(a->cos_cache);
  p.sin = static_cast<const __half*>(a->sin_cache);
  p.pk = static_cast<__half*>(a->present_key);
  p.pv = static_cast<__half*>(a->present_value);
  p.status = a->device_status;
  p.B = (int)a->batch;
  p.S = (int)a->seq_len;
  p.Hkv = (int)a->kv_num_heads;
  p.D = (int)D;
  p.MCS = a->max_cache_seq;
  p.rotary_dim = (int)a->rotary_dim;
  p.rotary_positions = (int)std::min<int64_t>(a->rotary_positions, INT32_MAX);
  p.interleaved = a->interleaved ? 1 : 0;
  p.row_path = row_path_ok(p.D, p.rotary_dim, p.interleaved, p.cos, p.sin) ? 1 : 0;
  if (a->query_out) {
    p.q_src = a->packed ? src : static_cast<const __half*>(a->query);
    p.q_stride = a->packed ? p.src_stride : a->num_heads * D;
    p.q_dst = static_cast<__half*>(a->query_out);
    p.Hq = (int)a->num_heads;
  }
  return launch_status(launch_append(p, static_cast<cudaStream_t>(stream)));
}

// ---------------------------------------------------------------- block-sparse
namespace {
// fp32 calls whose shape runs on the tensor core take Q as split fp16 rows (workspace)
bool sparse_split_q(const pkv_sparse_args* a) {
  // the factors are positive and at most INT32_MAX here (checked before the call)
  const int64_t hp = a->hkv * a->page_size;
  const int64_t pool = a->num_pages <= INT32_MAX / hp ? a->num_pages * hp : INT64_MAX;
  const int64_t qrows = a->num_queries <= INT32_MAX / a->hq ? a->num_queries * a->hq : INT64_MAX;
  return a->dtype != PKV_F16 && a->num_queries > 0 &&
         sparse_tc_shape((int)a->head_dim, (int)a->block_size, (int)a->qhead,
                         (int)a->page_size, (int)a->pages_per_block, pool, qrows);
}
int check_sparse(const pkv_sparse_args* a, int64_t* nblk, int64_t* ngroups, size_t* bytes) {
  if (!a) return PKV_ERR_NULL;
  // the sizes below are int64 products of these: bound the factors first
  if (a->hkv > INT32_MAX || a->qhead > INT32_MAX || a->page_size > INT32_MAX ||
      a->pages_per_block > INT32_MAX || a->max_pages > INT32_MAX || a->num_pages > INT32_MAX ||
      a->num_seqs > INT32_MAX)
    return PKV_ERR_UNSUPPORTED;
  if (a->hkv <= 0 || a->qhead <= 0 || a->hq != a->hkv * a->qhead) return PKV_ERR_HEADS;
  if (a->num_edges < 0 || a->num_queries < 0 || a->num_seqs < 0 || a->max_pages <= 0 ||
      a->num_pages < 0 || a->page_size <= 0 || a->pages_per_block <= 0 ||
      a->block_size <= 0 || a->block_size > a->page_size * a->pages_per_block)
    return PKV_ERR_SHAPE;
  if (a->head_dim != 64 && a->head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if (a->block_size > 128 || a->qhead > 64) return PKV_ERR_UNSUPPORTED;
  if (a->dtype != 0 && a->dtype != PKV_F32 && a->dtype != PKV_F16) return PKV_ERR_DTYPE;
  if (a->dtype == PKV_F16 &&
      (a->block_size > 64 || a->page_size % 8 != 0 || a->page_size * a->pages_per_block > 64 ||
       a->num_pages > INT32_MAX / (a->hkv * a->page_size)))
    return PKV_ERR_UNSUPPORTED;
  if (a->num_edges > INT32_MAX / 64) return PKV_ERR_UNSUPPORTED;
  const int64_t nb = (a->max_pages + a->pages_per_block - 1) / a->pages_per_block;
  if (a->num_seqs > (INT32_MAX / 2) / (nb * a->hkv)) return PKV_ERR_UNSUPPORTED;
  const int64_t ng = a->num_seqs * nb * a->hkv;
  *nblk = nb;
  *ngroups = ng;
  *bytes = 2 * align_up(4 * (size_t)(ng + 1)) + align_up(4 * (size_t)ng) +
           align_up(4 * (size_t)a->num_edges) + align_up(16 * (size_t)a->num_edges);
  if (sparse_split_q(a)) {   // split Q rows: hi, lo (fp16) and the shift of each row
    const size_t rows = (size_t)a->num_queries * (size_t)a->hq;
    *bytes += 2 * align_up(rows * (size_t)a->head_dim * 2) + align_up(rows * 4);
  }
  return PKV_OK;
}
}  // namespace

int pkv_sparse_attention_partials_workspace_size(const pkv_sparse_args* a, size_t* bytes) {
  if (!bytes) return PKV_ERR_NULL;
  int64_t nb, ng;
  return check_sparse(a, &nb, &ng, bytes);
}

int pkv_sparse_attention_partials(const pkv_sparse_args* a, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  int64_t nb = 0, ng = 0;
  size_t need = 0;
  const int st = check_sparse(a, &nb, &ng, &need);
  if (st != PKV_OK) return st;
  if (a->num_edges == 0) return PKV_OK;
  // with no query rows every edge is out of range: q is never read and may be NULL
  if ((!a->q && a->num_queries > 0) || !a->k_pages || !a->v_pages || !a->edge_meta ||
      !a->block_tables || !a->o_partial || !a->m_partial || !a->l_partial)
    return PKV_ERR_NULL;
  if (!aligned16(a->q) || !aligned16(a->k_pages) || !aligned16(a->v_pages) ||
      !aligned16(a->o_partial))
    return PKV_ERR_ALIGN;
  if (!workspace || workspace_bytes < need ||
      (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0)
    return PKV_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  SparseParams p{};
  p.f16 = a->dtype == PKV_F16 ? 1 : 0;
  if (p.f16) {
    p.q16 = static_cast<const __half*>(a->q);
    p.kp16 = static_cast<const __half*>(a->k_pages);
    p.vp16 = static_cast<const __half*>(a->v_pages);
  } else {
    p.q = static_cast<const float*>(a->q);
    p.kp = static_cast<const float*>(a->k_pages);
    p.vp = static_cast<const float*>(a->v_pages);
  }
  p.meta = a->edge_meta;
  p.bt = a->block_tables;
  p.o = a->o_partial;
  p.m = a->m_partial;
  p.l = a->l_partial;
  p.status = a->device_status;
  p.Tq = a->num_queries;
  p.E = a->num_edges;
  p.nseq = a->num_seqs;
  p.max_pages = a->max_pages;
  p.num_pages = a->num_pages;
  p.qhead = (int)a->qhead;
  p.hq = (int)a->hq;
  p.hkv = (int)a->hkv;
  p.D = (int)a->head_dim;
  p.block_size = (int)a->block_size;
  p.page_size = (int)a->page_size;
  p.ppb = (int)a->pages_per_block;
  p.scale = a->softmax_scale;
  p.qpos = a->query_positions;
  p.wait_tries = testing_wait_tries();
  p.withhold_copy = testing_withhold_copy();
  p.nblk = nb;
  p.ngroups = ng;
  size_t off = 0;
  p.group_count = reinterpret_cast<int32_t*>(ws + off);
  off += align_up(4 * (size_t)(ng + 1));
  p.group_off = reinterpret_cast<int32_t*>(ws + off);
  off += align_up(4 * (size_t)(ng + 1));
  p.group_cursor = reinterpret_cast<int32_t*>(ws + off);
  off += align_up(4 * (size_t)ng);
  p.perm = reinterpret_cast<int32_t*>(ws + off);
  off += align_up(4 * (size_t)a->num_edges);
  p.edge_rec = reinterpret_cast<int4*>(ws + off);
  off += align_up(16 * (size_t)a->num_edges);
  if (sparse_split_q(a)) {
    const size_t rows = (size_t)a->num_queries * (size_t)a->hq;
    p.qhi = reinterpret_cast<__half*>(ws + off);
    off += align_up(rows * (size_t)a->head_dim * 2);
    p.qlo = reinterpret_cast<__half*>(ws + off);
    off += align_up(rows * (size_t)a->head_dim * 2);
    p.qshift = reinterpret_cast<int32_t*>(ws + off);
  }
  return launch_status(launch_sparse(p, static_cast<cudaStream_t>(stream)));
}

// ---------------------------------------------------------------- combine
int pkv_combine_partials(const pkv_combine_args* a, void* stream) {
  if (!a) return PKV_ERR_NULL;
  if (a->num_segments < 0 || a->lanes < 1) return PKV_ERR_SHAPE;
  if (a->head_dim != 64 && a->head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if (a->out_dtype != PKV_F16 && a->out_dtype != PKV_F32) return PKV_ERR_DTYPE;
  if (!a->segment_offsets && a->uniform_count < 0) return PKV_ERR_SHAPE;
  if (a->num_segments == 0) return PKV_OK;
  if (!a->o || !a->m || !a->l || !a->out) return PKV_ERR_NULL;
  if (!aligned16(a->o) || !aligned16(a->out)) return PKV_ERR_ALIGN;
  CombineParams p{};
  p.o = a->o;
  p.m = a->m;
  p.l = a->l;
  p.seg_off = a->segment_offsets;
  p.uniform = a->uniform_count;
  p.out = a->out;
  p.lse = a->lse;
  p.num_segments = a->num_segments;
  p.lanes = a->lanes;
  p.D = (int)a->head_dim;
  p.out_f16 = a->out_dtype == PKV_F16 ? 1 : 0;
  return launch_status(launch_combine(p, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
