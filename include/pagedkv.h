/*
 * pagedkv.h - C ABI of the GB300 paged / block-sparse grouped-query attention library.
 *
 * Operations (each names the page and passage that defines it):
 *
 *   pkv_paged_attention        "com.microsoft.PagedAttention manifest.json": operator
 *                              inputs/outputs/attributes, the derive table and the
 *                              ScatterKV -> AttendSplitK -> AttendSplitKMerge passes.
 *   pkv_paged_scatter_kv       the ScatterKV pass of the same manifest on its own.
 *   pkv_kv_append_rotary       "com.microsoft.SparseAttention sparse-kv-append.wgsl.jinja":
 *                              sparse_schedule, sparse_rotary and the KV-append main.
 *   pkv_sparse_attention_partials
 *                              "alice-llm src/shaders/sparse_attention_forward.wgsl":
 *                              sparse_forward and its layout comment block.
 *   pkv_combine_partials       log-sum-exp merge of (o, m, l) partials: the manifest's
 *                              AttendSplitKMerge pass and the merge of sparse partials.
 *
 * Conventions for every call:
 *   - Tensor pointers are DEVICE pointers owned by the caller; the library never frees
 *     or retains them. Scratch memory is a caller-provided device workspace whose size
 *     the matching *_workspace_size call returns; the library allocates nothing.
 *   - `stream` is a cudaStream_t (CUstream) handle passed as void*; NULL is the legacy
 *     default stream. Calls enqueue work and return without synchronising.
 *   - Host-side argument errors return a pkv_status before anything is enqueued.
 *     Invalid DATA found on the device (a block id outside the pool, a slot past the
 *     pool, ...) never traps: the offending row is skipped or masked as documented and
 *     a PKV_DEV_* bit is OR-ed into the optional `device_status` int32 word.
 *   - All layouts are row-major and dense; sizes are element counts.
 *   - fp16 tensors and every row stride must be 16-byte aligned (head_size % 8 == 0).
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKV_ABI_VERSION 3

typedef enum pkv_status {
  PKV_OK = 0,
  PKV_ERR_NULL = 1,        /* a required pointer is NULL */
  PKV_ERR_SHAPE = 2,       /* a size breaks the contract (cacheShapeOk, ioShapeOk,
                              scheduleShapeOk or slotShapeOk of the manifest) */
  PKV_ERR_HEADS = 3,       /* num_heads or kv_num_heads <= 0, or not divisible */
  PKV_ERR_DTYPE = 4,       /* dtype other than the operation's type constraint */
  PKV_ERR_KV_MODE = 5,     /* exactly one of key / value given (neither separateKv
                              nor packedKv holds) */
  PKV_ERR_CAUSAL = 6,      /* is_causal != 1 (the manifest admits only 1) */
  PKV_ERR_WORKSPACE = 7,   /* workspace NULL, too small or not 256-byte aligned */
  PKV_ERR_ALIGN = 8,       /* a tensor pointer is not 16-byte aligned */
  PKV_ERR_UNSUPPORTED = 9, /* a size outside the compiled kernel variants (see each call) */
  PKV_ERR_LAUNCH = 10      /* a CUDA launch or API call failed */
} pkv_status;

/* Bits OR-ed into *device_status by kernels that meet invalid data. */
#define PKV_DEV_BAD_BLOCK 1u     /* block-table entry outside [0, num_blocks), or a key
                                    position past max_blocks * block_size: key masked,
                                    row not written */
#define PKV_DEV_BAD_SLOT 2u      /* slot_mapping entry >= num_blocks * block_size: the
                                    token's K/V are not written (negative = padding,
                                    skipped without a flag) */
#define PKV_DEV_BAD_POSITION 4u  /* KV-append position >= max_cache_seq: row skipped */
#define PKV_DEV_BAD_SEQUENCE 8u  /* cumulative_sequence_length / past_seqlens
                                    inconsistent for a sequence: its tokens get zero
                                    output and are not scattered */
#define PKV_DEV_BAD_EDGE 16u     /* edge_meta field out of range: block_len clipped to
                                    block_size, or a page slot / page id treated as
                                    unmapped; an edge whose q_idx, head, batch or
                                    block lies outside the tensors gets the empty
                                    partial */
#define PKV_DEV_TIMEOUT 32u      /* a bounded wait of a tensor-core kernel gave up: the
                                    outputs that CTA had not yet written (prefill tiles,
                                    block-sparse partials) are not written; it waited
                                    (bounded) for what it had issued, freed its tensor
                                    memory and returned */

typedef enum pkv_dtype { PKV_F16 = 1, PKV_BF16 = 2, PKV_F32 = 3, PKV_I32 = 4 } pkv_dtype;

/* ---------------------------------------------------------------------------------
 * Paged attention (PagedAttention manifest)
 * ------------------------------------------------------------------------------- */

/* Split policy for the attention pass. */
#define PKV_SPLIT_AUTO 0   /* per-sequence split count chosen on the device: up to
                              max_splits splits of >= split_min_keys keys, sized so the
                              whole batch covers the GPU several times over */
#define PKV_SPLIT_PAGES 1  /* every decoding sequence uses the manifest's numSplits */
#define PKV_SPLIT_FIXED 2  /* every decoding sequence uses fixed_splits (tests) */

typedef struct pkv_paged_attention_args {
  /* query  fp16 [num_tokens, query_hidden]. query_hidden = num_heads*head_size when
            key/value are given (separateKv); (num_heads + 2*kv_num_heads)*head_size for
            packed [Q | K | V] rows when key == value == NULL (packedKv). */
  const void* query;
  /* key, value  fp16 [num_tokens, kv_num_heads*head_size] or both NULL. */
  const void* key;
  const void* value;
  /* key_cache, value_cache  fp16 [num_blocks, block_size, kv_num_heads, head_size];
            updated in place by the scatter pass (the manifest's optional outputs). */
  void* key_cache;
  void* value_cache;
  /* cumulative_sequence_length int32 [batch + 1]: tokens of sequence b are rows
            [cu[b], cu[b+1]) of query. past_seqlens int32 [batch]: tokens already in
            the cache. block_table int32 [batch, max_blocks]: entry c is the physical
            block holding keys [c*block_size, (c+1)*block_size) of the sequence; -1 (or
            any id outside the pool) = unmapped. */
  const int32_t* cumulative_sequence_length;
  const int32_t* past_seqlens;
  const int32_t* block_table;
  /* slot_mapping int32 [num_tokens] or NULL: flat pool row blk*block_size + offset of
            each new token (negative = padding, not written). When NULL the scatter
            destination comes from block_table at the token's absolute position. The
            attention pass always reads keys through block_table. */
  const int32_t* slot_mapping;
  /* output fp16 [num_tokens, num_heads*head_size]. */
  void* output;
  /* optional int32 word that kernels OR PKV_DEV_* bits into (may be NULL). */
  int32_t* device_status;
  /* optional rotary of the new keys before they enter the cache (NULL = none):
            fp16 [rotary_positions, rotary_dim/2] cos / sin tables, rotation rule of the
            SparseAttention append page at the token's absolute position. */
  const void* cos_cache;
  const void* sin_cache;

  int64_t num_tokens;
  int64_t query_hidden;
  int64_t batch;
  int64_t num_heads;
  int64_t kv_num_heads;
  int64_t head_size;
  int64_t block_size;
  int64_t num_blocks;
  int64_t max_blocks;
  int64_t rotary_dim;        /* 0 = no rotary; else even and <= head_size */
  int64_t rotary_positions;  /* rows of cos_cache / sin_cache */
  int32_t rotary_interleaved;/* 0 = NeoX split pairs, 1 = interleaved pairs */
  int32_t is_causal;         /* must be 1 */
  int32_t dtype;             /* must be PKV_F16 (type constraint T = float16) */
  float scale;               /* softmax scale; 0 means 1/sqrt(head_size) */
  int32_t split_policy;      /* PKV_SPLIT_* */
  int32_t fixed_splits;      /* for PKV_SPLIT_FIXED */
  int32_t max_splits;        /* 0 = 16 (manifest MAX_SPLITS) */
  int32_t split_min_keys;    /* 0 = 128 (manifest SPLIT_MIN_KEYS) */
  /* 1 (with rotary_dim > 0): every query head of a new token is rotated at the token's
            absolute position with the key's rule and cos/sin tables before the
            attention (the append page rotates keys only; this is the query half of
            rotary attention). The rotated query is rounded to fp16 into the workspace
            (num_tokens*num_heads*head_size*2 more bytes); the query input is not
            written. A token whose position has no cos/sin row keeps its query
            unrotated (its key is skipped with PKV_DEV_BAD_POSITION). 0: keys only. */
  int32_t rotary_query;
  int32_t reserved;
} pkv_paged_attention_args;

typedef struct pkv_paged_plan {
  int32_t mode;              /* 1 = separate K/V, 2 = packed QKV */
  int32_t group_size;        /* num_heads / kv_num_heads */
  int32_t pages_num_splits;  /* the manifest's derive.numSplits for these shapes */
  int32_t max_splits;        /* per-sequence split bound used by this call */
  int64_t pages_partial_bytes; /* the manifest's pagedSplitScratchBytes at its numSplits */
  int64_t pages_stats_bytes;   /* the manifest's pagedSplitStatsBytes */
  int64_t workspace_bytes;     /* bytes pkv_paged_attention needs */
  int64_t decode_item_bound;   /* grid bound of the split-KV decode pass */
  int64_t prefill_item_bound;  /* grid bound of the tiled prefill pass */
  int64_t partial_slot_bound;  /* tokens that may need split partials */
} pkv_paged_plan;

/* Host only (no CUDA call): validates the arguments against the contract and fills
 * *plan. Returns PKV_OK or the first failing status. Pointers are checked for NULL /
 * alignment only if non-NULL values are required by the chosen mode. */
int pkv_paged_attention_plan(const pkv_paged_attention_args* args, pkv_paged_plan* plan);

/* Host only: workspace bytes pkv_paged_attention needs for these sizes. */
int pkv_paged_attention_workspace_size(const pkv_paged_attention_args* args,
                                       size_t* bytes);

/* ScatterKV + AttendSplitK + AttendSplitKMerge of the manifest, GB300 form:
 *   1. scatter: new K/V rows (rotated first when cos/sin are given) -> caches;
 *   2. plan (device): per-sequence work items; multi-token sequences become query
 *      tiles, short sequences become split-KV items;
 *   3. attention: causal GQA, token at absolute position pos sees keys 0..pos, query
 *      head hq uses kv head hq / (num_heads / kv_num_heads); tiles write the output
 *      directly, split items write fp32 (o, m, l) partials to the workspace;
 *   4. combine: LSE merge of the partials into output.
 * When every sequence has one split (the resolved split bound is 1: short caches under
 * PKV_SPLIT_AUTO, max_splits = 1, fixed_splits = 1, or a manifest numSplits of 1) and
 * the call is small (ceil(num_tokens * group / 16) * max_blocks * block_size <= 2^18),
 * the manifest's non-split form (ScatterKV then Attend) runs as ONE launch: each CTA
 * scatters one (sequence, kv head)'s new rows and attends all of that pair's query rows;
 * no partials, no combine. Larger one-split calls skip only the combine.
 * workspace: device memory of at least pkv_paged_attention_workspace_size bytes,
 * 256-byte aligned, owned by the caller, contents need not be initialised and are
 * scratch after the call. Supported: head_size in {64, 128}; num_heads/kv_num_heads
 * <= 16; any block_size >= 1. Otherwise PKV_ERR_UNSUPPORTED. */
int pkv_paged_attention(const pkv_paged_attention_args* args, void* workspace,
                        size_t workspace_bytes, void* stream);

/* Paged attention without a caller-provided workspace. The pages have no counterpart
 * to this call: it serves callers that may not allocate device memory (for example an
 * engine plugin whose enqueue step must not allocate, or a framework that has given
 * all device memory to its own pool). Scratch comes from a __device__ array of
 * PKV_STATIC_WORKSPACE_BYTES inside this library, which every GPU that loads the
 * library holds until the process exits; the call itself allocates nothing.
 *   - Same arguments, results and status codes as pkv_paged_attention; returns
 *     PKV_ERR_WORKSPACE when pkv_paged_attention_workspace_size exceeds
 *     PKV_STATIC_WORKSPACE_BYTES.
 *   - The first call on a device looks up the array's device address (a runtime
 *     call, once per device, with that device current): make that first call before
 *     any stream capture. With CUDA's default lazy module loading that first call is
 *     also when the library's device code is loaded on the device and the array's
 *     memory is committed: make it before a caller's own pool reserves the device's
 *     memory (or load modules eagerly, CUDA_MODULE_LOADING=EAGER), else it fails with
 *     PKV_ERR_LAUNCH.
 *   - The address is cached per device for the life of the process: a device reset
 *     (cudaDeviceReset) after the first call is not supported, because the reloaded
 *     module may place the array elsewhere.
 *   - All calls on a device share the one array and it keeps the last call's contents;
 *     nothing in it needs to start at zero. Calls whose work overlaps on the GPU (other
 *     streams, other threads) race on it: serialise them. */
#define PKV_STATIC_WORKSPACE_BYTES (32u << 20)
int pkv_paged_attention_static_workspace(const pkv_paged_attention_args* args,
                                         void* stream);

/* The ScatterKV pass alone (same argument block; query is read only in packed mode,
 * output and the attention fields are ignored). Bit-exact copy when rotary_dim == 0. */
int pkv_paged_scatter_kv(const pkv_paged_attention_args* args, void* stream);

/* Shape-level contract check of the manifest (host only). Each tensor is described
 * by presence, rank, dtype (pkv_dtype) and up to 4 dims. On return *failed holds
 * PKV_PRED_* bits of the predicates that are false and *mode is 1 (separate),
 * 2 (packed) or 0 (neither). Returns PKV_OK when pagedContractOk holds, a mode
 * exists and is_causal == 1; else the status of the first failure. */
typedef struct pkv_tensor_desc {
  int32_t present;
  int32_t rank;
  int32_t dtype;
  int32_t reserved;
  int64_t dims[4];
} pkv_tensor_desc;

typedef struct pkv_paged_shapes {
  pkv_tensor_desc query, key, value, key_cache, value_cache;
  pkv_tensor_desc cumulative_sequence_length, past_seqlens, block_table, slot_mapping;
  pkv_tensor_desc output;
  int64_t num_heads;
  int64_t kv_num_heads;
  int32_t is_causal;
  int32_t reserved;
} pkv_paged_shapes;

#define PKV_PRED_CACHE_SHAPE 1u
#define PKV_PRED_HEAD_LAYOUT 2u
#define PKV_PRED_SCHEDULE_SHAPE 4u
#define PKV_PRED_IO_SHAPE 8u
#define PKV_PRED_SEPARATE_KV 16u
#define PKV_PRED_PACKED_KV 32u
#define PKV_PRED_SLOT_SHAPE 64u

int pkv_paged_contract_check(const pkv_paged_shapes* shapes, uint32_t* failed,
                             int32_t* mode);

/* ---------------------------------------------------------------------------------
 * KV append + RoPE into a [batch, kv_heads, max_cache_seq, head] cache
 * (SparseAttention append page)
 * ------------------------------------------------------------------------------- */
typedef struct pkv_kv_append_args {
  /* source fp16: packed [batch*seq_len, (num_heads + 2*kv_num_heads)*head_size] rows
     [Q | K | V] when packed != 0, else key rows [batch*seq_len, kv_num_heads*head_size]. */
  const void* source;
  const void* value;                         /* separate mode: [batch*seq_len, kv*head] */
  const int32_t* total_sequence_length;      /* device scalar: == seq_len -> prompt mode */
  const int32_t* key_total_sequence_lengths; /* [batch]: history = total - seq_len */
  const void* cos_cache;                     /* fp16 [rotary_positions, rotary_dim/2] */
  const void* sin_cache;
  void* present_key;                         /* fp16 [batch, kv, max_cache_seq, head] */
  void* present_value;
  int32_t* device_status;                    /* optional */
  int64_t batch;
  int64_t seq_len;
  int64_t num_heads;
  int64_t kv_num_heads;
  int64_t head_size;
  int64_t max_cache_seq;
  int64_t rotary_dim;                        /* 0 = plain copy; else even, <= head_size */
  int64_t rotary_positions;
  int32_t packed;
  int32_t interleaved;
  int32_t dtype;                             /* PKV_F16 */
  int32_t reserved;
  /* optional query rotation (query_out NULL: none). The num_heads query heads of each
     new row, read from the packed row's leading heads or, in separate mode, from
     `query` [batch*seq_len, num_heads*head_size], are rotated at the row's position
     with K's rule and tables and written to query_out fp16 [batch*seq_len,
     num_heads*head_size]; with rotary_dim == 0, or at a position without a cos/sin
     row, the row is copied unrotated. The page rotates keys only; the query half
     uses nothing it does not define. Independent of max_cache_seq. */
  const void* query;
  void* query_out;
} pkv_kv_append_args;

/* For each (batch b, kv head h, new token t): position = history(b) + t with the
 * sparse_schedule rule (both totals read as u32); K rotated at that position when
 * rotary_dim > 0 (leading member own*cos - partner*sin, trailing own*cos +
 * partner*sin, fp32 math, fp16 round-to-nearest-even), V copied; written to row
 * `position` of (b, h). Rows no new token lands on are untouched. position >=
 * max_cache_seq (or >= rotary_positions when rotating) skips the row and sets
 * PKV_DEV_BAD_POSITION. With query_out, the query heads are rotated the same way.
 * query_out must not overlap the source or the caches. */
int pkv_kv_append_rotary(const pkv_kv_append_args* args, void* stream);

/* ---------------------------------------------------------------------------------
 * Block-sparse partials (sparse_attention_forward.wgsl)
 * ------------------------------------------------------------------------------- */
typedef struct pkv_sparse_args {
  const void* q;               /* [num_queries, hq, head_dim], element type `dtype`;
                                  may be NULL when num_queries is 0 */
  const void* k_pages;         /* [num_pages, hkv, page_size, head_dim], `dtype` */
  const void* v_pages;
  const int32_t* edge_meta;    /* [num_edges, 5]: q_idx, h (kv head), blk, batch, block_len */
  const int32_t* block_tables; /* [num_seqs, max_pages]: page id or -1 (unmapped) */
  float* o_partial;            /* [num_edges*qhead, head_dim]; 16-byte aligned (the
                                  fp16 path stores 32 bytes a lane when it is 32-byte
                                  aligned, which is faster) */
  float* m_partial;            /* [num_edges*qhead] */
  float* l_partial;            /* [num_edges*qhead] */
  int32_t* device_status;      /* optional */
  int64_t num_queries;
  int64_t num_edges;
  int64_t num_seqs;
  int64_t max_pages;
  int64_t num_pages;
  int64_t qhead;               /* query heads per kv head; hq = hkv * qhead */
  int64_t hq;
  int64_t hkv;
  int64_t head_dim;
  int64_t block_size;          /* keys per block (<= page_size * pages_per_block) */
  int64_t page_size;
  int64_t pages_per_block;
  float softmax_scale;
  /* element type of q, k_pages, v_pages: PKV_F32 (0 is taken as PKV_F32) or PKV_F16.
     The partials are fp32 either way. */
  int32_t dtype;
  /* optional [num_queries] int32: absolute position of each query in its sequence
     (right-aligned causal; the page leaves it unimplemented). Key t of block blk takes
     part only when blk*block_size + t <= position; right-aligned queries of a sequence
     with n queries and used length u sit at u - n + i. NULL: no causal mask. */
  const int32_t* query_positions;
} pkv_sparse_args;

/* Host only: workspace bytes of pkv_sparse_attention_partials: the edge grouping and,
 * for fp32 calls whose shape runs on the tensor core (head_dim 64/128, block_size <= 64,
 * page_size a multiple of 8 with pages_per_block * page_size <= 64), the Q rows split
 * into fp16 (hi, lo) pairs: 4 * head_dim + 4 bytes per (query, head) row. */
int pkv_sparse_attention_partials_workspace_size(const pkv_sparse_args* args,
                                                 size_t* bytes);

/* One partial per (edge e, lane qh), index e*qhead + qh: query row q[q_idx, h*qhead+qh];
 * key t < block_len of block blk lives in page slot blk*pages_per_block + t/page_size
 * of the sequence's table row, row t % page_size; unmapped page -> score -1e30.
 * s = softmax_scale * <q, k>; m = max s (>= -1e30); weights exp(s - m) for s > -5e29
 * else 0; l = sum of weights; o = weighted sum of value rows (unnormalised).
 * block_len <= 0 -> (o = 0, m = -1e30, l = 0). No causal mask unless query_positions
 * is given. fp32 throughout for dtype PKV_F32.
 * The GPU form groups edges by (batch, kv head, block) so each K/V block is read
 * once for all edges that name it. Supported: head_dim in {64, 128}, block_size
 * <= 128, qhead <= 64.
 * dtype PKV_F16 (the page computes in fp32; this is the half-precision variant): scores
 * are fp16 products summed in fp32, the weights are computed in fp32 and summed into l,
 * and rounded once to fp16 for the weighted sum of value rows; the partials are fp32;
 * everything else as above.
 * fp32 on the tensor core: each Q row and each K / V block is scaled by a power of two
 * and split into fp16 (hi, lo) pairs, and every product is formed from three fp16 MMAs
 * with fp32 accumulation (hi*hi + hi*lo + lo*hi), about 2^-21 of |q||k| per score.
 * Supported for fp16: head_dim in {64, 128}, block_size <= 64, page_size a multiple of
 * 8 with pages_per_block * page_size <= 64; else PKV_ERR_UNSUPPORTED.
 * With query_positions the keys after the query's position take no part (they are not
 * read and flag nothing); an edge left with no key gets the empty partial. */
int pkv_sparse_attention_partials(const pkv_sparse_args* args, void* workspace,
                                  size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------------
 * Combine of (o, m, l) partials
 * ------------------------------------------------------------------------------- */
typedef struct pkv_combine_args {
  const float* o;              /* [num_partials, head_dim] unnormalised */
  const float* m;              /* [num_partials] running max (natural-log units) */
  const float* l;              /* [num_partials] sum of exp(s - m) */
  const int32_t* segment_offsets; /* [num_segments + 1] CSR over partial groups, or NULL */
  void* out;                   /* [num_segments*lanes, head_dim], dtype out_dtype */
  float* lse;                  /* optional [num_segments*lanes]: M + ln L, -inf if empty */
  int64_t num_segments;
  int64_t lanes;               /* partials per group (e.g. query heads per kv head) */
  int64_t head_dim;
  int64_t uniform_count;       /* groups per segment when segment_offsets == NULL */
  int32_t out_dtype;           /* PKV_F16 or PKV_F32 */
  int32_t reserved;
} pkv_combine_args;

/* Output row s*lanes + c merges partial rows e*lanes + c for groups e in
 * [off[s], off[s+1]) (or [s*uniform_count, (s+1)*uniform_count)): over partials with
 * l > 0, M = max m, w = exp(m - M), L = sum w*l, out = sum w*o / L, lse = M + ln L.
 * A partial with l == 0 is empty and its o row is not read. No non-empty partial:
 * out = 0, lse = -inf. Supported: head_dim in {64, 128}. */
int pkv_combine_partials(const pkv_combine_args* args, void* stream);

/* ---------------------------------------------------------------------------------
 * Runtime utilities
 * ------------------------------------------------------------------------------- */
int pkv_abi_version(void);
const char* pkv_status_string(int status);
/* sizeof of each argument struct, so a binding can check its layout. */
size_t pkv_sizeof_struct(const char* name);
/* Kernels this library has launched since load (all entry points, all streams). */
int64_t pkv_launch_count(void);
/* Per-kernel timing: when enabled, every launch is bracketed by CUDA events on its own
 * stream; pkv_profiler_query synchronises those events and returns the summed device
 * time (ms) and launch count of `kernel` ("scatter", "append", "plan", "decode",
 * "prefill", "combine", "sparse_group", "sparse_partials"). Not thread-safe. */
void pkv_profiler_enable(int on);

/* Testing hook for the give-up path of the tensor-core kernels' bounded waits (the
 * tcgen05 prefill and the two block-sparse partial kernels). The pages have no
 * counterpart. max_polls replaces the default poll bound of every such wait (0 restores
 * the default); with withhold_first_copy != 0 (which needs max_polls > 0) every CTA of
 * those kernels announces its first bulk copy (the first K box of its first prefill
 * tile, or its first K/V staging) on the copy's barrier but never issues it, so the wait
 * for it gives up with no copy or MMA of that data in flight. A CTA whose wait gave up
 * ORs PKV_DEV_TIMEOUT into device_status, waits (bounded) for what it did issue, frees
 * its tensor memory and returns; outputs it had not written stay unwritten. Applies to
 * calls made after it, process-wide; not thread-safe; for tests only. Returns PKV_OK,
 * or PKV_ERR_SHAPE for withhold_first_copy without a bound. */
int pkv_testing_wait_limit(uint32_t max_polls, int32_t withhold_first_copy);
void pkv_profiler_reset(void);
int pkv_profiler_query(const char* kernel, double* total_ms, int64_t* launches);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
