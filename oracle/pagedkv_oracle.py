"""CPU fp64 oracle for paged / block-sparse grouped-query attention.

TEST INFRASTRUCTURE ONLY. This module is the plain, slow statement of what the
attention path computes, used to check the CUDA library. Only the test suite, the
smoke check and the benchmark's CPU-baseline leg may import it; the library never
does, and nothing here is shared with the CUDA sources (no kernels, tables, helpers
or index code in common).

Sources (page title, then the part of the page each function follows):

* "com.microsoft.SparseAttention sparse-kv-append.wgsl.jinja" (WebGPU kernel page):
  the ``sparse_schedule`` macro (history length), the ``sparse_rotary`` macro
  (RoPE pair geometry and the rotation of one component) and the KV-append
  ``main`` entry point (BNSH destination index, packed [Q|K|V] offsets).
* "alice-llm src/shaders/sparse_attention_forward.wgsl" (docs.rs source page): the
  ``sparse_forward`` entry point and its layout comment block (edge_meta, paged K/V,
  partial layout, masked-block and unmapped-page sentinels).
* "com.microsoft.PagedAttention manifest.json" (WebGPU kernel page): operator
  inputs/outputs/attributes, the ``derive`` table (shapes, contract predicates,
  split count, scratch sizes) and the ScatterKV / AttendSplitK /
  AttendSplitKMerge pass list.

Where the pages are silent the oracle takes these readings (each is also listed in
the design notes): scale 0 means 1/sqrt(head_size); kv head of query head hq is
hq // (num_heads // kv_num_heads); a new token at absolute position pos sees keys
0..pos; a block-table entry outside [0, num_blocks) or a table column at or past
max_blocks is unmapped and its keys take no part; a negative slot is padding and is
skipped; positions at or past the BNSH cache length are skipped; partial o is
unnormalised and stats are (m, l) with natural-log exponent; in a combine a
partial with l == 0 is empty and contributes nothing; a row with no keys gives
output 0 and lse -inf.

Arithmetic is fp64 throughout; fp16 / fp32 inputs are widened exactly first.
Stored caches stay fp16 (a rotated key is rounded once to fp16 when written, the
one rounding the stored cache format forces).
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np

NEG_LARGE = -1.0e30          # masked-score / empty-partial sentinel of sparse_forward
HALF_NEG_LARGE = -5.0e29     # a score at or below this gets weight 0 (sparse_forward phase 2b)

# Status bits the oracle reports for invalid device-side data (mirrors no code: the
# meaning of each bit is part of the library's documented contract).
ST_BAD_BLOCK = 1      # block-table entry out of range / table column past max_blocks
ST_BAD_SLOT = 2       # slot_mapping entry past the pool
ST_BAD_POSITION = 4   # append position at or past the cache length
ST_BAD_SEQUENCE = 8   # cu / past inconsistent (negative length or past)
ST_BAD_EDGE = 16      # edge_meta field out of range


def _f64(x) -> np.ndarray:
    return np.asarray(x).astype(np.float64)


# ======================================================================================
# SparseAttention KV append (sparse-kv-append.wgsl.jinja)
# ======================================================================================
def past_sequence_length(total_sequence_length_0: int, key_total_b: int,
                         seq_len: int) -> int:
    """History length of batch row b (``sparse_schedule`` macro).

    Prompt mode is decided by the scalar total: when it equals the call's new-token
    count the history is zero for every row. Otherwise the history is the row's
    total minus the new-token count, or zero if that would be negative. The page
    reads both totals as u32, so a negative i32 total wraps to a huge value.
    """
    if (int(total_sequence_length_0) & 0xFFFFFFFF) == seq_len:
        return 0
    total = int(key_total_b) & 0xFFFFFFFF
    return total - seq_len if total >= seq_len else 0


def rotary_slot(d: int, half: int, interleaved: bool) -> int:
    """cos/sin column of component d (``sparse_rotary``: rotary_slot)."""
    if interleaved:
        return d // 2
    return d if d < half else d - half


def rotary_partner(d: int, half: int, interleaved: bool) -> int:
    """Other member of d's rotation pair (``sparse_rotary``: rotary_partner)."""
    if interleaved:
        return d + 1 if d % 2 == 0 else d - 1
    return d + half if d < half else d - half


def rotary_is_first(d: int, half: int, interleaved: bool) -> bool:
    """Whether d leads its pair (``sparse_rotary``: rotary_is_first)."""
    if interleaved:
        return d % 2 == 0
    return d < half


def rotary_value(own: float, partner: float, cs: float, sn: float, first: bool):
    """One rotated component (``sparse_rotary``: rotary_value): the leading member
    becomes own*cos - partner*sin, the trailing one own*cos + partner*sin."""
    return np.where(first, own * cs - partner * sn, own * cs + partner * sn)


def rotary_geometry(rotary_dim: int, interleaved: bool):
    """Per-component (slot, partner, is_first) arrays for d in [0, rotary_dim),
    built one component at a time from the three geometry functions above."""
    half = rotary_dim // 2
    d = range(rotary_dim)
    return (np.array([rotary_slot(i, half, interleaved) for i in d], dtype=np.int64),
            np.array([rotary_partner(i, half, interleaved) for i in d], dtype=np.int64),
            np.array([rotary_is_first(i, half, interleaved) for i in d], dtype=bool))


def rotate_rows(rows, positions, cos_cache, sin_cache, rotary_dim: int,
                interleaved: bool) -> np.ndarray:
    """Key rows [R, D] rotated at absolute positions [R]: every component d below
    rotary_dim becomes rotary_value(own = x[d], partner = x[partner(d)],
    cos[pos, slot(d)], sin[pos, slot(d)], is_first(d)); components at or above
    rotary_dim are copied (KV-append ``main``, rotary branch)."""
    x = _f64(rows)
    x = x.reshape(-1, x.shape[-1])
    pos = np.asarray(positions, dtype=np.int64).reshape(-1)
    out = x.copy()
    if rotary_dim <= 0:
        return out
    slot, partner, first = rotary_geometry(rotary_dim, interleaved)
    cs = _f64(cos_cache)[pos[:, None], slot[None, :]]
    sn = _f64(sin_cache)[pos[:, None], slot[None, :]]
    own = x[:, :rotary_dim]
    par = x[:, partner]
    out[:, :rotary_dim] = rotary_value(own, par, cs, sn, first[None, :])
    return out


def rotate_row(row, pos: int, cos_cache, sin_cache, rotary_dim: int,
               interleaved: bool) -> np.ndarray:
    """One key row rotated at absolute position ``pos`` (see rotate_rows)."""
    return rotate_rows(np.asarray(row)[None, :], [pos], cos_cache, sin_cache,
                       rotary_dim, interleaved)[0]


def kv_append_rotary(source, value, *, packed: bool, num_heads: int, kv_num_heads: int,
                     head_size: int, batch: int, seq_len: int, total_sequence_length,
                     key_total_sequence_lengths, cos_cache, sin_cache, rotary_dim: int,
                     interleaved: bool, present_key, present_value):
    """KV append into a [batch, kv_heads, max_cache_seq, head] cache (``main``).

    For every (batch b, kv head h, new token t): position = past(b) + t; the key row
    (rotated at that position when rotary_dim > 0) and the value row land at cache
    row ``position`` of (b, h). Packed rows hold [Q | K | V] with K starting after
    the num_heads query heads and V after the kv heads; separate input rows hold
    the kv heads directly. Rows that no new token lands on are untouched.

    Returns (key_out, value_out, written, status) where key_out / value_out are fp64
    copies of the caches after the append, ``written`` marks the (b, h, pos) rows the
    call wrote, and rotated components are left unrounded (fp64) so a comparison
    can apply the rotation tolerance; unrotated components equal their fp16 source.
    """
    Hq, Hkv, D = num_heads, kv_num_heads, head_size
    MCS = present_key.shape[2]
    key_out = _f64(present_key).copy()
    value_out = _f64(present_value).copy()
    written = np.zeros(present_key.shape[:3], dtype=bool)
    status = 0
    src = np.asarray(source)
    total0 = int(np.asarray(total_sequence_length).reshape(-1)[0])
    for b in range(batch):
        past = past_sequence_length(total0, int(key_total_sequence_lengths[b]), seq_len)
        for t in range(seq_len):
            pos = past + t
            row = b * seq_len + t
            if pos >= MCS:
                status |= ST_BAD_POSITION
                continue
            if packed:
                k_rows = src[row, Hq * D:(Hq + Hkv) * D].reshape(Hkv, D)
                v_rows = src[row, (Hq + Hkv) * D:(Hq + 2 * Hkv) * D].reshape(Hkv, D)
            else:
                k_rows = src[row, :Hkv * D].reshape(Hkv, D)
                v_rows = np.asarray(value)[row, :Hkv * D].reshape(Hkv, D)
            key_out[b, :, pos] = rotate_rows(k_rows, [pos] * Hkv, cos_cache, sin_cache,
                                             rotary_dim, interleaved)
            value_out[b, :, pos] = _f64(v_rows)
            written[b, :, pos] = True
    return key_out, value_out, written, status


def append_query_rotary(source, query, *, packed: bool, num_heads: int, kv_num_heads: int,
                        head_size: int, batch: int, seq_len: int, total_sequence_length,
                        key_total_sequence_lengths, cos_cache, sin_cache, rotary_dim: int,
                        interleaved: bool):
    """The query heads of the new tokens rotated at the same absolute position as their
    keys, with the same ``sparse_rotary`` rule and cos/sin tables.

    The append page rotates the key only; rotating the query at the token's position
    is the other half of rotary attention and uses nothing the page does not already
    define (history length from ``sparse_schedule``, pair geometry and rotation from
    ``sparse_rotary``). Query rows come from the packed row's leading num_heads
    heads, or from ``query`` [batch*seq_len, num_heads*head_size] in separate mode.
    A position without a cos/sin row (or rotary_dim == 0) leaves the row unrotated.
    Returns fp64 [batch*seq_len, num_heads*head_size], unrounded."""
    Hq, D = num_heads, head_size
    src = np.asarray(source if packed else query)
    out = _f64(src[:, :Hq * D]).copy()
    total0 = int(np.asarray(total_sequence_length).reshape(-1)[0])
    for b in range(batch):
        past = past_sequence_length(total0, int(key_total_sequence_lengths[b]), seq_len)
        for t in range(seq_len):
            pos = past + t
            row = b * seq_len + t
            if rotary_dim <= 0 or pos >= cos_cache.shape[0]:
                continue
            out[row] = rotate_rows(src[row, :Hq * D].reshape(Hq, D), [pos] * Hq, cos_cache,
                                   sin_cache, rotary_dim, interleaved).reshape(Hq * D)
    return out


# ======================================================================================
# PagedAttention (manifest.json)
# ======================================================================================
TUNABLES = dict(MAX_SPLITS=16, SPLIT_MIN_KEYS=128, SPLIT_TARGET_WORKGROUPS=1024)


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def pages_num_splits(token_count: int, kv_num_heads: int, max_blocks: int,
                     block_size: int, tunables: Optional[dict] = None) -> int:
    """Split count of the manifest's ``derive`` table: base workgroups = tokens x kv
    heads; cap = max(1, min(MAX_SPLITS, floor(max_blocks*block_size /
    SPLIT_MIN_KEYS))); splits = max(1, min(cap, ceilDiv(TARGET, max(1, base))))."""
    tn = dict(TUNABLES, **(tunables or {}))
    base = token_count * kv_num_heads
    key_ceiling = max_blocks * block_size
    cap = max(1, min(tn["MAX_SPLITS"], key_ceiling // tn["SPLIT_MIN_KEYS"]))
    return max(1, min(cap, ceil_div(tn["SPLIT_TARGET_WORKGROUPS"], max(1, base))))


def pages_split_scratch_bytes(token_count: int, num_heads: int, head_size: int,
                              num_splits: int):
    """(partialOut bytes, partialStats bytes) of the manifest's split variants."""
    return (token_count * num_heads * num_splits * head_size * 4,
            2 * token_count * num_heads * num_splits * 4)


def paged_contract(*, query_shape, key_shape, value_shape, key_cache_shape,
                   value_cache_shape, cu_shape, past_shape, block_table_shape,
                   slot_mapping_shape, output_shape, num_heads, kv_num_heads,
                   dtypes: dict, is_causal: int = 1) -> dict:
    """The manifest's contract predicates on tensor ranks, shapes and dtypes.

    Returns a dict of predicate name -> bool, plus ``pagedContractOk`` and the
    input mode ('separate', 'packed' or None). ``dtypes`` maps query/key/value/
    key_cache/value_cache/output to dtype names ('float16', ...) for the tensors
    that are present. Absent optional tensors have shape None.
    """
    def rank(s):
        return None if s is None else len(s)

    def dim(s, i):
        return s[i]

    r = {}
    kc, vc = key_cache_shape, value_cache_shape
    head_size = dim(kc, 3) if rank(kc) == 4 else 0
    block_size = dim(kc, 1) if rank(kc) == 4 else 0
    q_hidden = num_heads * head_size
    kv_hidden = kv_num_heads * head_size
    packed_stride = q_hidden + 2 * kv_hidden
    token_count = dim(query_shape, 0)
    r["cacheShapeOk"] = (rank(kc) == 4 and rank(vc) == 4 and tuple(vc) == tuple(kc)
                         and dim(kc, 2) == kv_num_heads and block_size > 0
                         and head_size > 0
                         and dtypes.get("key_cache") == dtypes.get("query")
                         and dtypes.get("value_cache") == dtypes.get("query"))
    r["headLayoutOk"] = (num_heads > 0 and kv_num_heads > 0
                         and num_heads % kv_num_heads == 0)
    batch = (dim(cu_shape, 0) - 1) if rank(cu_shape) == 1 else -1
    max_blocks = dim(block_table_shape, 1) if rank(block_table_shape) == 2 else 0
    r["scheduleShapeOk"] = (rank(cu_shape) == 1 and rank(past_shape) == 1
                            and rank(block_table_shape) == 2 and batch >= 1
                            and dim(past_shape, 0) == batch
                            and dim(block_table_shape, 0) == batch and max_blocks >= 1)
    r["ioShapeOk"] = (rank(query_shape) == 2 and rank(output_shape) == 2
                      and dim(output_shape, 0) == token_count
                      and dim(output_shape, 1) == q_hidden
                      and dtypes.get("output") == dtypes.get("query")
                      and dtypes.get("query") == "float16")
    have_k = key_shape is not None
    have_v = value_shape is not None
    r["separateKv"] = (have_k and have_v and rank(key_shape) == 2
                       and rank(value_shape) == 2 and dim(key_shape, 0) == token_count
                       and dim(value_shape, 0) == token_count
                       and dim(key_shape, 1) == kv_hidden
                       and dim(value_shape, 1) == kv_hidden
                       and dtypes.get("key") == dtypes.get("query")
                       and dtypes.get("value") == dtypes.get("query")
                       and dim(query_shape, 1) == q_hidden)
    r["packedKv"] = (not have_k and not have_v and dim(query_shape, 1) == packed_stride)
    if slot_mapping_shape is not None:
        r["slotShapeOk"] = (rank(slot_mapping_shape) == 1
                            and dim(slot_mapping_shape, 0) == token_count)
    else:
        r["slotShapeOk"] = True
    r["causalOk"] = (is_causal == 1)
    r["pagedContractOk"] = (r["cacheShapeOk"] and r["headLayoutOk"]
                            and r["scheduleShapeOk"] and r["ioShapeOk"]
                            and r["slotShapeOk"])
    r["mode"] = "separate" if r["separateKv"] else ("packed" if r["packedKv"] else None)
    return r


def sequence_map(cu_seqlens, past_seqlens, num_tokens: Optional[int] = None):
    """Token i in [cu[b], cu[b+1]) belongs to sequence b as new token t = i - cu[b]
    at absolute position past[b] + t. Returns (entries, status): entries[i] is
    (b, t, pos) or None for a token no valid sequence covers.

    Reading for data the manifest does not check: sequence b is valid when
    0 <= cu[b] <= cu[b+1] <= num_tokens and past[b] >= 0; an invalid sequence
    contributes no tokens and sets ST_BAD_SEQUENCE. Uncovered tokens (e.g. padding
    after cu[batch]) are not an error."""
    cu = [int(x) for x in cu_seqlens]
    past = [int(x) for x in past_seqlens]
    T = cu[-1] if num_tokens is None else int(num_tokens)
    out = [None] * T
    status = 0
    for b in range(len(past)):
        lo, hi = cu[b], cu[b + 1]
        if not (0 <= lo <= hi <= T and past[b] >= 0):
            status |= ST_BAD_SEQUENCE
            continue
        for i in range(lo, hi):
            out[i] = (b, i - lo, past[b] + i - lo)
    return out, status


def split_new_kv(case_query, case_key, case_value, num_heads, kv_num_heads, head_size):
    """New K and V rows as [T, kv_heads, head] arrays: from separate inputs, or from
    packed [Q | K | V] query rows (K after the query heads, V after the kv heads)."""
    Hq, Hkv, D = num_heads, kv_num_heads, head_size
    T = case_query.shape[0]
    if case_key is None:
        k = case_query[:, Hq * D:(Hq + Hkv) * D]
        v = case_query[:, (Hq + Hkv) * D:(Hq + 2 * Hkv) * D]
    else:
        k, v = case_key, case_value
    return (np.asarray(k).reshape(T, Hkv, D), np.asarray(v).reshape(T, Hkv, D),
            np.asarray(case_query)[:, :Hq * D].reshape(T, Hq, D))


def paged_scatter(k_new, v_new, key_cache, value_cache, cu_seqlens, past_seqlens,
                  block_table, slot_mapping=None, cos_cache=None, sin_cache=None,
                  rotary_dim: int = 0, rotary_interleaved: bool = False):
    """The ScatterKV pass: write each new token's K and V rows into the paged cache.

    The destination of token i is given by slot_mapping[i] (blk = slot //
    block_size, offset = slot % block_size; a negative slot is padding) when a slot
    mapping is present, else by the block table at the token's absolute position
    (blk = block_table[b, pos // block_size], offset = pos % block_size). When
    rotary_dim > 0 the key row is first rotated at its absolute position with the
    append page's rotation rule and rounded once to fp16. Returns (key_cache,
    value_cache, status) as new fp16 arrays. Readings for unchecked data: a slot past
    the pool, a table column past max_blocks or a block id outside the pool skips the
    token (status bit); with rotation, a position past the cos/sin table skips it.
    """
    kc = np.array(key_cache, copy=True)
    vc = np.array(value_cache, copy=True)
    NB, BS = kc.shape[0], kc.shape[1]
    MB = block_table.shape[1]
    smap, status = sequence_map(cu_seqlens, past_seqlens, k_new.shape[0])
    for i, entry in enumerate(smap):
        if entry is None:
            continue
        b, t, pos = entry
        if slot_mapping is not None:
            slot = int(slot_mapping[i])
            if slot < 0:
                continue
            blk, off = slot // BS, slot % BS
            if blk >= NB:
                status |= ST_BAD_SLOT
                continue
        else:
            col = pos // BS
            if pos < 0 or col >= MB:
                status |= ST_BAD_BLOCK
                continue
            blk, off = int(block_table[b, col]), pos % BS
            if blk < 0 or blk >= NB:
                status |= ST_BAD_BLOCK
                continue
        k_row = k_new[i]
        if rotary_dim > 0 and pos >= cos_cache.shape[0]:
            status |= ST_BAD_POSITION      # no cos/sin row for this position
            continue
        if rotary_dim > 0:
            k_row = rotate_rows(k_new[i], [pos] * k_new.shape[1], cos_cache, sin_cache,
                                rotary_dim, rotary_interleaved).astype(np.float16)
        kc[blk, off] = k_row
        vc[blk, off] = v_new[i]
    return kc, vc, status


def gather_sequence_kv(key_cache, value_cache, block_table_row, n_keys: int):
    """Keys/values 0..n_keys-1 of one sequence read through its block-table row.

    Returns (K [n, Hkv, D] fp64, V [n, Hkv, D] fp64, valid [n] bool); a key whose
    table column is past the row or whose block id is outside the pool is invalid
    (its K/V rows are zero and it must be excluded)."""
    NB, BS = key_cache.shape[0], key_cache.shape[1]
    j = np.arange(n_keys)
    col = j // BS
    valid = col < block_table_row.shape[0]
    blk = np.full(n_keys, -1, dtype=np.int64)
    blk[valid] = block_table_row[col[valid]]
    valid &= (blk >= 0) & (blk < NB)
    K = np.zeros((n_keys,) + key_cache.shape[2:], dtype=np.float64)
    V = np.zeros_like(K)
    K[valid] = key_cache[blk[valid], j[valid] % BS]
    V[valid] = value_cache[blk[valid], j[valid] % BS]
    return K, V, valid


def attention_rows(q_rows, K, V, valid, limits, scale: float,
                   return_weights: bool = False, row_chunk: int = 256):
    """Plain softmax attention for several query rows over one key/value sequence.

    Row r attends to key j iff valid[j] and j <= limits[r]: s_rj = scale * <q_r, k_j>,
    p_r = softmax over its visible keys, out_r = sum_j p_rj v_j. A row with no
    visible key gives zeros. Rows are evaluated a few hundred at a time only to
    bound memory; every row is computed independently by the definition.
    """
    q_rows = _f64(q_rows)
    R, n = q_rows.shape[0], K.shape[0]
    out = np.zeros((R, V.shape[-1]))
    weights = np.zeros((R, n)) if return_weights else None
    j = np.arange(n)
    limits = np.asarray(limits, dtype=np.int64)
    for r0 in range(0, R, row_chunk):
        r1 = min(R, r0 + row_chunk)
        vis = valid[None, :] & (j[None, :] <= limits[r0:r1, None])
        s = scale * (q_rows[r0:r1] @ K.T)
        s = np.where(vis, s, -np.inf)
        row_max = s.max(axis=1, keepdims=True)
        any_vis = vis.any(axis=1)
        row_max[~any_vis] = 0.0
        w = np.where(vis, np.exp(s - row_max), 0.0)
        denom = w.sum(axis=1, keepdims=True)
        denom[~any_vis] = 1.0
        w /= denom
        out[r0:r1] = w @ V
        if return_weights:
            weights[r0:r1] = w
    return (out, weights) if return_weights else out


def paged_attention(query, key, value, key_cache, value_cache, cu_seqlens,
                    past_seqlens, block_table, slot_mapping=None, *, num_heads: int,
                    kv_num_heads: int, scale: float = 0.0, cos_cache=None,
                    sin_cache=None, rotary_dim: int = 0,
                    rotary_interleaved: bool = False, tokens: Optional[Sequence] = None,
                    rotary_query: bool = False):
    """The PagedAttention operator: ScatterKV, then causal GQA attention of every new
    token over its sequence's keys read back through the block table.

    Query head hq uses kv head hq // (num_heads // kv_num_heads). Token i of
    sequence b at absolute position pos sees keys 0..pos. ``tokens`` restricts the
    attention to a subset of token indices (the scatter always runs in full).
    With ``rotary_query`` (and rotary_dim > 0) every query head of token i is first
    rotated at pos with the key's rotation rule and tables (unrounded); a position
    without a cos/sin row leaves the query unrotated.

    Returns (out [T, Hq*D] fp64 with rows outside ``tokens`` left zero,
    key_cache, value_cache, status).
    """
    Hq, Hkv = num_heads, kv_num_heads
    D = key_cache.shape[3]
    G = Hq // Hkv
    scale = scale if scale != 0.0 else 1.0 / math.sqrt(D)
    k_new, v_new, q_all = split_new_kv(query, key, value, Hq, Hkv, D)
    kc, vc, status = paged_scatter(k_new, v_new, key_cache, value_cache, cu_seqlens,
                                   past_seqlens, block_table, slot_mapping, cos_cache,
                                   sin_cache, rotary_dim, rotary_interleaved)
    T = q_all.shape[0]
    out = np.zeros((T, Hq, D), dtype=np.float64)
    smap, _ = sequence_map(cu_seqlens, past_seqlens, T)
    if rotary_query and rotary_dim > 0:
        q_all = _f64(q_all).copy()
        for i in range(T):
            if smap[i] is not None and smap[i][2] < cos_cache.shape[0]:
                q_all[i] = rotate_rows(q_all[i], [smap[i][2]] * Hq, cos_cache, sin_cache,
                                       rotary_dim, rotary_interleaved)
    wanted = range(T) if tokens is None else tokens
    by_seq = {}
    for i in wanted:
        if smap[i] is not None:
            by_seq.setdefault(smap[i][0], []).append(i)
    for b, rows in by_seq.items():
        n_keys = max(smap[i][2] for i in rows) + 1
        if n_keys <= 0:
            continue
        if n_keys > block_table.shape[1] * kc.shape[1]:
            status |= ST_BAD_BLOCK
        K, V, valid = gather_sequence_kv(kc, vc, block_table[b], n_keys)
        if not valid.all():
            status |= ST_BAD_BLOCK
        limits = np.array([smap[i][2] for i in rows], dtype=np.int64)
        for h in range(Hkv):
            heads = list(range(h * G, (h + 1) * G))
            q_rows = _f64(q_all[rows][:, heads]).reshape(len(rows) * G, D)
            res = attention_rows(q_rows, K[:, h], V[:, h], valid,
                                 np.repeat(limits, G), scale)
            out[np.asarray(rows)[:, None], np.asarray(heads)[None, :]] = \
                res.reshape(len(rows), G, D)
    return out.reshape(T, Hq * D), kc, vc, status


def attention_partial(q, K, V, visible, scale: float):
    """(o, m, l) of one query row over a key subset: m = max score, l = sum of
    exp(s - m), o = sum exp(s - m) v (unnormalised). No visible key gives the empty
    partial (0, NEG_LARGE, 0)."""
    if not np.any(visible):
        return np.zeros(V.shape[-1]), NEG_LARGE, 0.0
    s = scale * (K[visible] @ _f64(q))
    m = s.max()
    p = np.exp(s - m)
    return p @ V[visible], float(m), float(p.sum())


# ======================================================================================
# Block-sparse forward (sparse_attention_forward.wgsl)
# ======================================================================================
def sparse_partial(q_buf, k_pages, v_pages, meta, block_tables, qh: int, *, qhead: int,
                   hq: int, head_dim: int, block_size: int, page_size: int,
                   pages_per_block: int, softmax_scale: float, query_positions=None):
    """(o, m, l, status) of one partial = (edge, query-head lane qh) (``sparse_forward``).

    edge meta = [q_idx, h, blk, batch, block_len]; block_len <= 0 gives the empty
    partial (o = 0, m = -1e30, l = 0). Key t < block_len lives in page slot
    blk * pages_per_block + t // page_size of the sequence's block-table row, at row
    t % page_size; an unmapped page (-1) gives score -1e30. m is the max score
    (never below -1e30), weights are exp(s - m) for scores above -5e29 and 0
    otherwise, l their sum and o the weighted sum of value rows (unnormalised).

    Readings for data the page leaves unchecked: block_len above block_size is
    clipped to block_size, and a page slot past the table row or a page id past
    the pool counts as unmapped; each sets a status bit. An edge with block_len > 0
    whose q_idx, head, batch or block lies outside the tensors gets the empty
    partial and a status bit.

    Right-aligned causal (the page leaves it unimplemented): with ``query_positions``
    (the absolute position of each query in its sequence; right-aligned queries of a
    sequence sit at used_len - n_queries + i), key t of the block (absolute position
    blk * block_size + t) takes part only when that position is at most the query's.
    Keys that take no part are not looked up (and flag nothing); a partial with no
    key taking part is the empty partial.
    """
    q_idx, h, blk, batch, block_len = (int(x) for x in meta)
    status = 0
    D = head_dim
    if block_len > block_size:
        block_len = block_size
        status |= ST_BAD_EDGE
    if block_len <= 0:
        return np.zeros(D), NEG_LARGE, 0.0, status
    if not (0 <= q_idx < q_buf.shape[0] and 0 <= h * qhead + qh < q_buf.shape[1]
            and 0 <= batch < block_tables.shape[0] and blk >= 0
            and blk * pages_per_block < block_tables.shape[1]):
        return np.zeros(D), NEG_LARGE, 0.0, status | ST_BAD_EDGE
    keys = range(block_len)
    if query_positions is not None:
        pos = int(query_positions[q_idx])
        keys = [t for t in keys if blk * block_size + t <= pos]
        if not keys:
            return np.zeros(D), NEG_LARGE, 0.0, status
    q = _f64(q_buf[q_idx, h * qhead + qh])
    num_pages = k_pages.shape[0]
    max_pages = block_tables.shape[1]
    scores = np.full(block_len, NEG_LARGE)
    rows_k = np.zeros((block_len, D))
    rows_v = np.zeros((block_len, D))
    taking_part = np.zeros(block_len, dtype=bool)
    for t in keys:
        taking_part[t] = True
        page_slot = blk * pages_per_block + t // page_size
        page_id = int(block_tables[batch, page_slot]) if page_slot < max_pages else -1
        if page_slot >= max_pages or page_id >= num_pages:
            status |= ST_BAD_EDGE
            page_id = -1
        if page_id >= 0:
            rows_k[t] = k_pages[page_id, h, t % page_size]
            rows_v[t] = v_pages[page_id, h, t % page_size]
            scores[t] = float(rows_k[t] @ q) * softmax_scale
    scores = scores[taking_part]
    rows_v = rows_v[taking_part]
    m = max(NEG_LARGE, float(scores.max()))
    p = np.where(scores > HALF_NEG_LARGE, np.exp(scores - m), 0.0)
    l = float(p.sum())
    o = p @ rows_v
    return o, m, l, status


def sparse_attention_partials(case_q, k_pages, v_pages, edge_meta, block_tables, *,
                              qhead: int, hq: int, head_dim: int, block_size: int,
                              page_size: int, pages_per_block: int, softmax_scale: float,
                              edges: Optional[Sequence[int]] = None, query_positions=None):
    """All partials (or those of the listed edges): partial index = edge * qhead + qh;
    o [P, D], m [P], l [P] fp64 plus the OR of status bits. Partials of unlisted
    edges are left as NaN. ``query_positions``: right-aligned causal mask (see
    sparse_partial)."""
    E = edge_meta.shape[0]
    P = E * qhead
    o = np.full((P, head_dim), np.nan)
    m = np.full(P, np.nan)
    l = np.full(P, np.nan)
    status = 0
    for e in (range(E) if edges is None else edges):
        for qh in range(qhead):
            oo, mm, ll, st = sparse_partial(
                case_q, k_pages, v_pages, edge_meta[e], block_tables, qh, qhead=qhead,
                hq=hq, head_dim=head_dim, block_size=block_size, page_size=page_size,
                pages_per_block=pages_per_block, softmax_scale=softmax_scale,
                query_positions=query_positions)
            i = e * qhead + qh
            o[i], m[i], l[i] = oo, mm, ll
            status |= st
    return o, m, l, status


# ======================================================================================
# Log-sum-exp combine (AttendSplitKMerge / merge of sparse partials)
# ======================================================================================
def combine_rows(o_rows, m_rows, l_rows):
    """Merge partials of one output row: over the non-empty partials (l > 0),
    M = max m, w_i = exp(m_i - M), L = sum w_i l_i, out = sum w_i o_i / L,
    lse = M + ln L. No non-empty partial: out = 0, lse = -inf."""
    o_rows = _f64(o_rows)
    m_rows = _f64(m_rows)
    l_rows = _f64(l_rows)
    keep = l_rows > 0
    if not np.any(keep):
        return np.zeros(o_rows.shape[-1]), -math.inf
    M = m_rows[keep].max()
    w = np.exp(m_rows[keep] - M)
    L = float((w * l_rows[keep]).sum())
    out = (w[:, None] * o_rows[keep]).sum(axis=0) / L
    return out, M + math.log(L)


def combine_partials(o, m, l, segment_offsets, lanes: int):
    """Combine over CSR segments: segment s, lane c merges partial rows
    e * lanes + c for e in [off[s], off[s+1]) into output row s * lanes + c.
    Returns (out [S*lanes, D], lse [S*lanes])."""
    off = [int(x) for x in segment_offsets]
    S = len(off) - 1
    D = o.shape[-1]
    out = np.zeros((S * lanes, D))
    lse = np.zeros(S * lanes)
    for s in range(S):
        for c in range(lanes):
            rows = [e * lanes + c for e in range(off[s], off[s + 1])]
            if rows:
                out[s * lanes + c], lse[s * lanes + c] = combine_rows(o[rows], m[rows],
                                                                      l[rows])
            else:
                lse[s * lanes + c] = -math.inf
    return out, lse
