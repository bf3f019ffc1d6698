"""Seeded synthetic inputs for the paged / block-sparse attention path.

This module only draws inputs: random values, block pools, block tables, sequence
lengths, edge lists and the cos/sin tables that the append pass reads. It computes no
attention, no rotation and no softmax, so the CUDA path and the CPU oracle can both
take their inputs from here without sharing any of the method's arithmetic.

All values are drawn with numpy's PCG64 generator from a fixed seed. N(0,1) values are
drawn by inverse-CDF lookup: a 16-bit uniform selects one of 65536 equiprobable normal
quantiles, stored in the tensor's dtype (fp16 rounding is nearest-even). This keeps the
1 GB caches of the decode workload quick to draw.

Workloads (shapes follow the operator pages):

* ``tiny_decode``      - 2 sequences, 4 query heads over 2 kv heads, head size 64.
* ``append_rotary``    - KV append with RoPE into a [batch, kv_heads, max_seq, head]
                         cache, packed [Q|K|V] rows, decode or prompt mode.
* ``llama8b_decode``   - 64 decoding sequences, 32 query / 8 kv heads, head size 128,
                         16-token blocks, contexts uniform in [512, 8192].
* ``varlen_mixed``     - 16 sequences, 8 prefilling 1..2048 tokens and 8 decoding one,
                         pasts uniform in [0, 4096], 32-token blocks, slot mapping.
* ``block_sparse``     - fp32 block-sparse edge list over paged K/V of layout
                         [num_pages, kv_heads, page_size, head].
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np


def rng_for(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


_CHUNKS = 16          # fixed split, so results do not depend on the thread count
_TABLES = {}


def _normal_table(dtype) -> np.ndarray:
    """65536 equiprobable N(0,1) quantiles (inverse CDF at (i + 0.5) / 65536)."""
    key = np.dtype(dtype).str
    if key not in _TABLES:
        from scipy.special import ndtri
        _TABLES[key] = ndtri((np.arange(65536) + 0.5) / 65536.0).astype(dtype)
    return _TABLES[key]


def _normal(rng: np.random.Generator, shape, dtype) -> np.ndarray:
    """N(0,1) draws: a 16-bit uniform per element picks one of 65536 equiprobable
    normal quantiles. The 16 chunks use child seeds of one draw from ``rng`` and are
    filled on a thread pool (uniform generation and the lookup release the GIL)."""
    from concurrent.futures import ThreadPoolExecutor
    table = _normal_table(dtype)
    n = int(np.prod(shape, dtype=np.int64))
    out = np.empty(n, dtype=dtype)
    children = np.random.SeedSequence(int(rng.integers(0, 2**63 - 1))).spawn(_CHUNKS)
    step = (n + _CHUNKS - 1) // _CHUNKS

    def fill(i):
        lo, hi = i * step, min(n, (i + 1) * step)
        if lo >= hi:
            return
        g = np.random.Generator(np.random.PCG64(children[i]))
        idx = np.frombuffer(g.bytes(2 * (hi - lo)), dtype=np.uint16)
        np.take(table, idx, out=out[lo:hi])

    if n < (1 << 20):
        for i in range(_CHUNKS):
            fill(i)
    else:
        with ThreadPoolExecutor(min(_CHUNKS, 8)) as ex:
            list(ex.map(fill, range(_CHUNKS)))
    return out.reshape(shape)


def normal_f16(rng: np.random.Generator, shape) -> np.ndarray:
    return _normal(rng, shape, np.float16)


def normal_f32(rng: np.random.Generator, shape) -> np.ndarray:
    return _normal(rng, shape, np.float32)


def rope_tables(max_positions: int, rotary_dim: int, theta: float = 10000.0):
    """cos/sin tables of shape [max_positions, rotary_dim // 2], stored as fp16.

    Entry (p, i) holds cos / sin of p * theta ** (-2 i / rotary_dim), evaluated in
    fp64 and rounded once to fp16. This is the standard RoPE frequency table; the
    pages only say that the append pass reads it, not how it is filled.
    """
    half = rotary_dim // 2
    inv_freq = theta ** (-(2.0 * np.arange(half, dtype=np.float64)) / rotary_dim)
    ang = np.arange(max_positions, dtype=np.float64)[:, None] * inv_freq[None, :]
    return np.cos(ang).astype(np.float16), np.sin(ang).astype(np.float16)


# --------------------------------------------------------------------------------------
# Paged attention inputs (PagedAttention operator contract)
# --------------------------------------------------------------------------------------
@dataclass
class PagedCase:
    num_heads: int
    kv_num_heads: int
    head_size: int
    block_size: int
    query: np.ndarray                  # [T, Hq*D] separate, or [T, (Hq+2Hkv)*D] packed
    key: Optional[np.ndarray]          # [T, Hkv*D] or None (packed)
    value: Optional[np.ndarray]        # [T, Hkv*D] or None (packed)
    key_cache: np.ndarray              # [NB, BS, Hkv, D] fp16
    value_cache: np.ndarray            # [NB, BS, Hkv, D] fp16
    cu_seqlens: np.ndarray             # [B+1] int32
    past_seqlens: np.ndarray           # [B] int32
    block_table: np.ndarray            # [B, MB] int32, -1 = unused
    slot_mapping: Optional[np.ndarray]  # [T] int32 or None
    scale: float
    cos_cache: Optional[np.ndarray] = None   # [P, R/2] fp16, rotary of new keys
    sin_cache: Optional[np.ndarray] = None
    rotary_dim: int = 0
    rotary_interleaved: bool = False

    @property
    def num_tokens(self) -> int:
        return int(self.query.shape[0])

    @property
    def batch(self) -> int:
        return int(self.past_seqlens.shape[0])

    @property
    def num_blocks(self) -> int:
        return int(self.key_cache.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def packed(self) -> bool:
        return self.key is None

    def context_lengths(self) -> np.ndarray:
        """Keys visible to the last new token of each sequence: past + new."""
        new = np.diff(self.cu_seqlens.astype(np.int64))
        return self.past_seqlens.astype(np.int64) + new


def paged_case(seed: int, *, num_heads: int, kv_num_heads: int, head_size: int,
               block_size: int, past, new_tokens, packed: bool = False,
               use_slot_mapping: bool = False, extra_blocks: int = 0,
               max_blocks: Optional[int] = None, scale: Optional[float] = None,
               rotary_dim: int = 0, rotary_interleaved: bool = False,
               theta: float = 10000.0, fill_cache: bool = True) -> PagedCase:
    """Random paged-attention inputs.

    Each sequence b owns ceil((past_b + new_b) / block_size) physical blocks, drawn
    from a seeded permutation of a pool of ``sum(need) + extra_blocks`` blocks; the
    rest of its block-table row is -1. Cache contents (including rows that the new
    tokens will overwrite) are N(0,1) fp16 draws.
    """
    rng = rng_for(seed)
    past = np.asarray(past, dtype=np.int64)
    new = np.asarray(new_tokens, dtype=np.int64)
    assert past.shape == new.shape
    B = past.shape[0]
    BS = block_size
    totals = past + new
    need = (totals + BS - 1) // BS
    MB = int(max_blocks) if max_blocks is not None else max(1, int(need.max()))
    assert MB >= need.max()
    NB = int(need.sum()) + int(extra_blocks)
    NB = max(NB, 1)
    perm = rng.permutation(NB).astype(np.int32)
    block_table = np.full((B, MB), -1, dtype=np.int32)
    cursor = 0
    for b in range(B):
        n = int(need[b])
        block_table[b, :n] = perm[cursor:cursor + n]
        cursor += n
    Hq, Hkv, D = num_heads, kv_num_heads, head_size
    if fill_cache:
        key_cache = normal_f16(rng, (NB, BS, Hkv, D))
        value_cache = normal_f16(rng, (NB, BS, Hkv, D))
    else:
        key_cache = np.zeros((NB, BS, Hkv, D), dtype=np.float16)
        value_cache = np.zeros((NB, BS, Hkv, D), dtype=np.float16)
    T = int(new.sum())
    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(new)
    if packed:
        query = normal_f16(rng, (T, (Hq + 2 * Hkv) * D))
        key = value = None
    else:
        query = normal_f16(rng, (T, Hq * D))
        key = normal_f16(rng, (T, Hkv * D))
        value = normal_f16(rng, (T, Hkv * D))
    slot_mapping = None
    if use_slot_mapping:
        # A slot is the flat row index blk * block_size + offset of the pool row
        # that the block table assigns to the token's absolute position.
        slot_mapping = np.empty(T, dtype=np.int32)
        i = 0
        for b in range(B):
            for t in range(int(new[b])):
                pos = int(past[b]) + t
                slot_mapping[i] = int(block_table[b, pos // BS]) * BS + pos % BS
                i += 1
    cos = sin = None
    if rotary_dim:
        cos, sin = rope_tables(int(totals.max()) + 1, rotary_dim, theta)
    return PagedCase(
        num_heads=Hq, kv_num_heads=Hkv, head_size=D, block_size=BS,
        query=query, key=key, value=value, key_cache=key_cache, value_cache=value_cache,
        cu_seqlens=cu, past_seqlens=past.astype(np.int32), block_table=block_table,
        slot_mapping=slot_mapping,
        scale=float(scale) if scale is not None else 1.0 / float(np.sqrt(D)),
        cos_cache=cos, sin_cache=sin, rotary_dim=int(rotary_dim),
        rotary_interleaved=bool(rotary_interleaved))


def tiny_decode(seed: int = 1) -> PagedCase:
    """Two decoding sequences with pasts {37, 90}; 4 query heads on 2 kv heads, D=64,
    16-token blocks from a pool of 16 physical blocks; separate K/V; scale 1/8."""
    return paged_case(seed, num_heads=4, kv_num_heads=2, head_size=64, block_size=16,
                      past=[37, 90], new_tokens=[1, 1], extra_blocks=16 - 9,
                      scale=1.0 / 8.0)


def llama8b_decode(seed: int = 3, batch: int = 64, min_ctx: int = 512,
                   max_ctx: int = 8192, rotary: bool = False,
                   fill_cache: bool = True) -> PagedCase:
    """Llama-3-8B-shaped decode: 32 query heads, 8 kv heads, head size 128, 16-token
    blocks, one new token per sequence, context n_b ~ U[min_ctx, max_ctx] so that
    past_b = n_b - 1; physical blocks are a random permutation of the pool."""
    rng = rng_for(seed)
    ctx = rng.integers(min_ctx, max_ctx + 1, size=batch)
    past = ctx - 1
    return paged_case(seed + 1000, num_heads=32, kv_num_heads=8, head_size=128,
                      block_size=16, past=past, new_tokens=np.ones(batch, np.int64),
                      max_blocks=(max_ctx + 15) // 16,
                      rotary_dim=128 if rotary else 0, fill_cache=fill_cache)


def varlen_mixed(seed: int = 4, n_prefill: int = 8, n_decode: int = 8,
                 max_new: int = 2048, max_past: int = 4096) -> PagedCase:
    """Mixed varlen batch: n_prefill sequences with U{1..max_new} new tokens and
    n_decode sequences with one, in seeded order; pasts U{0..max_past}; 32-token
    blocks; new K/V scattered through slot_mapping."""
    rng = rng_for(seed)
    new = np.concatenate([rng.integers(1, max_new + 1, size=n_prefill),
                          np.ones(n_decode, dtype=np.int64)])
    new = new[rng.permutation(new.shape[0])]
    past = rng.integers(0, max_past + 1, size=new.shape[0])
    return paged_case(seed + 1000, num_heads=32, kv_num_heads=8, head_size=128,
                      block_size=32, past=past, new_tokens=new,
                      max_blocks=(max_past + max_new + 31) // 32,
                      use_slot_mapping=True)


# --------------------------------------------------------------------------------------
# KV append + RoPE into a [batch, kv_heads, max_cache_seq, head] cache
# --------------------------------------------------------------------------------------
@dataclass
class AppendCase:
    num_heads: int
    kv_num_heads: int
    head_size: int
    batch: int
    seq_len: int
    packed: bool
    source: np.ndarray                  # packed [B*S, (Hq+2Hkv)*D] or key [B*S, Hkv*D]
    value: Optional[np.ndarray]         # [B*S, Hkv*D] when not packed
    total_sequence_length: np.ndarray   # [1] int32
    key_total_sequence_lengths: np.ndarray  # [B] int32
    cos_cache: np.ndarray               # [P, R/2] fp16
    sin_cache: np.ndarray
    rotary_dim: int
    interleaved: bool
    present_key: np.ndarray             # [B, Hkv, MCS, D] fp16 (prior contents)
    present_value: np.ndarray


def append_rotary(seed: int = 2, *, mode: str = "decode", interleaved: bool = False,
                  batch: int = 4, num_heads: int = 32, kv_num_heads: int = 8,
                  head_size: int = 128, rotary_dim: int = 128,
                  max_cache_seq: int = 4096, prompt_len: int = 512,
                  max_past: int = 4000, packed: bool = True,
                  theta: float = 10000.0) -> AppendCase:
    """KV-append workload. decode: one new token, past_b ~ U{0..max_past},
    key totals past_b + 1 and the scalar total = max over the batch; prompt:
    prompt_len new tokens with no past and scalar total = prompt_len. The cache is
    pre-filled with N(0,1) fp16 so untouched rows can be checked bit for bit."""
    rng = rng_for(seed)
    B, Hq, Hkv, D = batch, num_heads, kv_num_heads, head_size
    if mode == "decode":
        S = 1
        past = rng.integers(0, max_past + 1, size=B)
        totals = past + S
        total_scalar = int(totals.max())
        if total_scalar == S:   # keep decode mode distinct from prompt mode
            totals[0] += 1
            total_scalar = int(totals.max())
    elif mode == "prompt":
        S = prompt_len
        totals = np.full(B, S, dtype=np.int64)
        total_scalar = S
    else:
        raise ValueError(mode)
    if packed:
        source = normal_f16(rng, (B * S, (Hq + 2 * Hkv) * D))
        value = None
    else:
        source = normal_f16(rng, (B * S, Hkv * D))
        value = normal_f16(rng, (B * S, Hkv * D))
    cos, sin = rope_tables(max_cache_seq, rotary_dim if rotary_dim else 2, theta)
    present_key = normal_f16(rng, (B, Hkv, max_cache_seq, D))
    present_value = normal_f16(rng, (B, Hkv, max_cache_seq, D))
    return AppendCase(
        num_heads=Hq, kv_num_heads=Hkv, head_size=D, batch=B, seq_len=S, packed=packed,
        source=source, value=value,
        total_sequence_length=np.array([total_scalar], dtype=np.int32),
        key_total_sequence_lengths=totals.astype(np.int32),
        cos_cache=cos, sin_cache=sin, rotary_dim=rotary_dim, interleaved=interleaved,
        present_key=present_key, present_value=present_value)


# --------------------------------------------------------------------------------------
# Block-sparse edge list over paged fp32 K/V
# --------------------------------------------------------------------------------------
@dataclass
class SparseCase:
    qhead: int
    hq: int
    hkv: int
    head_dim: int
    block_size: int
    page_size: int
    pages_per_block: int
    q: np.ndarray             # [Tq, hq, D] fp32
    k_pages: np.ndarray       # [num_pages, hkv, page_size, D] fp32
    v_pages: np.ndarray
    edge_meta: np.ndarray     # [E, 5] int32: q_idx, h, blk, batch, block_len
    block_tables: np.ndarray  # [B, max_pages] int32, -1 = unmapped
    softmax_scale: float
    used_kv_lens: np.ndarray  # [B] int64 (how block_len was derived)
    seg_offsets: np.ndarray   # [Tq*hkv + 1] int32: edges of (q_idx, h) are contiguous

    def query_positions(self) -> np.ndarray:
        """Right-aligned absolute position of each query in its sequence: with n queries
        per sequence, query i of sequence b sits at used_b - n + i."""
        B = int(self.used_kv_lens.shape[0])
        n = int(self.q.shape[0]) // B
        return (np.repeat(self.used_kv_lens, n) - n + np.tile(np.arange(n), B)).astype(np.int32)

    @property
    def num_edges(self) -> int:
        return int(self.edge_meta.shape[0])

    @property
    def max_pages(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def num_pages(self) -> int:
        return int(self.k_pages.shape[0])


def block_sparse(seed: int = 5, *, n_seqs: int = 8, kv_len: int = 16384,
                 queries_per_seq: int = 512, hq: int = 32, hkv: int = 8,
                 head_dim: int = 128, page_size: int = 16, pages_per_block: int = 4,
                 blocks_per_query: int = 16, clip_max: int = 63,
                 unmapped_frac: float = 0.02, n_empty_edges: int = 0,
                 dtype=np.float32) -> SparseCase:
    """Block-sparse workload. Each sequence holds kv_len tokens in pages of
    page_size; its used length is U{kv_len - clip_max .. kv_len} so the last block
    is clipped. Query i of sequence b sits at position used_b - queries_per_seq + i
    (right-aligned); for every (query, kv head) the edge list names the query's
    local block plus blocks_per_query - 1 other distinct blocks at or below the
    last used block, sorted by (query, head, block). block_len is the used length
    clipped to the block. A fraction of block-table entries is set to -1, and
    n_empty_edges edges get block_len 0 (or a negative value) to exercise the
    empty-edge rule. dtype float16 draws q and the pages as fp16 instead of fp32."""
    rng = rng_for(seed)
    qhead = hq // hkv
    BSZ = page_size * pages_per_block
    max_pages = kv_len // page_size
    n_blocks = kv_len // BSZ
    num_pages = n_seqs * max_pages
    perm = rng.permutation(num_pages).astype(np.int32)
    block_tables = perm.reshape(n_seqs, max_pages).copy()
    unmapped = rng.random(block_tables.shape) < unmapped_frac
    block_tables[unmapped] = -1
    used = kv_len - rng.integers(0, clip_max + 1, size=n_seqs)
    Tq = n_seqs * queries_per_seq
    draw = normal_f16 if np.dtype(dtype) == np.float16 else normal_f32
    q = draw(rng, (Tq, hq, head_dim))
    k_pages = draw(rng, (num_pages, hkv, page_size, head_dim))
    v_pages = draw(rng, (num_pages, hkv, page_size, head_dim))
    last_blk = (used - 1) // BSZ
    edges = []
    for b in range(n_seqs):
        nb_avail = int(last_blk[b]) + 1
        pos = used[b] - queries_per_seq + np.arange(queries_per_seq)
        local = pos // BSZ
        for i in range(queries_per_seq):
            q_idx = b * queries_per_seq + i
            keys = rng.random((hkv, nb_avail))
            keys[:, local[i]] = -1.0        # the local block is always taken
            chosen = np.argsort(keys, axis=1)[:, :min(blocks_per_query, nb_avail)]
            for h in range(hkv):
                for blk in np.sort(chosen[h]):
                    blen = int(min(max(used[b] - int(blk) * BSZ, 0), BSZ))
                    edges.append((q_idx, h, int(blk), b, blen))
    edge_meta = np.asarray(edges, dtype=np.int32)
    if n_empty_edges:
        idx = rng.choice(edge_meta.shape[0], size=n_empty_edges, replace=False)
        edge_meta[idx, 4] = np.where(np.arange(n_empty_edges) % 2 == 0, 0, -3)
    counts = np.bincount(edge_meta[:, 0].astype(np.int64) * hkv + edge_meta[:, 1],
                         minlength=Tq * hkv)
    seg_offsets = np.zeros(Tq * hkv + 1, dtype=np.int32)
    seg_offsets[1:] = np.cumsum(counts)
    return SparseCase(
        qhead=qhead, hq=hq, hkv=hkv, head_dim=head_dim, block_size=BSZ,
        page_size=page_size, pages_per_block=pages_per_block, q=q, k_pages=k_pages,
        v_pages=v_pages, edge_meta=edge_meta, block_tables=block_tables,
        softmax_scale=1.0 / float(np.sqrt(head_dim)), used_kv_lens=used.astype(np.int64),
        seg_offsets=seg_offsets)
