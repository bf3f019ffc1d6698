"""Thin Python binding of ``libpagedkv`` (the C ABI in include/pagedkv.h).

Argument marshalling only: torch tensors supply device pointers, sizes and the
current CUDA stream; every step of the computation runs in the library's kernels.
There is no fallback: if the shared library is missing or fails to load, every call
raises. Function names match the C entry points.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libpagedkv.so")

PKV_OK = 0
STATUS_NAMES = {0: "PKV_OK", 1: "PKV_ERR_NULL", 2: "PKV_ERR_SHAPE", 3: "PKV_ERR_HEADS",
                4: "PKV_ERR_DTYPE", 5: "PKV_ERR_KV_MODE", 6: "PKV_ERR_CAUSAL",
                7: "PKV_ERR_WORKSPACE", 8: "PKV_ERR_ALIGN", 9: "PKV_ERR_UNSUPPORTED",
                10: "PKV_ERR_LAUNCH"}
PKV_F16, PKV_BF16, PKV_F32, PKV_I32 = 1, 2, 3, 4
PKV_SPLIT_AUTO, PKV_SPLIT_PAGES, PKV_SPLIT_FIXED = 0, 1, 2
DEV_BAD_BLOCK, DEV_BAD_SLOT, DEV_BAD_POSITION, DEV_BAD_SEQUENCE, DEV_BAD_EDGE = 1, 2, 4, 8, 16
PRED_BITS = {"cacheShapeOk": 1, "headLayoutOk": 2, "scheduleShapeOk": 4, "ioShapeOk": 8,
             "separateKv": 16, "packedKv": 32, "slotShapeOk": 64}

c_i32, c_i64, c_f32, c_vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p


class PagedKVError(RuntimeError):
    def __init__(self, call: str, status: int):
        self.status = status
        self.name = STATUS_NAMES.get(status, str(status))
        super().__init__(f"{call} failed: {self.name} ({_status_string(status)})")


class PagedAttentionArgs(ctypes.Structure):
    _fields_ = [("query", c_vp), ("key", c_vp), ("value", c_vp), ("key_cache", c_vp),
                ("value_cache", c_vp), ("cumulative_sequence_length", c_vp),
                ("past_seqlens", c_vp), ("block_table", c_vp), ("slot_mapping", c_vp),
                ("output", c_vp), ("device_status", c_vp), ("cos_cache", c_vp),
                ("sin_cache", c_vp),
                ("num_tokens", c_i64), ("query_hidden", c_i64), ("batch", c_i64),
                ("num_heads", c_i64), ("kv_num_heads", c_i64), ("head_size", c_i64),
                ("block_size", c_i64), ("num_blocks", c_i64), ("max_blocks", c_i64),
                ("rotary_dim", c_i64), ("rotary_positions", c_i64),
                ("rotary_interleaved", c_i32), ("is_causal", c_i32), ("dtype", c_i32),
                ("scale", c_f32), ("split_policy", c_i32), ("fixed_splits", c_i32),
                ("max_splits", c_i32), ("split_min_keys", c_i32), ("rotary_query", c_i32),
                ("reserved", c_i32)]


class PagedPlan(ctypes.Structure):
    _fields_ = [("mode", c_i32), ("group_size", c_i32), ("pages_num_splits", c_i32),
                ("max_splits", c_i32), ("pages_partial_bytes", c_i64),
                ("pages_stats_bytes", c_i64), ("workspace_bytes", c_i64),
                ("decode_item_bound", c_i64), ("prefill_item_bound", c_i64),
                ("partial_slot_bound", c_i64)]


class TensorDesc(ctypes.Structure):
    _fields_ = [("present", c_i32), ("rank", c_i32), ("dtype", c_i32), ("reserved", c_i32),
                ("dims", c_i64 * 4)]


class PagedShapes(ctypes.Structure):
    _fields_ = [(n, TensorDesc) for n in ("query", "key", "value", "key_cache",
                                          "value_cache", "cumulative_sequence_length",
                                          "past_seqlens", "block_table", "slot_mapping",
                                          "output")] + \
               [("num_heads", c_i64), ("kv_num_heads", c_i64), ("is_causal", c_i32),
                ("reserved", c_i32)]


class KVAppendArgs(ctypes.Structure):
    _fields_ = [("source", c_vp), ("value", c_vp), ("total_sequence_length", c_vp),
                ("key_total_sequence_lengths", c_vp), ("cos_cache", c_vp),
                ("sin_cache", c_vp), ("present_key", c_vp), ("present_value", c_vp),
                ("device_status", c_vp), ("batch", c_i64), ("seq_len", c_i64),
                ("num_heads", c_i64), ("kv_num_heads", c_i64), ("head_size", c_i64),
                ("max_cache_seq", c_i64), ("rotary_dim", c_i64), ("rotary_positions", c_i64),
                ("packed", c_i32), ("interleaved", c_i32), ("dtype", c_i32),
                ("reserved", c_i32), ("query", c_vp), ("query_out", c_vp)]


class SparseArgs(ctypes.Structure):
    _fields_ = [("q", c_vp), ("k_pages", c_vp), ("v_pages", c_vp), ("edge_meta", c_vp),
                ("block_tables", c_vp), ("o_partial", c_vp), ("m_partial", c_vp),
                ("l_partial", c_vp), ("device_status", c_vp), ("num_queries", c_i64),
                ("num_edges", c_i64), ("num_seqs", c_i64), ("max_pages", c_i64),
                ("num_pages", c_i64), ("qhead", c_i64), ("hq", c_i64), ("hkv", c_i64),
                ("head_dim", c_i64), ("block_size", c_i64), ("page_size", c_i64),
                ("pages_per_block", c_i64), ("softmax_scale", c_f32), ("dtype", c_i32),
                ("query_positions", c_vp)]


class CombineArgs(ctypes.Structure):
    _fields_ = [("o", c_vp), ("m", c_vp), ("l", c_vp), ("segment_offsets", c_vp),
                ("out", c_vp), ("lse", c_vp), ("num_segments", c_i64), ("lanes", c_i64),
                ("head_dim", c_i64), ("uniform_count", c_i64), ("out_dtype", c_i32),
                ("reserved", c_i32)]


STRUCTS = {"pkv_paged_attention_args": PagedAttentionArgs, "pkv_paged_plan": PagedPlan,
           "pkv_tensor_desc": TensorDesc, "pkv_paged_shapes": PagedShapes,
           "pkv_kv_append_args": KVAppendArgs, "pkv_sparse_args": SparseArgs,
           "pkv_combine_args": CombineArgs}

_LIB = None


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libpagedkv (once) and check ABI version and struct layouts. Raises if the
    library is absent: build it with ``__graft_entry__.build()``."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libpagedkv not built ({p} missing); run __graft_entry__.build()")
    lib = ctypes.CDLL(p)
    lib.pkv_abi_version.restype = c_i32
    lib.pkv_status_string.restype = ctypes.c_char_p
    lib.pkv_status_string.argtypes = [c_i32]
    lib.pkv_sizeof_struct.restype = ctypes.c_size_t
    lib.pkv_sizeof_struct.argtypes = [ctypes.c_char_p]
    lib.pkv_launch_count.restype = c_i64
    lib.pkv_profiler_enable.argtypes = [c_i32]
    lib.pkv_profiler_query.argtypes = [ctypes.c_char_p, ctypes.POINTER(ctypes.c_double),
                                       ctypes.POINTER(c_i64)]
    for name, args in (
            ("pkv_paged_attention_plan", [ctypes.POINTER(PagedAttentionArgs),
                                          ctypes.POINTER(PagedPlan)]),
            ("pkv_paged_attention_workspace_size", [ctypes.POINTER(PagedAttentionArgs),
                                                    ctypes.POINTER(ctypes.c_size_t)]),
            ("pkv_paged_attention", [ctypes.POINTER(PagedAttentionArgs), c_vp,
                                     ctypes.c_size_t, c_vp]),
            ("pkv_paged_scatter_kv", [ctypes.POINTER(PagedAttentionArgs), c_vp]),
            ("pkv_paged_contract_check", [ctypes.POINTER(PagedShapes),
                                          ctypes.POINTER(ctypes.c_uint32),
                                          ctypes.POINTER(c_i32)]),
            ("pkv_kv_append_rotary", [ctypes.POINTER(KVAppendArgs), c_vp]),
            ("pkv_sparse_attention_partials_workspace_size",
             [ctypes.POINTER(SparseArgs), ctypes.POINTER(ctypes.c_size_t)]),
            ("pkv_sparse_attention_partials", [ctypes.POINTER(SparseArgs), c_vp,
                                               ctypes.c_size_t, c_vp]),
            ("pkv_combine_partials", [ctypes.POINTER(CombineArgs), c_vp]),
            ("pkv_testing_wait_limit", [ctypes.c_uint32, c_i32])):
        fn = getattr(lib, name)
        fn.restype = c_i32
        fn.argtypes = args
    if lib.pkv_abi_version() != 3:
        raise RuntimeError("libpagedkv ABI version mismatch")
    for name, cls in STRUCTS.items():
        n = lib.pkv_sizeof_struct(name.encode())
        if n != ctypes.sizeof(cls):
            raise RuntimeError(f"struct {name}: library {n} bytes, binding "
                               f"{ctypes.sizeof(cls)} bytes")
    if path is None:
        _LIB = lib
    return lib


def _status_string(status: int) -> str:
    try:
        return load_library().pkv_status_string(status).decode()
    except Exception:  # noqa: BLE001 - message only
        return ""


def _check(call: str, status: int):
    if status != PKV_OK:
        raise PagedKVError(call, status)


# ----------------------------------------------------------------------------- helpers
def _torch():
    import torch
    return torch


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _require(t, dtype, name, device=True):
    torch = _torch()
    if t is None:
        return
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if device and not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")


_DT = {"float16": PKV_F16, "bfloat16": PKV_BF16, "float32": PKV_F32, "int32": PKV_I32}


def _dtype_code(t) -> int:
    return _DT.get(str(t.dtype).replace("torch.", ""), 0)


def _desc(t) -> TensorDesc:
    d = TensorDesc()
    if t is None:
        return d
    d.present = 1
    d.rank = t.dim()
    d.dtype = _dtype_code(t)
    for i, s in enumerate(list(t.shape)[:4]):
        d.dims[i] = int(s)
    return d


# ----------------------------------------------------------------------------- paged
def pkv_paged_contract_check(query, key, value, key_cache, value_cache,
                             cumulative_sequence_length, past_seqlens, block_table,
                             slot_mapping, output, *, num_heads: int, kv_num_heads: int,
                             is_causal: int = 1):
    """Shape/dtype contract of the PagedAttention manifest (host only; tensors may live
    on any device). Returns (status, failed_predicates_set, mode)."""
    lib = load_library()
    sh = PagedShapes()
    for name, t in (("query", query), ("key", key), ("value", value),
                    ("key_cache", key_cache), ("value_cache", value_cache),
                    ("cumulative_sequence_length", cumulative_sequence_length),
                    ("past_seqlens", past_seqlens), ("block_table", block_table),
                    ("slot_mapping", slot_mapping), ("output", output)):
        setattr(sh, name, _desc(t))
    sh.num_heads = num_heads
    sh.kv_num_heads = kv_num_heads
    sh.is_causal = is_causal
    failed = ctypes.c_uint32(0)
    mode = c_i32(0)
    st = lib.pkv_paged_contract_check(ctypes.byref(sh), ctypes.byref(failed),
                                      ctypes.byref(mode))
    names = {n for n, bit in PRED_BITS.items() if failed.value & bit}
    return st, names, {1: "separate", 2: "packed"}.get(mode.value)


def make_paged_args(query, key, value, key_cache, value_cache, cumulative_sequence_length,
                    past_seqlens, block_table, slot_mapping=None, output=None, *,
                    num_heads: int, kv_num_heads: int, scale: float = 0.0,
                    is_causal: int = 1, device_status=None, cos_cache=None, sin_cache=None,
                    rotary_dim: int = 0, rotary_interleaved: bool = False,
                    split_policy: int = PKV_SPLIT_AUTO, fixed_splits: int = 0,
                    max_splits: int = 0, split_min_keys: int = 0,
                    rotary_query: bool = False) -> PagedAttentionArgs:
    """Fill the C argument block from tensors (no validation beyond rank checks; the
    library validates). Works for host-only planning too (pointers may be host)."""
    a = PagedAttentionArgs()
    a.query, a.key, a.value = _ptr(query), _ptr(key), _ptr(value)
    a.key_cache, a.value_cache = _ptr(key_cache), _ptr(value_cache)
    a.cumulative_sequence_length = _ptr(cumulative_sequence_length)
    a.past_seqlens = _ptr(past_seqlens)
    a.block_table = _ptr(block_table)
    a.slot_mapping = _ptr(slot_mapping)
    a.output = _ptr(output)
    a.device_status = _ptr(device_status)
    a.cos_cache, a.sin_cache = _ptr(cos_cache), _ptr(sin_cache)
    a.num_tokens = int(query.shape[0])
    a.query_hidden = int(query.shape[1]) if query.dim() == 2 else 0
    a.batch = int(cumulative_sequence_length.shape[0]) - 1
    a.num_heads, a.kv_num_heads = int(num_heads), int(kv_num_heads)
    a.num_blocks, a.block_size = int(key_cache.shape[0]), int(key_cache.shape[1])
    a.head_size = int(key_cache.shape[3])
    a.max_blocks = int(block_table.shape[1])
    a.rotary_dim = int(rotary_dim)
    a.rotary_positions = int(cos_cache.shape[0]) if cos_cache is not None else 0
    a.rotary_interleaved = 1 if rotary_interleaved else 0
    a.is_causal = int(is_causal)
    a.dtype = _dtype_code(query)
    a.scale = float(scale)
    a.split_policy, a.fixed_splits = int(split_policy), int(fixed_splits)
    a.max_splits, a.split_min_keys = int(max_splits), int(split_min_keys)
    a.rotary_query = 1 if rotary_query else 0
    return a


def pkv_paged_attention_plan(args: PagedAttentionArgs) -> PagedPlan:
    plan = PagedPlan()
    _check("pkv_paged_attention_plan",
           load_library().pkv_paged_attention_plan(ctypes.byref(args), ctypes.byref(plan)))
    return plan


def pkv_paged_attention_workspace_size(args: PagedAttentionArgs) -> int:
    n = ctypes.c_size_t(0)
    _check("pkv_paged_attention_workspace_size",
           load_library().pkv_paged_attention_workspace_size(ctypes.byref(args),
                                                             ctypes.byref(n)))
    return int(n.value)


def _check_paged_tensors(query, key, value, key_cache, value_cache, cu, past, bt, slot,
                         output, num_heads, kv_num_heads, is_causal):
    torch = _torch()
    for t, n in ((query, "query"), (key, "key"), (value, "value"), (key_cache, "key_cache"),
                 (value_cache, "value_cache"), (output, "output")):
        _require(t, torch.float16, n)
    for t, n in ((cu, "cumulative_sequence_length"), (past, "past_seqlens"),
                 (bt, "block_table"), (slot, "slot_mapping")):
        _require(t, torch.int32, n)
    st, failed, mode = pkv_paged_contract_check(
        query, key, value, key_cache, value_cache, cu, past, bt, slot, output,
        num_heads=num_heads, kv_num_heads=kv_num_heads, is_causal=is_causal)
    _check(f"pkv_paged_contract_check (false: {sorted(failed)})", st)


def pkv_paged_attention(query, key, value, key_cache, value_cache,
                        cumulative_sequence_length, past_seqlens, block_table,
                        slot_mapping=None, *, num_heads: int, kv_num_heads: int,
                        scale: float = 0.0, is_causal: int = 1, output=None, workspace=None,
                        device_status=None, cos_cache=None, sin_cache=None,
                        rotary_dim: int = 0, rotary_interleaved: bool = False,
                        split_policy: int = PKV_SPLIT_AUTO, fixed_splits: int = 0,
                        max_splits: int = 0, split_min_keys: int = 0,
                        rotary_query: bool = False, stream=None):
    """PagedAttention: scatter new K/V into the caches (in place), then causal GQA
    attention. Returns the fp16 output [num_tokens, num_heads*head_size]."""
    torch = _torch()
    if output is None:
        output = torch.empty((query.shape[0], num_heads * key_cache.shape[3]),
                             dtype=torch.float16, device=query.device)
    _check_paged_tensors(query, key, value, key_cache, value_cache,
                         cumulative_sequence_length, past_seqlens, block_table,
                         slot_mapping, output, num_heads, kv_num_heads, is_causal)
    if cos_cache is not None:
        _require(cos_cache, torch.float16, "cos_cache")
        _require(sin_cache, torch.float16, "sin_cache")
    a = make_paged_args(query, key, value, key_cache, value_cache,
                        cumulative_sequence_length, past_seqlens, block_table, slot_mapping,
                        output, num_heads=num_heads, kv_num_heads=kv_num_heads, scale=scale,
                        is_causal=is_causal, device_status=device_status,
                        cos_cache=cos_cache, sin_cache=sin_cache, rotary_dim=rotary_dim,
                        rotary_interleaved=rotary_interleaved, split_policy=split_policy,
                        fixed_splits=fixed_splits, max_splits=max_splits,
                        split_min_keys=split_min_keys, rotary_query=rotary_query)
    need = pkv_paged_attention_workspace_size(a)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=query.device)
    _check("pkv_paged_attention",
           load_library().pkv_paged_attention(ctypes.byref(a), workspace.data_ptr(), need,
                                              _stream(stream)))
    return output


def pkv_paged_scatter_kv(query, key, value, key_cache, value_cache,
                         cumulative_sequence_length, past_seqlens, block_table,
                         slot_mapping=None, *, num_heads: int, kv_num_heads: int,
                         device_status=None, cos_cache=None, sin_cache=None,
                         rotary_dim: int = 0, rotary_interleaved: bool = False,
                         stream=None):
    """The ScatterKV pass alone (caches updated in place)."""
    torch = _torch()
    for t, n in ((query, "query"), (key, "key"), (value, "value"),
                 (key_cache, "key_cache"), (value_cache, "value_cache")):
        _require(t, torch.float16, n)
    a = make_paged_args(query, key, value, key_cache, value_cache,
                        cumulative_sequence_length, past_seqlens, block_table, slot_mapping,
                        None, num_heads=num_heads, kv_num_heads=kv_num_heads,
                        device_status=device_status, cos_cache=cos_cache,
                        sin_cache=sin_cache, rotary_dim=rotary_dim,
                        rotary_interleaved=rotary_interleaved)
    _check("pkv_paged_scatter_kv",
           load_library().pkv_paged_scatter_kv(ctypes.byref(a), _stream(stream)))


# ----------------------------------------------------------------------------- append
def make_append_args(source, value, total_sequence_length, key_total_sequence_lengths,
                     present_key, present_value, *, num_heads: int, kv_num_heads: int,
                     batch: int, seq_len: int, packed: bool, cos_cache=None, sin_cache=None,
                     rotary_dim: int = 0, interleaved: bool = False,
                     device_status=None, query=None, query_out=None) -> KVAppendArgs:
    """Fill the C argument block of pkv_kv_append_rotary from tensors."""
    a = KVAppendArgs()
    a.source, a.value = _ptr(source), _ptr(value)
    a.total_sequence_length = _ptr(total_sequence_length)
    a.key_total_sequence_lengths = _ptr(key_total_sequence_lengths)
    a.cos_cache, a.sin_cache = _ptr(cos_cache), _ptr(sin_cache)
    a.present_key, a.present_value = _ptr(present_key), _ptr(present_value)
    a.device_status = _ptr(device_status)
    a.batch, a.seq_len = int(batch), int(seq_len)
    a.num_heads, a.kv_num_heads = int(num_heads), int(kv_num_heads)
    a.head_size = int(present_key.shape[3])
    a.max_cache_seq = int(present_key.shape[2])
    a.rotary_dim = int(rotary_dim)
    a.rotary_positions = int(cos_cache.shape[0]) if cos_cache is not None else 0
    a.packed = 1 if packed else 0
    a.interleaved = 1 if interleaved else 0
    a.dtype = _dtype_code(source)
    a.query, a.query_out = _ptr(query), _ptr(query_out)
    return a


def pkv_kv_append_rotary(source, value, total_sequence_length, key_total_sequence_lengths,
                         present_key, present_value, *, num_heads: int, kv_num_heads: int,
                         batch: int, seq_len: int, packed: bool, cos_cache=None,
                         sin_cache=None, rotary_dim: int = 0, interleaved: bool = False,
                         device_status=None, query=None, query_out=None, stream=None):
    """KV append (+ RoPE of K); with ``query_out`` the query heads are rotated at the
    same positions into it ([batch*seq_len, num_heads*head_size] fp16; ``query`` gives
    the query rows in separate mode)."""
    torch = _torch()
    for t, n in ((source, "source"), (value, "value"), (present_key, "present_key"),
                 (present_value, "present_value"), (cos_cache, "cos_cache"),
                 (sin_cache, "sin_cache"), (query, "query"), (query_out, "query_out")):
        _require(t, torch.float16, n)
    a = make_append_args(source, value, total_sequence_length, key_total_sequence_lengths,
                         present_key, present_value, num_heads=num_heads,
                         kv_num_heads=kv_num_heads, batch=batch, seq_len=seq_len,
                         packed=packed, cos_cache=cos_cache, sin_cache=sin_cache,
                         rotary_dim=rotary_dim, interleaved=interleaved,
                         device_status=device_status, query=query, query_out=query_out)
    _check("pkv_kv_append_rotary",
           load_library().pkv_kv_append_rotary(ctypes.byref(a), _stream(stream)))


# ----------------------------------------------------------------------------- sparse
def make_sparse_args(q, k_pages, v_pages, edge_meta, block_tables, o, m, l, *, qhead: int,
                     block_size: int, page_size: int, pages_per_block: int,
                     softmax_scale: float, device_status=None,
                     query_positions=None) -> SparseArgs:
    a = SparseArgs()
    a.q, a.k_pages, a.v_pages = _ptr(q), _ptr(k_pages), _ptr(v_pages)
    a.edge_meta, a.block_tables = _ptr(edge_meta), _ptr(block_tables)
    a.o_partial, a.m_partial, a.l_partial = _ptr(o), _ptr(m), _ptr(l)
    a.device_status = _ptr(device_status)
    a.num_queries, a.hq, a.head_dim = int(q.shape[0]), int(q.shape[1]), int(q.shape[2])
    a.num_edges = int(edge_meta.shape[0])
    a.num_seqs, a.max_pages = int(block_tables.shape[0]), int(block_tables.shape[1])
    a.num_pages, a.hkv = int(k_pages.shape[0]), int(k_pages.shape[1])
    a.qhead = int(qhead)
    a.block_size, a.page_size = int(block_size), int(page_size)
    a.pages_per_block = int(pages_per_block)
    a.softmax_scale = float(softmax_scale)
    a.dtype = _dtype_code(q)
    a.query_positions = _ptr(query_positions)
    return a


def pkv_sparse_attention_partials_workspace_size(args: SparseArgs) -> int:
    n = ctypes.c_size_t(0)
    _check("pkv_sparse_attention_partials_workspace_size",
           load_library().pkv_sparse_attention_partials_workspace_size(ctypes.byref(args),
                                                                       ctypes.byref(n)))
    return int(n.value)


def pkv_sparse_attention_partials(q, k_pages, v_pages, edge_meta, block_tables, *,
                                  qhead: int, block_size: int, page_size: int,
                                  pages_per_block: int, softmax_scale: float,
                                  o=None, m=None, l=None, workspace=None,
                                  device_status=None, query_positions=None, stream=None):
    """Block-sparse (o, m, l) partials, partial index edge*qhead + lane. q and the pages
    are all fp32 or all fp16; the partials are fp32. ``query_positions`` (int32 per
    query) applies the right-aligned causal mask."""
    torch = _torch()
    dt = torch.float16 if q.dtype == torch.float16 else torch.float32
    for t, n in ((q, "q"), (k_pages, "k_pages"), (v_pages, "v_pages")):
        _require(t, dt, n)
    _require(edge_meta, torch.int32, "edge_meta")
    _require(block_tables, torch.int32, "block_tables")
    _require(query_positions, torch.int32, "query_positions")
    P = int(edge_meta.shape[0]) * qhead
    D = int(q.shape[2])
    if o is None:
        o = torch.empty((P, D), dtype=torch.float32, device=q.device)
    if m is None:
        m = torch.empty(P, dtype=torch.float32, device=q.device)
    if l is None:
        l = torch.empty(P, dtype=torch.float32, device=q.device)
    a = make_sparse_args(q, k_pages, v_pages, edge_meta, block_tables, o, m, l, qhead=qhead,
                         block_size=block_size, page_size=page_size,
                         pages_per_block=pages_per_block, softmax_scale=softmax_scale,
                         device_status=device_status, query_positions=query_positions)
    need = pkv_sparse_attention_partials_workspace_size(a)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _check("pkv_sparse_attention_partials",
           load_library().pkv_sparse_attention_partials(ctypes.byref(a), workspace.data_ptr(),
                                                        need, _stream(stream)))
    return o, m, l


# ----------------------------------------------------------------------------- combine
def pkv_combine_partials(o, m, l, segment_offsets=None, *, num_segments: int, lanes: int,
                         uniform_count: int = 0, out=None, out_dtype=None, lse=None,
                         stream=None):
    """LSE merge: output row s*lanes + c from partial rows e*lanes + c, e in segment s."""
    torch = _torch()
    _require(o, torch.float32, "o")
    _require(m, torch.float32, "m")
    _require(l, torch.float32, "l")
    _require(segment_offsets, torch.int32, "segment_offsets")
    D = int(o.shape[-1])
    if out is None:
        out = torch.empty((num_segments * lanes, D), dtype=out_dtype or torch.float32,
                          device=o.device)
    a = CombineArgs()
    a.o, a.m, a.l = _ptr(o), _ptr(m), _ptr(l)
    a.segment_offsets = _ptr(segment_offsets)
    a.out, a.lse = _ptr(out), _ptr(lse)
    a.num_segments, a.lanes, a.head_dim = int(num_segments), int(lanes), D
    a.uniform_count = int(uniform_count)
    a.out_dtype = _dtype_code(out)
    _check("pkv_combine_partials",
           load_library().pkv_combine_partials(ctypes.byref(a), _stream(stream)))
    return out, lse


# ----------------------------------------------------------------------------- runtime
def pkv_launch_count() -> int:
    return int(load_library().pkv_launch_count())


def pkv_profiler_enable(on: bool = True):
    load_library().pkv_profiler_enable(1 if on else 0)


def pkv_profiler_reset():
    load_library().pkv_profiler_reset()


def pkv_profiler_query(kernel: str):
    """(total_ms, launches) of one kernel family since the last reset."""
    ms = ctypes.c_double(0.0)
    n = c_i64(0)
    _check("pkv_profiler_query",
           load_library().pkv_profiler_query(kernel.encode(), ctypes.byref(ms), ctypes.byref(n)))
    return float(ms.value), int(n.value)


def pkv_testing_wait_limit(max_polls: int = 0, withhold_first_copy: bool = False):
    """Testing hook of the tensor-core kernels' bounded waits (see pagedkv.h): a lower
    poll bound and, optionally, a withheld first bulk copy per CTA so that a wait gives
    up. pkv_testing_wait_limit() restores the defaults."""
    _check("pkv_testing_wait_limit",
           load_library().pkv_testing_wait_limit(int(max_polls), 1 if withhold_first_copy else 0))


def pkv_paged_attention_static_workspace(query, key, value, key_cache, value_cache,
                                         cumulative_sequence_length, past_seqlens,
                                         block_table, slot_mapping=None, *, num_heads: int,
                                         kv_num_heads: int, scale: float = 0.0,
                                         output, device_status=None, stream=None, **kw):
    """Paged attention for callers that may not allocate device memory: scratch comes
    from the library's fixed device array (PKV_STATIC_WORKSPACE_BYTES per GPU), so this
    call allocates nothing, not even the output, which the caller passes in. Calls that
    overlap on the GPU share that array and must be serialised."""
    lib = load_library()
    fn = lib.pkv_paged_attention_static_workspace
    fn.restype = c_i32
    fn.argtypes = [ctypes.POINTER(PagedAttentionArgs), c_vp]
    a = make_paged_args(query, key, value, key_cache, value_cache,
                        cumulative_sequence_length, past_seqlens, block_table, slot_mapping,
                        output, num_heads=num_heads, kv_num_heads=kv_num_heads, scale=scale,
                        device_status=device_status, **kw)
    _check("pkv_paged_attention_static_workspace", fn(ctypes.byref(a), _stream(stream)))
    return output
