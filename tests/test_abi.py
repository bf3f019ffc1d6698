"""C-ABI checks that need no GPU: the library loads, exports every declared symbol,
its structs match the binding, and its host-side logic (contract predicates, split
count, status codes, workspace sizing) agrees with the oracle and the pages."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

from oracle import pagedkv_oracle as orc
from paged_kv_cache_231_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(B.LIB_PATH):
        from paged_kv_cache_231_gb300 import build
        build.build()
    return B.load_library()


def declared_symbols():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            names |= set(re.findall(r"^\s*(?:int|int64_t|size_t|void|const char\*)\s+"
                                    r"(pkv_\w+)\s*\(", text, re.M))
    return sorted(names)


def test_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert len(names) >= 16, names
    for n in names:
        assert hasattr(lib, n), n


def test_struct_layouts_match(lib):
    for name, cls in B.STRUCTS.items():
        assert lib.pkv_sizeof_struct(name.encode()) == ctypes.sizeof(cls), name
    assert lib.pkv_sizeof_struct(b"nope") == 0


def test_status_strings(lib):
    for code in range(11):
        assert lib.pkv_status_string(code)
    assert lib.pkv_status_string(99) == b"unknown status"


def _host_case(T=2, B=2, Hq=4, Hkv=2, D=64, BS=16, NB=16, MB=6, packed=False, slot=False):
    f16 = torch.float16
    q = torch.zeros((T, (Hq + 2 * Hkv) * D if packed else Hq * D), dtype=f16)
    k = None if packed else torch.zeros((T, Hkv * D), dtype=f16)
    v = None if packed else torch.zeros((T, Hkv * D), dtype=f16)
    kc = torch.zeros((NB, BS, Hkv, D), dtype=f16)
    vc = torch.zeros_like(kc)
    cu = torch.zeros(B + 1, dtype=torch.int32)
    past = torch.zeros(B, dtype=torch.int32)
    bt = torch.zeros((B, MB), dtype=torch.int32)
    sm = torch.zeros(T, dtype=torch.int32) if slot else None
    out = torch.zeros((T, Hq * D), dtype=f16)
    return q, k, v, kc, vc, cu, past, bt, sm, out


def test_plan_matches_pages_split_count(golden, lib):
    g = golden("paged_split_counts.json")
    for c in g["cases"]:
        T = c["tokens"]
        args = B.make_paged_args(*_host_case(T=max(T, 1), Hkv=c["kv_heads"],
                                             Hq=c["kv_heads"] * 2, D=64,
                                             BS=c["block_size"], MB=c["max_blocks"])[:9],
                                 output=torch.zeros((max(T, 1), c["kv_heads"] * 2 * 64),
                                                    dtype=torch.float16),
                                 num_heads=c["kv_heads"] * 2, kv_num_heads=c["kv_heads"])
        args.num_tokens = T
        plan = B.pkv_paged_attention_plan(args)
        assert plan.pages_num_splits == c["expected"], c
        assert plan.pages_num_splits == orc.pages_num_splits(
            T, c["kv_heads"], c["max_blocks"], c["block_size"])
    s = g["scratch"]
    args = B.make_paged_args(*_host_case(T=s["tokens"], B=64, Hq=s["num_heads"], Hkv=8,
                                         D=s["head"], MB=512)[:9],
                             output=torch.zeros((s["tokens"], s["num_heads"] * s["head"]),
                                                dtype=torch.float16),
                             num_heads=s["num_heads"], kv_num_heads=8)
    plan = B.pkv_paged_attention_plan(args)
    assert plan.pages_num_splits == s["splits"]
    assert plan.pages_partial_bytes == s["expected_partial_bytes"]
    assert plan.pages_stats_bytes == s["expected_stats_bytes"]


def test_plan_split_count_random_against_oracle(lib):
    rng = np.random.default_rng(0)
    for _ in range(300):
        T = int(rng.integers(0, 3000))
        Hkv = int(rng.choice([1, 2, 4, 8, 16]))
        MB = int(rng.integers(1, 700))
        BS = int(rng.choice([1, 8, 16, 32, 64, 100]))
        args = B.PagedAttentionArgs()
        args.query = args.key_cache = args.value_cache = 256
        args.cumulative_sequence_length = args.past_seqlens = args.block_table = 256
        args.output = 256
        args.num_tokens, args.batch = T, 4
        args.num_heads, args.kv_num_heads = Hkv * 2, Hkv
        args.head_size, args.block_size, args.num_blocks, args.max_blocks = 64, BS, 10, MB
        args.query_hidden = Hkv * 2 * 64
        args.key, args.value = 256, 256
        args.is_causal, args.dtype = 1, B.PKV_F16
        plan = B.pkv_paged_attention_plan(args)
        assert plan.pages_num_splits == orc.pages_num_splits(T, Hkv, MB, BS)


def test_contract_check_matches_oracle_golden(golden, lib):
    g = golden("paged_contract.json")
    dt = {"float16": torch.float16, "float32": torch.float32}
    for c in g["cases"]:
        a = dict(g["base"])
        a.update(c["change"])
        mk = lambda shape, name: None if shape is None else torch.empty(
            shape, dtype=dt[a["dtypes"].get(name, "float16")])
        mi = lambda shape: None if shape is None else torch.empty(shape, dtype=torch.int32)
        st, failed, mode = B.pkv_paged_contract_check(
            mk(a["query"], "query"), mk(a["key"], "key"), mk(a["value"], "value"),
            mk(a["key_cache"], "key_cache"), mk(a["value_cache"], "value_cache"),
            mi(a["cu"]), mi(a["past"]), mi(a["block_table"]), mi(a["slot_mapping"]),
            mk(a["output"], "output"), num_heads=a["num_heads"],
            kv_num_heads=a["kv_num_heads"])
        assert sorted(failed) == sorted(c["false"]), c["name"]
        assert mode == c["mode"], c["name"]
        if c["ok"] and c["mode"]:
            assert st == B.PKV_OK, c["name"]
        else:
            assert st != B.PKV_OK, c["name"]


def test_contract_check_random_against_oracle(lib):
    rng = np.random.default_rng(1)
    for _ in range(400):
        Hq = int(rng.choice([1, 2, 3, 4, 8]))
        Hkv = int(rng.choice([1, 2, 3, 4]))
        D = int(rng.choice([8, 16]))
        T = int(rng.integers(1, 4))
        Bt = int(rng.integers(0, 3))
        pert = lambda x: x + int(rng.choice([0, 0, 0, 0, 1, -1]))
        packed = bool(rng.integers(0, 2))
        shapes = dict(
            query=[pert(T), pert((Hq + 2 * Hkv) * D if packed else Hq * D)],
            key=None if packed else [pert(T), pert(Hkv * D)],
            value=None if (packed or rng.random() < 0.1) else [T, Hkv * D],
            key_cache=[3, pert(4), pert(Hkv), D], value_cache=[3, 4, Hkv, D],
            cu=[pert(Bt + 1)], past=[pert(Bt)], block_table=[pert(Bt), pert(2)],
            slot_mapping=[pert(T)] if rng.random() < 0.3 else None, output=[pert(T), Hq * D])
        shapes = {k: (None if v is None else [max(0, x) for x in v])
                  for k, v in shapes.items()}
        ref = orc.paged_contract(
            query_shape=shapes["query"], key_shape=shapes["key"], value_shape=shapes["value"],
            key_cache_shape=shapes["key_cache"], value_cache_shape=shapes["value_cache"],
            cu_shape=shapes["cu"], past_shape=shapes["past"],
            block_table_shape=shapes["block_table"],
            slot_mapping_shape=shapes["slot_mapping"], output_shape=shapes["output"],
            num_heads=Hq, kv_num_heads=Hkv,
            dtypes={n: "float16" for n in ("query", "key", "value", "key_cache",
                                           "value_cache", "output")})
        mk = lambda s: None if s is None else torch.empty(s, dtype=torch.float16)
        mi = lambda s: None if s is None else torch.empty(s, dtype=torch.int32)
        st, failed, mode = B.pkv_paged_contract_check(
            mk(shapes["query"]), mk(shapes["key"]), mk(shapes["value"]),
            mk(shapes["key_cache"]), mk(shapes["value_cache"]), mi(shapes["cu"]),
            mi(shapes["past"]), mi(shapes["block_table"]), mi(shapes["slot_mapping"]),
            mk(shapes["output"]), num_heads=Hq, kv_num_heads=Hkv)
        names = ["cacheShapeOk", "headLayoutOk", "scheduleShapeOk", "ioShapeOk",
                 "separateKv", "packedKv", "slotShapeOk"]
        assert sorted(failed) == sorted(n for n in names if not ref[n]), shapes
        assert mode == ref["mode"]
        assert (st == B.PKV_OK) == (ref["pagedContractOk"] and ref["mode"] is not None)


def _args(**kw):
    a = B.make_paged_args(*_host_case()[:9], output=torch.zeros((2, 256), dtype=torch.float16),
                          num_heads=4, kv_num_heads=2)
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("change,status", [
    (dict(num_heads=5), 3),
    (dict(kv_num_heads=0), 3),
    (dict(is_causal=0), 6),
    (dict(dtype=B.PKV_F32), 4),
    (dict(value=None), 5),
    (dict(query_hidden=255), 2),
    (dict(block_size=0), 2),
    (dict(max_blocks=0), 2),
    (dict(batch=0), 2),
    (dict(output=None), 1),
    (dict(block_table=None), 1),
    (dict(rotary_dim=3), 2),
    (dict(rotary_dim=8), 1),
    (dict(split_policy=7), 2),
])
def test_plan_rejects_bad_arguments(lib, change, status):
    with pytest.raises(B.PagedKVError) as e:
        B.pkv_paged_attention_plan(_args(**change))
    assert e.value.status == status


def test_plan_unsupported_and_alignment(lib):
    a = _args()
    a.query = a.query + 2
    with pytest.raises(B.PagedKVError) as e:
        B.pkv_paged_attention_plan(a)
    assert e.value.status == 8
    # head size 96 is a valid contract shape but outside the compiled set
    args = B.make_paged_args(*_host_case(D=96)[:9],
                             output=torch.zeros((2, 4 * 96), dtype=torch.float16),
                             num_heads=4, kv_num_heads=2)
    with pytest.raises(B.PagedKVError) as e:
        B.pkv_paged_attention_plan(args)
    assert e.value.status == 9


def test_workspace_bounds(lib):
    # decode batch: every sequence may need up to max_splits partials per query head
    args = B.make_paged_args(*_host_case(T=64, B=64, Hq=32, Hkv=8, D=128, MB=512)[:9],
                             output=torch.zeros((64, 4096), dtype=torch.float16),
                             num_heads=32, kv_num_heads=8)
    plan = B.pkv_paged_attention_plan(args)
    assert plan.max_splits == 16 and plan.group_size == 4
    # the automatic policy runs the stream-K decode: no per-split items, partial rows
    # for up to 16 pieces of every (token, query head)
    assert plan.partial_slot_bound == 64 and plan.decode_item_bound == 0
    assert plan.workspace_bytes >= 64 * 32 * 16 * (128 + 2) * 4
    assert B.pkv_paged_attention_workspace_size(args) == plan.workspace_bytes
    # fixed split policy bounds the splits
    args.split_policy, args.fixed_splits = B.PKV_SPLIT_FIXED, 3
    plan = B.pkv_paged_attention_plan(args)
    assert plan.max_splits == 3 and plan.decode_item_bound == 64 * 3
    args.split_policy = B.PKV_SPLIT_PAGES
    assert B.pkv_paged_attention_plan(args).max_splits == orc.pages_num_splits(64, 8, 512, 16)


def test_sparse_and_combine_argument_checks(lib):
    a = B.SparseArgs()
    a.hkv, a.qhead, a.hq, a.head_dim = 2, 4, 8, 128
    a.max_pages, a.page_size, a.pages_per_block, a.block_size = 16, 16, 4, 64
    a.num_seqs, a.num_edges, a.num_pages = 2, 10, 32
    n = B.pkv_sparse_attention_partials_workspace_size(a)
    groups = 2 * 4 * 2
    assert n >= 4 * (2 * (groups + 1) + groups + 10)
    a.hq = 7
    with pytest.raises(B.PagedKVError):
        B.pkv_sparse_attention_partials_workspace_size(a)
    a.hq, a.block_size = 8, 65
    with pytest.raises(B.PagedKVError):
        B.pkv_sparse_attention_partials_workspace_size(a)
    c = B.CombineArgs()
    c.num_segments, c.lanes, c.head_dim, c.out_dtype = 1, 1, 100, B.PKV_F32
    assert lib.pkv_combine_partials(ctypes.byref(c), None) == 9
    c.head_dim, c.out_dtype = 128, 99
    assert lib.pkv_combine_partials(ctypes.byref(c), None) == 4
    c.out_dtype = B.PKV_F32
    assert lib.pkv_combine_partials(ctypes.byref(c), None) == 1   # NULL pointers


def test_sparse_pointer_checks_come_before_any_launch(lib):
    """The partials call checks pointers, their alignment (16 bytes; o_partial need not be
    32-byte aligned) and the workspace before it touches the device, so fake addresses
    exercise every refusal here; nothing is launched."""
    base = 1 << 20   # a fake, 256-byte aligned address: never dereferenced on these paths

    def call(ws=base, ws_bytes=1 << 30, num_edges=10, **ptr):
        a = B.SparseArgs(num_queries=100, num_edges=num_edges, num_seqs=2, max_pages=16,
                         num_pages=32, qhead=4, hq=32, hkv=8, head_dim=128, block_size=64,
                         page_size=16, pages_per_block=4, softmax_scale=0.1, dtype=B.PKV_F16)
        for i, k in enumerate(("q", "k_pages", "v_pages", "edge_meta", "block_tables",
                               "o_partial", "m_partial", "l_partial")):
            setattr(a, k, ptr.get(k, base + (i + 1) * (1 << 16)))
        return lib.pkv_sparse_attention_partials(ctypes.byref(a), ws, ws_bytes, None)

    o = base + 6 * (1 << 16)
    assert call(o_partial=o + 8) == 8            # PKV_ERR_ALIGN
    assert call(q=base + 8) == 8
    assert call(o_partial=o + 16, ws=None) == 7   # 16-byte aligned o passes; no workspace
    assert call(ws=base + 128) == 7              # workspace not 256-byte aligned
    assert call(ws_bytes=16) == 7                # workspace too small
    assert call(o_partial=None) == 1             # PKV_ERR_NULL
    assert call(num_edges=0, o_partial=None, q=None) == 0   # nothing to do, nothing read


def test_sparse_workspace_holds_the_split_q_rows(lib):
    # fp32 calls that run on the tensor core take Q as split fp16 (hi, lo) rows plus one
    # shift per row in the workspace; fp16 calls and other shapes do not
    def size(**kw):
        a = B.SparseArgs(num_queries=100, num_edges=10, num_seqs=2, max_pages=16, num_pages=32,
                         qhead=4, hq=32, hkv=8, head_dim=128, block_size=64, page_size=16,
                         pages_per_block=4, softmax_scale=0.1, dtype=0)
        for k, v in kw.items():
            setattr(a, k, v)
        return B.pkv_sparse_attention_partials_workspace_size(a)
    rows = 100 * 32
    assert size() - size(num_queries=0) == 2 * rows * 128 * 2 + rows * 4
    assert size(dtype=B.PKV_F16) == size(dtype=B.PKV_F16, num_queries=0)
    # 128-key blocks run on fp32 FMA: no split rows
    assert size(block_size=128, pages_per_block=8) == size(block_size=128, pages_per_block=8,
                                                           num_queries=0)


def test_binding_raises_without_library(tmp_path):
    with pytest.raises(RuntimeError):
        B.load_library(str(tmp_path / "missing.so"))


def test_huge_sizes_are_refused_before_any_product_overflows(lib):
    # Sizes whose int64 products would overflow are refused up front (no launch, no GPU).
    big = 1 << 40
    a = B.make_paged_args(*_host_case()[:9], output=torch.zeros((2, 4 * 64), dtype=torch.float16),
                          num_heads=4, kv_num_heads=2)
    for field in ("max_blocks", "block_size", "num_blocks", "num_heads"):
        b = B.PagedAttentionArgs.from_buffer_copy(a)
        setattr(b, field, big)
        if field == "num_heads":
            b.kv_num_heads = big // 2   # keep the head ratio valid
        plan = B.PagedPlan()
        st = lib.pkv_paged_attention_plan(ctypes.byref(b), ctypes.byref(plan))
        assert B.STATUS_NAMES[st] == "PKV_ERR_UNSUPPORTED", field
    s = B.SparseArgs(num_queries=4, num_edges=4, num_seqs=1, max_pages=8, num_pages=8,
                     qhead=4, hq=32, hkv=8, head_dim=128, block_size=64, page_size=16,
                     pages_per_block=4, softmax_scale=0.1, dtype=0)
    n = ctypes.c_size_t(0)
    assert lib.pkv_sparse_attention_partials_workspace_size(ctypes.byref(s), ctypes.byref(n)) == 0
    for field, value in (("num_seqs", big), ("max_pages", big), ("num_pages", big),
                         ("num_seqs", (1 << 31) - 1)):
        t = B.SparseArgs.from_buffer_copy(s)
        setattr(t, field, value)
        st = lib.pkv_sparse_attention_partials_workspace_size(ctypes.byref(t), ctypes.byref(n))
        assert B.STATUS_NAMES[st] == "PKV_ERR_UNSUPPORTED", (field, value)
