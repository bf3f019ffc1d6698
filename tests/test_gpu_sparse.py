"""GPU parity of pkv_sparse_attention_partials and pkv_combine_partials."""
import numpy as np
import pytest
import torch

from oracle import pagedkv_oracle as orc
from paged_kv_cache_231_gb300 import binding as B
from paged_kv_cache_231_gb300 import workloads as wl

from .gpu_util import DEV, assert_f16_close, assert_f32_close, dev, f32_margins, host

pytestmark = pytest.mark.gpu


def run_gpu(c, qpos=None):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, m, l = B.pkv_sparse_attention_partials(
        dev(c.q), dev(c.k_pages), dev(c.v_pages), dev(c.edge_meta), dev(c.block_tables),
        qhead=c.qhead, block_size=c.block_size, page_size=c.page_size,
        pages_per_block=c.pages_per_block, softmax_scale=c.softmax_scale,
        device_status=status, query_positions=dev(qpos))
    nseg = c.seg_offsets.shape[0] - 1
    lse = torch.empty(nseg * c.qhead, dtype=torch.float32, device=DEV)
    out, _ = B.pkv_combine_partials(o, m, l, dev(c.seg_offsets), num_segments=nseg,
                                    lanes=c.qhead, lse=lse)
    torch.cuda.synchronize()
    return host(o), host(m), host(l), host(out), host(lse), int(status.item())


def oracle_partials(c, edges=None, qpos=None):
    return orc.sparse_attention_partials(
        c.q, c.k_pages, c.v_pages, c.edge_meta, c.block_tables, qhead=c.qhead, hq=c.hq,
        head_dim=c.head_dim, block_size=c.block_size, page_size=c.page_size,
        pages_per_block=c.pages_per_block, softmax_scale=c.softmax_scale, edges=edges,
        query_positions=qpos)


# fp16 inputs: scores are exact fp16 products summed in fp32 (m to fp32 level), but the
# weights are rounded once to fp16 (relative 2^-12) before O = P V and in l
F16_PARTIAL_RTOL = 5e-3


def compare_partials(go, gm, gl, ro, rm, rl, rows, f16=False):
    np.testing.assert_array_equal(gl[rows] == 0, rl[rows] == 0)
    empty = rl[rows] == 0
    assert (gm[rows][empty] == -1e30).all() and (go[rows][empty] == 0).all()
    live = rows[~empty]
    rt = F16_PARTIAL_RTOL if f16 else None
    assert_f32_close(go[live], ro[live], "o partial", rtol=rt)
    if not f16:   # the 1e-4 relative bar read as a row norm: o rows of the partials
        assert f32_margins(go[live], ro[live], "o partials") <= 1e-4
    assert_f32_close(gm[live], rm[live], "m partial", scalars=True)
    assert_f32_close(gl[live], rl[live], "l partial", scalars=True, rtol=rt)


# blocks of 64 and 32 keys run on the tensor core (split fp16 operands), 128-key blocks on
# fp32 FMA;
# qhead 3 leaves two rows of each 128-row tile unused
@pytest.mark.parametrize("head_dim,pages_per_block,qhead", [(128, 4, 4), (64, 2, 2),
                                                            (128, 8, 1), (128, 4, 3)])
def test_small_full_parity(head_dim, pages_per_block, qhead):
    c = wl.block_sparse(51, n_seqs=3, kv_len=1024, queries_per_seq=24, hq=4 * qhead,
                        hkv=4, head_dim=head_dim, pages_per_block=pages_per_block,
                        blocks_per_query=5, n_empty_edges=6, unmapped_frac=0.05)
    go, gm, gl, gout, glse, gst = run_gpu(c)
    ro, rm, rl, rst = oracle_partials(c)
    assert gst == rst
    compare_partials(go, gm, gl, ro, rm, rl, np.arange(rl.shape[0]))
    rout, rlse = orc.combine_partials(ro, rm, rl, c.seg_offsets, c.qhead)
    assert_f32_close(gout, rout, "combined output")
    assert f32_margins(gout, rout, "combined output") <= 1e-4
    fin = np.isfinite(rlse)
    np.testing.assert_array_equal(np.isfinite(glse), fin)
    assert_f32_close(glse[fin], rlse[fin], "lse", scalars=True)


# more than four query heads per kv head: the Q shifts do not fit the edge record and the
# tensor-core kernel reads them per row (and a 128-row tile holds 16 or 8 edges)
@pytest.mark.parametrize("qhead", [8, 16])
def test_many_query_heads_per_kv_head(qhead):
    c = wl.block_sparse(67, n_seqs=2, kv_len=1024, queries_per_seq=40, hq=2 * qhead, hkv=2,
                        head_dim=128, pages_per_block=4, blocks_per_query=5,
                        unmapped_frac=0.05)
    assert c.qhead == qhead
    go, gm, gl, gout, glse, gst = run_gpu(c)
    ro, rm, rl, rst = oracle_partials(c)
    assert gst == rst
    compare_partials(go, gm, gl, ro, rm, rl, np.arange(rl.shape[0]))
    rout, rlse = orc.combine_partials(ro, rm, rl, c.seg_offsets, c.qhead)
    assert f32_margins(gout, rout, "combined output, many query heads") <= 1e-4


# a query-row count (queries x query heads) that is not a multiple of 8: the split pass
# takes rows eight at a time
@pytest.mark.parametrize("head_dim,pages_per_block,qhead", [(128, 4, 3), (64, 2, 1)])
def test_ragged_query_rows(head_dim, pages_per_block, qhead):
    c = wl.block_sparse(61, n_seqs=3, kv_len=1024, queries_per_seq=25, hq=4 * qhead,
                        hkv=4, head_dim=head_dim, pages_per_block=pages_per_block,
                        blocks_per_query=5, unmapped_frac=0.05)
    assert (c.q.shape[0] * c.hq) % 8 != 0
    go, gm, gl, gout, glse, gst = run_gpu(c)
    ro, rm, rl, rst = oracle_partials(c)
    assert gst == rst
    compare_partials(go, gm, gl, ro, rm, rl, np.arange(rl.shape[0]))


# The tensor-core path scales each Q row and each K / V block by a power of two before
# splitting it into fp16 (hi, lo) pairs. Magnitudes far outside fp16's range (q x 2^eq,
# k x 2^ek, v x 2^ev, with eq + ek kept small so that the scores stay ordinary) and pages
# of different magnitude inside one block must give the same partials as the fp64 oracle.
@pytest.mark.parametrize("eq,ek,ev", [(40, -40, 60), (-50, 45, -70)])
def test_split_scaling_wide_magnitudes(eq, ek, ev):
    c = wl.block_sparse(57, n_seqs=2, kv_len=512, queries_per_seq=16, hq=16, hkv=4,
                        head_dim=128, pages_per_block=4, blocks_per_query=4,
                        unmapped_frac=0.05)
    page_f = 2.0 ** np.random.default_rng(7).integers(-3, 4, size=(c.k_pages.shape[0], 1, 1, 1))
    c.q = (c.q * 2.0 ** eq).astype(np.float32)
    c.k_pages = (c.k_pages * 2.0 ** ek * page_f).astype(np.float32)
    c.v_pages = (c.v_pages * 2.0 ** ev * page_f[::-1]).astype(np.float32)
    go, gm, gl, gout, glse, gst = run_gpu(c)
    ro, rm, rl, rst = oracle_partials(c)
    assert gst == rst
    compare_partials(go, gm, gl, ro, rm, rl, np.arange(rl.shape[0]))
    rout, _ = orc.combine_partials(ro, rm, rl, c.seg_offsets, c.qhead)
    assert f32_margins(gout, rout, "combined output, wide magnitudes") <= 1e-4


def test_groups_spanning_several_row_tiles():
    # 8 blocks per sequence and 96 queries naming 6 of them: about 72 edges x 4 query
    # heads = 288 rows per (sequence, block, kv head) group, i.e. three 128-row tiles
    c = wl.block_sparse(53, n_seqs=2, kv_len=512, queries_per_seq=96, hq=16, hkv=4,
                        head_dim=128, pages_per_block=4, blocks_per_query=6,
                        unmapped_frac=0.05)
    go, gm, gl, gout, glse, gst = run_gpu(c)
    ro, rm, rl, rst = oracle_partials(c)
    assert gst == rst
    compare_partials(go, gm, gl, ro, rm, rl, np.arange(rl.shape[0]))


@pytest.mark.parametrize("dtype", [np.float32, np.float16])
def test_groups_of_many_row_tiles(dtype):
    # 400 queries naming all 8 blocks of their sequence: 400 edges x 4 query heads per
    # (block, kv head) group, about 13 row tiles of one group in a row (more than the fp32
    # kernel's ring of per-tile scale slots, so its slots are reused inside a group)
    c = wl.block_sparse(59, n_seqs=1, kv_len=512, queries_per_seq=400, hq=16, hkv=4,
                        head_dim=128, pages_per_block=4, blocks_per_query=8,
                        unmapped_frac=0.05, dtype=dtype)
    go, gm, gl, gout, glse, gst = run_gpu(c)
    ro, rm, rl, rst = oracle_partials(c)
    assert gst == rst
    compare_partials(go, gm, gl, ro, rm, rl, np.arange(rl.shape[0]),
                     f16=np.dtype(dtype) == np.float16)


def test_bad_edges_and_pages_are_flagged():
    c = wl.block_sparse(52, n_seqs=2, kv_len=512, queries_per_seq=8, hq=8, hkv=2,
                        head_dim=128, blocks_per_query=3, unmapped_frac=0.0)
    c.edge_meta[0, 4] = 1000          # block_len past the block: clipped, flagged
    c.edge_meta[1, 0] = 9999          # q_idx out of range: empty partial, flagged
    c.block_tables[0, 3] = c.num_pages + 2   # page id past the pool: unmapped, flagged
    go, gm, gl, gout, glse, gst = run_gpu(c)
    ro, rm, rl, rst = oracle_partials(c)
    assert gst == rst == orc.ST_BAD_EDGE
    compare_partials(go, gm, gl, ro, rm, rl, np.arange(rl.shape[0]))


def test_block_sparse_full_size_sampled():
    """The full block-sparse workload (524 288 edges, 2 097 152 partials) in the same
    launch configuration as the benchmark; the oracle checks 1500 sampled edges plus
    every edge of 40 sampled (query, head) segments, whose combined rows are checked
    too."""
    c = wl.block_sparse(5, n_empty_edges=16)
    go, gm, gl, gout, glse, gst = run_gpu(c)
    rng = np.random.default_rng(7)
    segs = rng.choice(c.seg_offsets.shape[0] - 1, size=40, replace=False)
    edges = set(rng.choice(c.num_edges, size=1500, replace=False).tolist())
    for s in segs:
        edges |= set(range(int(c.seg_offsets[s]), int(c.seg_offsets[s + 1])))
    edges |= set(np.nonzero(c.edge_meta[:, 4] <= 0)[0].tolist())
    edges = sorted(edges)
    ro, rm, rl, rst = oracle_partials(c, edges)
    rows = (np.asarray(edges)[:, None] * c.qhead + np.arange(c.qhead)[None, :]).reshape(-1)
    compare_partials(go, gm, gl, ro, rm, rl, rows)
    for s in segs:
        e0, e1 = int(c.seg_offsets[s]), int(c.seg_offsets[s + 1])
        for qh in range(c.qhead):
            pr = [e * c.qhead + qh for e in range(e0, e1)]
            ref, rlse = orc.combine_rows(ro[pr], rm[pr], rl[pr])
            assert_f32_close(gout[s * c.qhead + qh], ref, "combined row")
            assert f32_margins(gout[s * c.qhead + qh], ref, "combined row") <= 1e-4


# fp16 q and pages: tensor-core kind::f16 kernel (blocks of 64 / 32 keys, qhead 3 and 1)
@pytest.mark.parametrize("head_dim,pages_per_block,qhead", [(128, 4, 4), (64, 2, 2),
                                                            (128, 2, 3), (64, 4, 1)])
def test_f16_small_full_parity(head_dim, pages_per_block, qhead):
    c = wl.block_sparse(54, n_seqs=3, kv_len=1024, queries_per_seq=24, hq=4 * qhead,
                        hkv=4, head_dim=head_dim, pages_per_block=pages_per_block,
                        blocks_per_query=5, n_empty_edges=6, unmapped_frac=0.05,
                        dtype=np.float16)
    go, gm, gl, gout, glse, gst = run_gpu(c)
    ro, rm, rl, rst = oracle_partials(c)
    assert gst == rst
    compare_partials(go, gm, gl, ro, rm, rl, np.arange(rl.shape[0]), f16=True)
    rout, rlse = orc.combine_partials(ro, rm, rl, c.seg_offsets, c.qhead)
    assert_f32_close(gout, rout, "combined output", rtol=F16_PARTIAL_RTOL)
    fin = np.isfinite(rlse)
    np.testing.assert_array_equal(np.isfinite(glse), fin)
    assert_f32_close(glse[fin], rlse[fin], "lse", scalars=True, rtol=F16_PARTIAL_RTOL)


def test_f16_groups_spanning_several_row_tiles_and_flags():
    c = wl.block_sparse(55, n_seqs=2, kv_len=512, queries_per_seq=96, hq=16, hkv=4,
                        head_dim=128, pages_per_block=4, blocks_per_query=6,
                        unmapped_frac=0.05, dtype=np.float16)
    c.edge_meta[0, 4] = 1000          # block_len past the block: clipped, flagged
    c.block_tables[1, 5] = c.num_pages + 2   # page id past the pool: flagged
    go, gm, gl, gout, glse, gst = run_gpu(c)
    ro, rm, rl, rst = oracle_partials(c)
    assert gst == rst == orc.ST_BAD_EDGE
    compare_partials(go, gm, gl, ro, rm, rl, np.arange(rl.shape[0]), f16=True)


def test_f16_block_sparse_full_size_sampled():
    """The block-sparse workload with fp16 q and pages, full size, in the benchmark's
    launch configuration; 1500 sampled edges and 40 whole segments against the oracle."""
    c = wl.block_sparse(5, n_empty_edges=16, dtype=np.float16)
    go, gm, gl, gout, glse, gst = run_gpu(c)
    rng = np.random.default_rng(8)
    segs = rng.choice(c.seg_offsets.shape[0] - 1, size=40, replace=False)
    edges = set(rng.choice(c.num_edges, size=1500, replace=False).tolist())
    for s in segs:
        edges |= set(range(int(c.seg_offsets[s]), int(c.seg_offsets[s + 1])))
    edges |= set(np.nonzero(c.edge_meta[:, 4] <= 0)[0].tolist())
    edges = sorted(edges)
    ro, rm, rl, rst = oracle_partials(c, edges)
    rows = (np.asarray(edges)[:, None] * c.qhead + np.arange(c.qhead)[None, :]).reshape(-1)
    compare_partials(go, gm, gl, ro, rm, rl, rows, f16=True)
    for s in segs:
        e0, e1 = int(c.seg_offsets[s]), int(c.seg_offsets[s + 1])
        for qh in range(c.qhead):
            pr = [e * c.qhead + qh for e in range(e0, e1)]
            ref, _ = orc.combine_rows(ro[pr], rm[pr], rl[pr])
            assert_f32_close(gout[s * c.qhead + qh], ref, "combined row",
                             rtol=F16_PARTIAL_RTOL)


def test_f16_rejects_blocks_past_64_keys():
    c = wl.block_sparse(56, n_seqs=1, kv_len=512, queries_per_seq=4, hq=4, hkv=1,
                        head_dim=128, pages_per_block=8, blocks_per_query=2,
                        dtype=np.float16)
    with pytest.raises(B.PagedKVError) as ei:
        run_gpu(c)
    assert ei.value.name == "PKV_ERR_UNSUPPORTED"


@pytest.mark.parametrize("dtype,head_dim", [(np.float16, 128), (np.float16, 64),
                                            (np.float32, 128)])
def test_blocks_of_eight_pages_of_eight_keys(dtype, head_dim):
    """64-key blocks of eight 8-key pages: the tensor-core kernels stage the most boxes per
    block (with head size 128, one for every lane of the staging warp)."""
    c = wl.block_sparse(58, n_seqs=2, kv_len=1024, queries_per_seq=24, hq=16, hkv=4,
                        head_dim=head_dim, page_size=8, pages_per_block=8,
                        blocks_per_query=5, n_empty_edges=3, unmapped_frac=0.05, dtype=dtype)
    go, gm, gl, gout, glse, gst = run_gpu(c)
    ro, rm, rl, rst = oracle_partials(c)
    assert gst == rst
    f16 = dtype == np.float16
    compare_partials(go, gm, gl, ro, rm, rl, np.arange(rl.shape[0]), f16=f16)
    rout, _ = orc.combine_partials(ro, rm, rl, c.seg_offsets, c.qhead)
    assert_f32_close(gout, rout, "combined output", rtol=F16_PARTIAL_RTOL if f16 else None)


@pytest.mark.parametrize("dtype,head_dim", [(np.float16, 128), (np.float16, 64),
                                            (np.float32, 128)])
def test_partials_at_16_byte_aligned_o(dtype, head_dim):
    """o_partial need only be 16-byte aligned: a 32-byte aligned o takes 32-byte stores, any
    other the 16-byte ones. Both write the same values (each partial row's arithmetic does
    not depend on where its row sits in a tile)."""
    c = wl.block_sparse(57, n_seqs=2, kv_len=1024, queries_per_seq=40, hq=16, hkv=4,
                        head_dim=head_dim, pages_per_block=4, blocks_per_query=5,
                        n_empty_edges=3, unmapped_frac=0.05, dtype=dtype)
    args = (dev(c.q), dev(c.k_pages), dev(c.v_pages), dev(c.edge_meta), dev(c.block_tables))
    kw = dict(qhead=c.qhead, block_size=c.block_size, page_size=c.page_size,
              pages_per_block=c.pages_per_block, softmax_scale=c.softmax_scale)
    P, D = c.num_edges * c.qhead, c.head_dim
    o32, m32, l32 = B.pkv_sparse_attention_partials(*args, **kw)
    buf = torch.full((P * D + 8,), 7.0, dtype=torch.float32, device=DEV)
    o16 = buf[4:4 + P * D].view(P, D)
    assert o32.data_ptr() % 32 == 0 and o16.data_ptr() % 32 == 16
    _, m16, l16 = B.pkv_sparse_attention_partials(*args, o=o16, **kw)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(o16), host(o32))
    np.testing.assert_array_equal(host(m16), host(m32))
    np.testing.assert_array_equal(host(l16), host(l32))
    edge = host(buf)   # nothing written outside o
    assert (edge[:4] == 7.0).all() and (edge[4 + P * D:] == 7.0).all()
    ro, rm, rl, _ = oracle_partials(c)
    compare_partials(host(o32), host(m32), host(l32), ro, rm, rl, np.arange(P),
                     f16=dtype == np.float16)


# right-aligned causal mask: split-fp16 tensor-core (64-key blocks), fp32 FMA (128-key
# blocks) and fp16 tensor-core paths
@pytest.mark.parametrize("head_dim,pages_per_block,qhead,dtype",
                         [(128, 4, 4, np.float32), (64, 8, 2, np.float32),
                          (128, 4, 3, np.float16), (64, 2, 2, np.float16)])
def test_causal_small_full_parity(head_dim, pages_per_block, qhead, dtype):
    c = wl.block_sparse(57, n_seqs=3, kv_len=1024, queries_per_seq=40, hq=4 * qhead,
                        hkv=4, head_dim=head_dim, pages_per_block=pages_per_block,
                        blocks_per_query=6, n_empty_edges=6, unmapped_frac=0.05, dtype=dtype)
    qpos = c.query_positions()
    bs = c.block_size
    starts = c.edge_meta[:, 2].astype(np.int64) * bs
    q_at = qpos[c.edge_meta[:, 0]]
    # blocks cut by the query position (and, for 32/64-key blocks, blocks wholly after it)
    assert ((starts <= q_at) & (q_at < starts + bs - 1)).any()
    assert bs > 64 or (starts > q_at).any()
    go, gm, gl, gout, glse, gst = run_gpu(c, qpos)
    ro, rm, rl, rst = oracle_partials(c, qpos=qpos)
    assert gst == rst
    f16 = dtype == np.float16
    compare_partials(go, gm, gl, ro, rm, rl, np.arange(rl.shape[0]), f16=f16)
    rout, rlse = orc.combine_partials(ro, rm, rl, c.seg_offsets, c.qhead)
    assert_f32_close(gout, rout, "combined output", rtol=F16_PARTIAL_RTOL if f16 else None)


@pytest.mark.parametrize("dtype", [np.float32, np.float16])
def test_causal_block_sparse_full_size_sampled(dtype):
    c = wl.block_sparse(5, dtype=dtype)
    qpos = c.query_positions()
    go, gm, gl, gout, glse, gst = run_gpu(c, qpos)
    rng = np.random.default_rng(9)
    edges = sorted(rng.choice(c.num_edges, size=1500, replace=False).tolist())
    ro, rm, rl, rst = oracle_partials(c, edges, qpos)
    rows = (np.asarray(edges)[:, None] * c.qhead + np.arange(c.qhead)[None, :]).reshape(-1)
    compare_partials(go, gm, gl, ro, rm, rl, rows, f16=dtype == np.float16)


@pytest.mark.parametrize("dtype", [np.float32, np.float16])
def test_no_edges_and_all_empty_edges(dtype):
    c = wl.block_sparse(58, n_seqs=2, kv_len=512, queries_per_seq=8, hq=8, hkv=2,
                        head_dim=128, blocks_per_query=3, dtype=dtype)
    # zero edges: nothing to compute, nothing written, no error
    c0 = wl.block_sparse(58, n_seqs=2, kv_len=512, queries_per_seq=8, hq=8, hkv=2,
                         head_dim=128, blocks_per_query=3, dtype=dtype)
    c0.edge_meta = c0.edge_meta[:0].copy()
    o, m, l = B.pkv_sparse_attention_partials(
        dev(c0.q), dev(c0.k_pages), dev(c0.v_pages), dev(c0.edge_meta),
        dev(c0.block_tables), qhead=c0.qhead, block_size=c0.block_size,
        page_size=c0.page_size, pages_per_block=c0.pages_per_block,
        softmax_scale=c0.softmax_scale)
    torch.cuda.synchronize()
    assert o.shape[0] == 0 and m.shape[0] == 0 and l.shape[0] == 0
    # every edge empty (block_len 0 or negative): every partial is the sentinel
    c.edge_meta = c.edge_meta.copy()
    c.edge_meta[:, 4] = np.where(np.arange(c.num_edges) % 2 == 0, 0, -5)
    go, gm, gl, gout, glse, gst = run_gpu(c)
    assert gst == 0
    assert (go == 0).all() and (gm == -1e30).all() and (gl == 0).all()
    assert (gout == 0).all() and np.isneginf(glse).all()
    # no query rows at all: every edge names a query out of range (flagged, sentinel)
    c2 = wl.block_sparse(58, n_seqs=2, kv_len=512, queries_per_seq=8, hq=8, hkv=2,
                         head_dim=128, blocks_per_query=3, dtype=dtype)
    c2.q = c2.q[:0].copy()
    go, gm, gl, gout, glse, gst = run_gpu(c2)
    ro, rm, rl, rst = oracle_partials(c2)
    assert gst == rst == orc.ST_BAD_EDGE
    compare_partials(go, gm, gl, ro, rm, rl, np.arange(rl.shape[0]), f16=dtype == np.float16)


def _random_partials(rng, n, D, empty_frac=0.2):
    o = rng.standard_normal((n, D)).astype(np.float32) * 3
    m = (rng.standard_normal(n) * 4).astype(np.float32)
    l = rng.uniform(0.5, 40, size=n).astype(np.float32)
    e = rng.random(n) < empty_frac
    o[e], m[e], l[e] = 0, -1e30, 0
    return o, m, l


@pytest.mark.parametrize("D,lanes,out_f16", [(128, 4, False), (64, 1, True), (128, 2, True)])
def test_combine_csr(D, lanes, out_f16):
    rng = np.random.default_rng(D + lanes)
    counts = rng.integers(0, 20, size=300)
    counts[:3] = [0, 1, 17]
    off = np.zeros(301, dtype=np.int32)
    off[1:] = np.cumsum(counts)
    o, m, l = _random_partials(rng, int(off[-1]) * lanes, D)
    lse = torch.empty(300 * lanes, dtype=torch.float32, device=DEV)
    out, _ = B.pkv_combine_partials(dev(o), dev(m), dev(l), dev(off), num_segments=300,
                                    lanes=lanes, lse=lse,
                                    out_dtype=torch.float16 if out_f16 else torch.float32)
    torch.cuda.synchronize()
    ref, rlse = orc.combine_partials(o, m, l, off, lanes)
    got = host(out).astype(np.float64)
    if out_f16:
        assert_f16_close(got, ref, "combine fp16")
    else:
        assert_f32_close(got, ref, "combine fp32")
    g = host(lse)
    fin = np.isfinite(rlse)
    np.testing.assert_array_equal(np.isfinite(g), fin)
    assert_f32_close(g[fin], rlse[fin], "lse", scalars=True)


def test_combine_uniform_segments():
    rng = np.random.default_rng(9)
    o, m, l = _random_partials(rng, 50 * 16, 128)
    out, _ = B.pkv_combine_partials(dev(o), dev(m), dev(l), None, num_segments=50, lanes=1,
                                    uniform_count=16)
    torch.cuda.synchronize()
    off = np.arange(0, 50 * 16 + 1, 16)
    ref, _ = orc.combine_partials(o, m, l, off, 1)
    assert_f32_close(host(out), ref, "uniform combine")
