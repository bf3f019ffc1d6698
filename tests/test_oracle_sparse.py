"""Pins for the oracle's block-sparse partials and the LSE combine (no GPU)."""
import math

import numpy as np
import pytest

from oracle import pagedkv_oracle as orc
from paged_kv_cache_231_gb300 import workloads as wl


def sp(q, kp, vp, meta, bt, qh=0, **kw):
    args = dict(qhead=1, hq=1, head_dim=q.shape[-1], block_size=4, page_size=2,
                pages_per_block=2, softmax_scale=1.0)
    args.update(kw)
    return orc.sparse_partial(q, kp, vp, meta, bt, qh, **args)


def tiny_pages():
    kp = np.zeros((2, 1, 2, 2))
    vp = np.zeros((2, 1, 2, 2))
    kp[1, 0, 0] = [1, 0]     # key t = 0: score 1
    kp[1, 0, 1] = [0, 0]     # key t = 1: score 0
    vp[1, 0, 0] = [2, 0]
    vp[1, 0, 1] = [0, 4]
    q = np.array([[[1.0, 0.0]]])
    bt = np.array([[1, -1]])  # page slot 0 -> page 1, page slot 1 unmapped
    return q, kp, vp, bt


def test_worked_example_with_unmapped_page():
    q, kp, vp, bt = tiny_pages()
    o, m, l, st = sp(q, kp, vp, [0, 0, 0, 0, 3], bt)
    # keys 0, 1 mapped (scores 1, 0), key 2 unmapped: m = 1, weights (1, e^-1, 0)
    assert m == 1.0 and st == 0
    assert l == pytest.approx(1 + math.exp(-1), rel=1e-15)
    np.testing.assert_allclose(o, [2.0, 4 * math.exp(-1)], rtol=1e-15)


@pytest.mark.parametrize("block_len", [0, -1, -100])
def test_empty_edge_sentinel(block_len):
    q, kp, vp, bt = tiny_pages()
    o, m, l, st = sp(q, kp, vp, [0, 0, 0, 0, block_len], bt)
    assert m == -1e30 and l == 0.0 and (o == 0).all()


def test_all_unmapped_gives_sentinel():
    q, kp, vp, _ = tiny_pages()
    o, m, l, st = sp(q, kp, vp, [0, 0, 0, 0, 4], np.array([[-1, -1]]))
    assert m == -1e30 and l == 0.0 and (o == 0).all()


def test_single_key_gives_value_score_one():
    q, kp, vp, bt = tiny_pages()
    o, m, l, st = sp(q, kp, vp, [0, 0, 0, 0, 1], bt, softmax_scale=0.5)
    assert m == 0.5 and l == 1.0
    np.testing.assert_array_equal(o, [2.0, 0.0])


def test_block_len_above_block_is_clipped_and_flagged():
    q, kp, vp, bt = tiny_pages()
    a = sp(q, kp, vp, [0, 0, 0, 0, 4], bt)
    b = sp(q, kp, vp, [0, 0, 0, 0, 9], bt)
    np.testing.assert_array_equal(a[0], b[0])
    assert a[1:3] == b[1:3] and a[3] == 0 and b[3] == orc.ST_BAD_EDGE


def test_partial_is_unnormalised_softmax_pieces():
    c = wl.block_sparse(21, n_seqs=1, kv_len=256, queries_per_seq=4, hq=4, hkv=2,
                        head_dim=8, blocks_per_query=3, unmapped_frac=0.0)
    e = 5
    qh = 1
    meta = c.edge_meta[e]
    o, m, l, st = orc.sparse_partial(
        c.q, c.k_pages, c.v_pages, meta, c.block_tables, qh, qhead=2, hq=4, head_dim=8,
        block_size=64, page_size=16, pages_per_block=4, softmax_scale=c.softmax_scale)
    q_idx, h, blk, b, bl = (int(x) for x in meta)
    K = np.stack([c.k_pages[c.block_tables[b, blk * 4 + t // 16], h, t % 16]
                  for t in range(bl)]).astype(np.float64)
    V = np.stack([c.v_pages[c.block_tables[b, blk * 4 + t // 16], h, t % 16]
                  for t in range(bl)]).astype(np.float64)
    s = c.softmax_scale * K @ c.q[q_idx, h * 2 + qh].astype(np.float64)
    assert m == pytest.approx(s.max(), rel=1e-15)
    assert l == pytest.approx(np.exp(s - s.max()).sum(), rel=1e-14)
    soft = orc.attention_rows(c.q[q_idx, h * 2 + qh][None], K, V, np.ones(bl, bool),
                              [bl], c.softmax_scale)[0]
    np.testing.assert_allclose(o / l, soft, rtol=1e-12, atol=1e-14)


def test_sparse_partials_then_combine_equals_dense_over_all_blocks():
    # If the edges of (q, h) cover every block of the sequence, the combined result is
    # plain (non-causal) softmax attention over all the sequence's used keys.
    c = wl.block_sparse(22, n_seqs=2, kv_len=256, queries_per_seq=3, hq=4, hkv=2,
                        head_dim=8, blocks_per_query=4, unmapped_frac=0.0, clip_max=40)
    o, m, l, st = orc.sparse_attention_partials(
        c.q, c.k_pages, c.v_pages, c.edge_meta, c.block_tables, qhead=2, hq=4,
        head_dim=8, block_size=64, page_size=16, pages_per_block=4,
        softmax_scale=c.softmax_scale)
    out, lse = orc.combine_partials(o, m, l, c.seg_offsets, 2)
    for q_idx in range(c.q.shape[0]):
        b = q_idx // 3
        n = int(c.used_kv_lens[b])
        pages = c.block_tables[b, np.arange(n) // 16]
        for h in range(2):
            K = c.k_pages[pages, h, np.arange(n) % 16].astype(np.float64)
            V = c.v_pages[pages, h, np.arange(n) % 16].astype(np.float64)
            for qh in range(2):
                ref = orc.attention_rows(c.q[q_idx, h * 2 + qh][None], K, V,
                                         np.ones(n, bool), [n], c.softmax_scale)[0]
                row = (q_idx * 2 + h) * 2 + qh
                np.testing.assert_allclose(out[row], ref, rtol=1e-11, atol=1e-13)
                s = c.softmax_scale * K @ c.q[q_idx, h * 2 + qh].astype(np.float64)
                assert lse[row] == pytest.approx(np.log(np.exp(s).sum()), rel=1e-12)


def test_combine_single_partial_is_o_over_l():
    o = np.array([[2.0, -4.0]])
    out, lse = orc.combine_rows(o, [3.0], [2.0])
    assert out.tolist() == [1.0, -2.0]
    assert lse == pytest.approx(3.0 + math.log(2.0), rel=1e-15)


def test_combine_ignores_empty_partials_and_all_empty_is_zero():
    o = np.array([[2.0, -4.0], [0.0, 0.0], [1.0, 1.0]])
    out, lse = orc.combine_rows(o, [3.0, -1e30, 5.0], [2.0, 0.0, 1.0])
    out2, lse2 = orc.combine_rows(o[[0, 2]], [3.0, 5.0], [2.0, 1.0])
    np.testing.assert_array_equal(out, out2)
    assert lse == lse2
    z, zl = orc.combine_rows(np.zeros((2, 2)), [-1e30, -1e30], [0.0, 0.0])
    assert (z == 0).all() and zl == -math.inf


def test_combine_two_partials_closed_form():
    # partials (o1, m1, l1) = ([1, 0], 0, 1), (o2, m2, l2) = ([0, 2], ln 3, 2):
    # M = ln 3, weights (1/3, 1), L = 1/3 + 2 = 7/3, out = ([1/3, 0] + [0, 2]) / (7/3)
    out, lse = orc.combine_rows(np.array([[1.0, 0.0], [0.0, 2.0]]), [0.0, math.log(3)],
                                [1.0, 2.0])
    np.testing.assert_allclose(out, [1 / 7, 6 / 7], rtol=1e-14)
    assert lse == pytest.approx(math.log(3) + math.log(7 / 3), rel=1e-14)


def test_combine_is_associative():
    rng = np.random.default_rng(6)
    o = rng.standard_normal((6, 4))
    m = rng.standard_normal(6) * 3
    l = rng.uniform(0.5, 5, size=6)
    full, lse = orc.combine_rows(o, m, l)
    a, la = orc.combine_rows(o[:2], m[:2], l[:2])
    b, lb = orc.combine_rows(o[2:], m[2:], l[2:])
    # a combined result re-enters as a partial with o = out, m = lse, l = 1
    ab, lab = orc.combine_rows(np.stack([a, b]), [la, lb], [1.0, 1.0])
    np.testing.assert_allclose(ab, full, rtol=1e-13)
    assert lab == pytest.approx(lse, rel=1e-14)


def test_combine_csr_layout():
    # segment s, lane c reads partial rows e*lanes + c for e in [off[s], off[s+1])
    o = np.arange(12, dtype=np.float64).reshape(6, 2)
    m = np.zeros(6)
    l = np.ones(6)
    out, lse = orc.combine_partials(o, m, l, [0, 1, 3, 3], 2)
    assert out.shape == (6, 2)
    np.testing.assert_array_equal(out[0], o[0])
    np.testing.assert_array_equal(out[1], o[1])
    np.testing.assert_array_equal(out[2], (o[2] + o[4]) / 2)
    np.testing.assert_array_equal(out[3], (o[3] + o[5]) / 2)
    assert (out[4:] == 0).all() and np.isneginf(lse[4:]).all()


def test_block_sparse_workload_structure():
    c = wl.block_sparse(23, n_seqs=2, kv_len=1024, queries_per_seq=8, hq=8, hkv=2,
                        head_dim=16, n_empty_edges=4)
    em = c.edge_meta
    keys = em[:, 0].astype(np.int64) * 1000000 + em[:, 1] * 1000 + em[:, 2]
    assert (np.diff(keys) > 0).all()            # sorted by (q, h, blk), distinct blocks
    assert (np.diff(c.seg_offsets) == 16).all()
    BSZ = 64
    for q_idx in range(16):
        b = q_idx // 8
        pos = c.used_kv_lens[b] - 8 + q_idx % 8
        for h in range(2):
            blks = em[c.seg_offsets[q_idx * 2 + h]:c.seg_offsets[q_idx * 2 + h + 1], 2]
            assert pos // BSZ in blks
            assert blks.max() <= (c.used_kv_lens[b] - 1) // BSZ
    assert (em[:, 4] <= 0).sum() == 4


def test_out_of_range_edge_fields_give_flagged_sentinel():
    q, kp, vp, bt = tiny_pages()
    for meta in ([1, 0, 0, 0, 3], [0, 1, 0, 0, 3], [0, 0, 0, 1, 3], [0, 0, -1, 0, 3],
                 [0, 0, 1, 0, 3]):
        o, m, l, st = sp(q, kp, vp, meta, bt)
        assert m == -1e30 and l == 0.0 and (o == 0).all() and st == orc.ST_BAD_EDGE, meta
    # an empty edge is never flagged, whatever its other fields hold
    o, m, l, st = sp(q, kp, vp, [9, 9, 9, 9, 0], bt)
    assert st == 0 and l == 0.0


# ---- right-aligned causal mask (the sparse page leaves it unimplemented) -------------
def test_causal_partials_then_combine_equals_dense_causal_attention():
    # Edges covering every block of the sequence: with the right-aligned causal mask the
    # combined result is softmax attention of the query at position p over keys 0..p,
    # computed here directly.
    c = wl.block_sparse(23, n_seqs=2, kv_len=256, queries_per_seq=70, hq=4, hkv=2,
                        head_dim=8, blocks_per_query=4, unmapped_frac=0.0, clip_max=40)
    pos = c.query_positions()
    assert pos.min() < 256 - 64   # some queries sit before the last block
    o, m, l, st = orc.sparse_attention_partials(
        c.q, c.k_pages, c.v_pages, c.edge_meta, c.block_tables, qhead=2, hq=4,
        head_dim=8, block_size=64, page_size=16, pages_per_block=4,
        softmax_scale=c.softmax_scale, query_positions=pos)
    assert st == 0
    out, lse = orc.combine_partials(o, m, l, c.seg_offsets, 2)
    for q_idx in range(0, c.q.shape[0], 7):
        b = q_idx // 70
        n = int(pos[q_idx]) + 1
        pages = c.block_tables[b, np.arange(n) // 16]
        for h in range(2):
            K = c.k_pages[pages, h, np.arange(n) % 16].astype(np.float64)
            V = c.v_pages[pages, h, np.arange(n) % 16].astype(np.float64)
            for qh in range(2):
                s = c.softmax_scale * (K @ c.q[q_idx, h * 2 + qh].astype(np.float64))
                w = np.exp(s - s.max())
                row = (q_idx * 2 + h) * 2 + qh
                np.testing.assert_allclose(out[row], (w / w.sum()) @ V, rtol=1e-11,
                                           atol=1e-13)
                assert lse[row] == pytest.approx(s.max() + np.log(w.sum()), rel=1e-12)


def test_causal_mask_keeps_the_keys_up_to_the_query():
    q, kp, vp, bt = tiny_pages()
    bt = np.array([[1, 0]])
    kp[0, 0, 0] = [3, 0]                      # key t = 2 (block 0, page slot 1)
    meta = [0, 0, 0, 0, 4]
    full = sp(q, kp, vp, meta, bt)
    # query at position 1: keys 0 and 1 only = the unmasked partial of block_len 2
    o, m, l, st = sp(q, kp, vp, meta, bt, query_positions=[1])
    o2, m2, l2, _ = sp(q, kp, vp, [0, 0, 0, 0, 2], bt)
    np.testing.assert_allclose(o, o2, rtol=1e-15)
    assert (m, l) == (m2, l2) and st == 0
    assert m == 1.0 and m != full[1]          # key 2 (score 3) is masked out
    # query at position 3 or later sees the whole block
    np.testing.assert_allclose(sp(q, kp, vp, meta, bt, query_positions=[9])[0], full[0])


def test_causal_block_after_the_query_is_the_empty_partial_and_unread():
    q, kp, vp, bt = tiny_pages()
    bt = np.array([[1, -1, 99, 99]])          # block 1 names a page past the pool
    o, m, l, st = sp(q, kp, vp, [0, 0, 1, 0, 4], bt, query_positions=[3])
    assert (o == 0).all() and m == orc.NEG_LARGE and l == 0 and st == 0
    # without the mask the bad page is read and flagged
    assert sp(q, kp, vp, [0, 0, 1, 0, 4], bt)[3] == orc.ST_BAD_EDGE
