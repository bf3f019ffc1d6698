"""Pins for the oracle's paged scatter / paged attention / split count (no GPU)."""
import math

import numpy as np
import pytest

from oracle import pagedkv_oracle as orc
from paged_kv_cache_231_gb300 import workloads as wl


def run(case, **kw):
    return orc.paged_attention(
        case.query, case.key, case.value, case.key_cache, case.value_cache,
        case.cu_seqlens, case.past_seqlens, case.block_table, case.slot_mapping,
        num_heads=case.num_heads, kv_num_heads=case.kv_num_heads, scale=case.scale,
        cos_cache=case.cos_cache, sin_cache=case.sin_cache, rotary_dim=case.rotary_dim,
        rotary_interleaved=case.rotary_interleaved, **kw)


def test_split_counts(golden):
    g = golden("paged_split_counts.json")
    for c in g["cases"]:
        got = orc.pages_num_splits(c["tokens"], c["kv_heads"], c["max_blocks"],
                                   c["block_size"])
        assert got == c["expected"], c
    s = g["scratch"]
    assert orc.pages_split_scratch_bytes(s["tokens"], s["num_heads"], s["head"],
                                         s["splits"]) == (s["expected_partial_bytes"],
                                                          s["expected_stats_bytes"])


def test_contract_cases(golden):
    g = golden("paged_contract.json")
    names = ["cacheShapeOk", "headLayoutOk", "scheduleShapeOk", "ioShapeOk",
             "separateKv", "packedKv", "slotShapeOk"]
    for c in g["cases"]:
        a = dict(g["base"])
        a.update(c["change"])
        r = orc.paged_contract(
            query_shape=a["query"], key_shape=a["key"], value_shape=a["value"],
            key_cache_shape=a["key_cache"], value_cache_shape=a["value_cache"],
            cu_shape=a["cu"], past_shape=a["past"], block_table_shape=a["block_table"],
            slot_mapping_shape=a["slot_mapping"], output_shape=a["output"],
            num_heads=a["num_heads"], kv_num_heads=a["kv_num_heads"], dtypes=a["dtypes"])
        assert sorted(n for n in names if not r[n]) == sorted(c["false"]), c["name"]
        assert r["pagedContractOk"] == c["ok"], c["name"]
        assert r["mode"] == c["mode"], c["name"]


def test_scatter_worked_example():
    # block_size 4, row [3, 1, -1], past 5, one new token: position 5 is column 1 ->
    # block 1, offset 1; slot mapping 1*4 + 1 = 5 names the same row.
    kc = np.zeros((4, 4, 1, 2), dtype=np.float16)
    k_new = np.array([[[7.0, 8.0]]], dtype=np.float16)
    v_new = np.array([[[9.0, 10.0]]], dtype=np.float16)
    bt = np.array([[3, 1, -1]], dtype=np.int32)
    a, b, st = orc.paged_scatter(k_new, v_new, kc, kc, [0, 1], [5], bt)
    assert st == 0
    assert a[1, 1, 0].tolist() == [7.0, 8.0] and b[1, 1, 0].tolist() == [9.0, 10.0]
    assert np.count_nonzero(a) == 2
    a2, b2, st2 = orc.paged_scatter(k_new, v_new, kc, kc, [0, 1], [5], bt, [5])
    np.testing.assert_array_equal(a, a2)
    np.testing.assert_array_equal(b, b2)
    # padding slot is skipped; slot past the pool is flagged
    a3, _, st3 = orc.paged_scatter(k_new, v_new, kc, kc, [0, 1], [5], bt, [-1])
    assert np.count_nonzero(a3) == 0 and st3 == 0
    _, _, st4 = orc.paged_scatter(k_new, v_new, kc, kc, [0, 1], [5], bt, [16])
    assert st4 == orc.ST_BAD_SLOT


def test_slot_mapping_equals_block_table_path():
    c = wl.paged_case(11, num_heads=4, kv_num_heads=2, head_size=8, block_size=4,
                      past=[3, 0, 9], new_tokens=[2, 5, 1], use_slot_mapping=True,
                      extra_blocks=3)
    o1, k1, v1, s1 = run(c)
    c.slot_mapping = None
    o2, k2, v2, s2 = run(c)
    np.testing.assert_array_equal(k1, k2)
    np.testing.assert_array_equal(v1, v2)
    np.testing.assert_array_equal(o1, o2)
    assert s1 == s2 == 0


def test_single_visible_key_returns_its_value():
    # past 0, one new token: the only visible key is the token's own, weight exactly 1
    c = wl.paged_case(12, num_heads=6, kv_num_heads=3, head_size=16, block_size=8,
                      past=[0, 0], new_tokens=[1, 1])
    out, kc, vc, st = run(c)
    v = c.value.reshape(2, 3, 16).astype(np.float64)
    expect = np.repeat(v, 2, axis=1).reshape(2, 6 * 16)
    np.testing.assert_array_equal(out, expect)


def test_equal_keys_give_mean_of_visible_values():
    c = wl.paged_case(13, num_heads=2, kv_num_heads=1, head_size=8, block_size=4,
                      past=[6], new_tokens=[3])
    c.key_cache[:] = 0.5
    c.key[:] = 0.5
    out, kc, vc, st = run(c)
    vals = vc[c.block_table[0, np.arange(9) // 4], np.arange(9) % 4, 0].astype(np.float64)
    for t in range(3):
        expect = vals[:6 + t + 1].mean(axis=0)
        np.testing.assert_allclose(out[t, :8], expect, rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(out[t, 8:], expect, rtol=1e-13, atol=1e-14)


def test_three_key_closed_form():
    # scores 0, 1, 2 with scale 1 -> weights (1, e, e^2) / (1 + e + e^2)
    kc = np.zeros((1, 4, 1, 2))
    vc = np.zeros((1, 4, 1, 2))
    kc[0, 0, 0] = [0, 5]
    kc[0, 1, 0] = [1, 0]
    vc[0, 0, 0] = [1, 0]
    vc[0, 1, 0] = [0, 1]
    q = np.array([[1.0, 0.0]])
    k_new = np.array([[2.0, 0.0]])
    v_new = np.array([[1.0, 1.0]])
    out, _, _, _ = orc.paged_attention(q, k_new, v_new, kc, vc, [0, 1], [2],
                                       np.array([[0]]), num_heads=1, kv_num_heads=1,
                                       scale=1.0)
    e = math.e
    Z = 1 + e + e * e
    np.testing.assert_allclose(out[0], [(1 + e * e) / Z, (e + e * e) / Z], rtol=1e-14)


def test_default_scale_is_inverse_sqrt_head():
    c = wl.paged_case(14, num_heads=2, kv_num_heads=1, head_size=16, block_size=4,
                      past=[5], new_tokens=[1])
    o1 = run(c)[0]
    c.scale = 0.0
    o0 = run(c)[0]
    c.scale = 0.25
    o2 = run(c)[0]
    np.testing.assert_array_equal(o0, o2)
    np.testing.assert_array_equal(o1, o2)


def brute_force(q, K, V, n_visible, scale):
    """Pure-Python softmax attention (no numpy): for tiny cross-checks."""
    s = [scale * sum(qi * ki for qi, ki in zip(q, K[j])) for j in range(n_visible)]
    mx = max(s)
    w = [math.exp(x - mx) for x in s]
    Z = sum(w)
    return [sum(w[j] * V[j][d] for j in range(n_visible)) / Z for d in range(len(V[0]))]


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_brute_force_tiny(seed):
    rng = np.random.default_rng(seed)
    B = 2
    past = rng.integers(0, 6, size=B)
    new = rng.integers(1, 4, size=B)
    c = wl.paged_case(100 + seed, num_heads=4, kv_num_heads=2, head_size=4,
                      block_size=2, past=past, new_tokens=new, extra_blocks=2,
                      packed=bool(seed % 2))
    out, kc, vc, st = run(c)
    assert st == 0
    k_new, v_new, q_all = orc.split_new_kv(c.query, c.key, c.value, 4, 2, 4)
    i = 0
    for b in range(B):
        # keys of sequence b in logical order: history from the prior cache, then new
        hist_k, hist_v = [], []
        for j in range(int(past[b])):
            blk = int(c.block_table[b, j // 2])
            hist_k.append(c.key_cache[blk, j % 2].astype(float).tolist())
            hist_v.append(c.value_cache[blk, j % 2].astype(float).tolist())
        for t in range(int(new[b])):
            hist_k.append(k_new[i + t].astype(float).tolist())
            hist_v.append(v_new[i + t].astype(float).tolist())
        for t in range(int(new[b])):
            for hq in range(4):
                h = hq // 2
                K = [row[h] for row in hist_k]
                V = [row[h] for row in hist_v]
                ref = brute_force(q_all[i + t, hq].astype(float).tolist(), K, V,
                                  int(past[b]) + t + 1, c.scale)
                np.testing.assert_allclose(out[i + t, hq * 4:(hq + 1) * 4], ref,
                                           rtol=1e-12, atol=1e-13)
        i += int(new[b])


def test_gqa_equals_mha_with_repeated_kv_heads():
    c = wl.paged_case(15, num_heads=6, kv_num_heads=2, head_size=8, block_size=4,
                      past=[4, 7], new_tokens=[2, 1])
    out_gqa = run(c)[0]
    rep = lambda x: np.repeat(x, 3, axis=-2)
    T = c.num_tokens
    m = wl.PagedCase(
        num_heads=6, kv_num_heads=6, head_size=8, block_size=4, query=c.query,
        key=rep(c.key.reshape(T, 2, 8)).reshape(T, 48),
        value=rep(c.value.reshape(T, 2, 8)).reshape(T, 48),
        key_cache=rep(c.key_cache), value_cache=rep(c.value_cache),
        cu_seqlens=c.cu_seqlens, past_seqlens=c.past_seqlens, block_table=c.block_table,
        slot_mapping=None, scale=c.scale)
    np.testing.assert_allclose(run(m)[0], out_gqa, rtol=1e-13, atol=1e-15)


def test_page_permutation_invariance():
    c = wl.paged_case(16, num_heads=4, kv_num_heads=2, head_size=8, block_size=4,
                      past=[5, 11, 0], new_tokens=[3, 1, 2], extra_blocks=4)
    out = run(c)[0]
    rng = np.random.default_rng(3)
    perm = rng.permutation(c.num_blocks)          # new block p holds old block perm[p]
    inv = np.argsort(perm)
    c.key_cache = c.key_cache[perm]
    c.value_cache = c.value_cache[perm]
    bt = c.block_table.copy()
    bt[bt >= 0] = inv[bt[bt >= 0]]
    c.block_table = bt
    np.testing.assert_array_equal(run(c)[0], out)


def test_causal_future_keys_do_not_matter():
    c = wl.paged_case(17, num_heads=2, kv_num_heads=1, head_size=8, block_size=4,
                      past=[3], new_tokens=[4])
    out = run(c)[0]
    c2 = wl.paged_case(17, num_heads=2, kv_num_heads=1, head_size=8, block_size=4,
                       past=[3], new_tokens=[4])
    c2.key[2:] = -c2.key[2:] * 3          # tokens 2, 3 change; tokens 0, 1 cannot see them
    c2.value[2:] = 7
    out2 = run(c2)[0]
    np.testing.assert_array_equal(out[:2], out2[:2])
    assert not np.array_equal(out[2:], out2[2:])


def test_weights_sum_to_one_and_follow_causal_limit():
    rng = np.random.default_rng(4)
    K = rng.standard_normal((20, 8))
    V = rng.standard_normal((20, 8))
    valid = np.ones(20, dtype=bool)
    valid[[3, 11]] = False
    q = rng.standard_normal((5, 8))
    limits = np.array([0, 3, 7, 15, 19])
    out, w = orc.attention_rows(q, K, V, valid, limits, 0.3, return_weights=True)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    j = np.arange(20)
    assert np.all(w[~(valid[None, :] & (j[None, :] <= limits[:, None]))] == 0)
    np.testing.assert_allclose(out, w @ V, rtol=1e-14)


def test_unmapped_blocks_are_excluded_and_flagged():
    c = wl.paged_case(18, num_heads=2, kv_num_heads=1, head_size=8, block_size=4,
                      past=[9], new_tokens=[1])
    full = run(c)[0]
    c.block_table[0, 0] = -1          # keys 0..3 become unmapped
    out, kc, vc, st = run(c)
    assert st & orc.ST_BAD_BLOCK
    K, V, valid = orc.gather_sequence_kv(kc, vc, c.block_table[0], 10)
    assert valid.tolist() == [False] * 4 + [True] * 6
    q = c.query.reshape(2, 8).astype(np.float64)
    ref = orc.attention_rows(q, K[:, 0], V[:, 0], valid, [9, 9], c.scale)
    np.testing.assert_allclose(out[0].reshape(2, 8), ref, rtol=1e-14)
    assert not np.allclose(full, out)


def test_rotary_on_append_rotates_new_keys_at_absolute_position():
    c = wl.paged_case(19, num_heads=4, kv_num_heads=2, head_size=16, block_size=4,
                      past=[6, 2], new_tokens=[2, 3], rotary_dim=8)
    out, kc, vc, st = run(c)
    k_new, v_new, _ = orc.split_new_kv(c.query, c.key, c.value, 4, 2, 16)
    smap, _ = orc.sequence_map(c.cu_seqlens, c.past_seqlens)
    for i, (b, t, pos) in enumerate(smap):
        blk = c.block_table[b, pos // 4]
        expect = orc.rotate_rows(k_new[i], [pos, pos], c.cos_cache, c.sin_cache, 8, False)
        np.testing.assert_array_equal(kc[blk, pos % 4], expect.astype(np.float16))
        np.testing.assert_array_equal(kc[blk, pos % 4, :, 8:], k_new[i, :, 8:])
        np.testing.assert_array_equal(vc[blk, pos % 4], v_new[i])


def test_split_then_combine_equals_unsplit():
    rng = np.random.default_rng(5)
    n, D = 37, 8
    K = rng.standard_normal((n, D))
    V = rng.standard_normal((n, D))
    q = rng.standard_normal(D)
    valid = np.ones(n, dtype=bool)
    full = orc.attention_rows(q[None], K, V, valid, [n - 1], 0.4)[0]
    for cuts in ([0, n], [0, 5, 6, 30, n], [0, 0, 12, 12, n], list(range(0, n + 1))):
        parts = []
        for a, b in zip(cuts[:-1], cuts[1:]):
            vis = np.zeros(n, dtype=bool)
            vis[a:b] = True
            parts.append(orc.attention_partial(q, K, V, vis, 0.4))
        o = np.array([p[0] for p in parts])
        m = np.array([p[1] for p in parts])
        l = np.array([p[2] for p in parts])
        out, lse = orc.combine_rows(o, m, l)
        np.testing.assert_allclose(out, full, rtol=1e-12, atol=1e-14)
        s = 0.4 * (K @ q)
        np.testing.assert_allclose(lse, np.log(np.exp(s).sum()), rtol=1e-13)


def test_llama8b_workload_shape():
    c = wl.llama8b_decode(batch=4, fill_cache=False)
    assert c.num_tokens == 4 and c.max_blocks == 512
    n = c.context_lengths()
    assert ((n >= 512) & (n <= 8192)).all()
    assert (np.diff(c.cu_seqlens) == 1).all()
    used = c.block_table[c.block_table >= 0]
    assert len(set(used.tolist())) == used.size == c.num_blocks


def test_invalid_sequence_and_uncovered_tokens():
    c = wl.paged_case(20, num_heads=2, kv_num_heads=1, head_size=8, block_size=4,
                      past=[3, 2, 5], new_tokens=[2, 1, 2])
    good = run(c)
    # sequence 1 gets a negative past: its token is neither scattered nor attended
    c.past_seqlens = c.past_seqlens.copy()
    c.past_seqlens[1] = -1
    out, kc, vc, st = run(c)
    assert st & orc.ST_BAD_SEQUENCE
    assert (out[2] == 0).all()
    np.testing.assert_array_equal(out[[0, 1, 3, 4]], good[0][[0, 1, 3, 4]])
    # cu ends before the last token: that token is padding (zero output, no flag)
    c2 = wl.paged_case(20, num_heads=2, kv_num_heads=1, head_size=8, block_size=4,
                       past=[3, 2, 5], new_tokens=[2, 1, 2])
    c2.cu_seqlens = c2.cu_seqlens.copy()
    c2.cu_seqlens[3] = 4
    out2, _, _, st2 = run(c2)
    assert st2 == 0 and (out2[4] == 0).all()
    np.testing.assert_array_equal(out2[:4], good[0][:4])


def test_rotary_position_past_table_skips_token():
    c = wl.paged_case(21, num_heads=2, kv_num_heads=1, head_size=8, block_size=4,
                      past=[5], new_tokens=[2], rotary_dim=8)
    c.cos_cache = c.cos_cache[:6]
    c.sin_cache = c.sin_cache[:6]
    k_new, v_new, _ = orc.split_new_kv(c.query, c.key, c.value, 2, 1, 8)
    kc, vc, st = orc.paged_scatter(k_new, v_new, c.key_cache, c.value_cache, c.cu_seqlens,
                                   c.past_seqlens, c.block_table, None, c.cos_cache,
                                   c.sin_cache, 8, False)
    assert st == orc.ST_BAD_POSITION
    blk6 = c.block_table[0, 6 // 4]
    np.testing.assert_array_equal(kc[blk6, 6 % 4], c.key_cache[blk6, 6 % 4])   # skipped
    blk5 = c.block_table[0, 5 // 4]
    assert not np.array_equal(kc[blk5, 5 % 4], c.key_cache[blk5, 5 % 4])       # written
