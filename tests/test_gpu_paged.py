"""GPU parity of pkv_paged_attention / pkv_paged_scatter_kv against the oracle."""
import numpy as np
import pytest
import torch

from oracle import pagedkv_oracle as orc
from paged_kv_cache_231_gb300 import binding as B
from paged_kv_cache_231_gb300 import workloads as wl

from .gpu_util import (DEV, assert_f16_close, compare_caches, dev, host, run_paged_gpu,
                       run_paged_oracle)

pytestmark = pytest.mark.gpu


def check(case, tokens=None, rotary_query=False, **kw):
    g = run_paged_gpu(case, rotary_query=rotary_query, **kw)
    r = run_paged_oracle(case, tokens, rotary_query=rotary_query)
    rows = slice(None) if tokens is None else np.asarray(tokens)
    err = assert_f16_close(g.out[rows], r.out[rows], "attention output")
    compare_caches(g, r, case.rotary_dim > 0, "caches")
    assert g.status == r.status, (g.status, r.status)
    return err


def test_tiny_decode():
    # every sequence fits one split: scatter and attention run as one launch
    before = B.pkv_launch_count()
    check(wl.tiny_decode())
    assert B.pkv_launch_count() - before == 1


CASES = [
    # (seed, Hq, Hkv, D, BS, past, new, packed, slot)
    (31, 8, 2, 128, 16, [0, 1, 63, 64, 65, 200, 1000], [1] * 7, False, False),
    (32, 4, 2, 64, 32, [0, 17, 300, 5], [5, 70, 33, 8], True, False),
    (33, 4, 4, 128, 8, [3, 0, 129, 1], [1, 16, 17, 40], False, True),
    (34, 16, 2, 128, 16, [100, 7, 640], [2, 3, 9], False, False),
    (35, 16, 1, 128, 16, [50, 0, 300], [1, 1, 2], True, True),
    (36, 6, 2, 64, 16, [10, 90, 3], [5, 6, 21], False, False),
    (37, 8, 2, 128, 5, [12, 0, 77], [1, 30, 4], False, True),
    (38, 4, 1, 64, 64, [1000, 2, 0], [1, 200, 129], True, False),
    # tensor-core prefill: 16-key boxes over 48-key blocks, 126-row tiles (G = 3)
    (39, 6, 2, 128, 48, [0, 200, 33], [150, 7, 300], False, True),
    # tensor-core prefill: 128-key boxes inside 256-key blocks
    (30, 8, 1, 128, 256, [0, 700], [260, 129], True, False),
]


@pytest.mark.parametrize("case", CASES, ids=[str(c[0]) for c in CASES])
def test_random_shapes(case):
    seed, Hq, Hkv, D, BS, past, new, packed, slot = case
    c = wl.paged_case(seed, num_heads=Hq, kv_num_heads=Hkv, head_size=D, block_size=BS,
                      past=past, new_tokens=new, packed=packed, use_slot_mapping=slot,
                      extra_blocks=3)
    check(c)


@pytest.mark.parametrize("case", CASES, ids=[str(c[0]) for c in CASES])
def test_single_pass_shapes(case):
    """With one split per sequence, small calls take the single-pass kernel (one CTA per
    (sequence, kv head) scatters, then attends every row of its sequence, prefill rows
    included) and launch nothing else."""
    seed, Hq, Hkv, D, BS, past, new, packed, slot = case
    c = wl.paged_case(seed, num_heads=Hq, kv_num_heads=Hkv, head_size=D, block_size=BS,
                      past=past, new_tokens=new, packed=packed, use_slot_mapping=slot,
                      extra_blocks=3)
    before = B.pkv_launch_count()
    check(c, max_splits=1)
    assert B.pkv_launch_count() - before == 1


@pytest.mark.parametrize("D,rotary_dim,inter", [(128, 128, False), (64, 12, True)])
def test_single_pass_rotary_query(D, rotary_dim, inter):
    c = wl.paged_case(44, num_heads=8, kv_num_heads=2, head_size=D, block_size=16,
                      past=[5, 300, 0, 1000], new_tokens=[1, 40, 130, 1], packed=True,
                      rotary_dim=rotary_dim, rotary_interleaved=inter)
    check(c, rotary_query=True, max_splits=1)


def test_single_pass_invalid_sequence_padding_and_slots():
    c = wl.paged_case(46, num_heads=4, kv_num_heads=2, head_size=64, block_size=16,
                      past=[10, 20, 30], new_tokens=[3, 2, 2], use_slot_mapping=True)
    c.past_seqlens[1] = -4                      # invalid sequence: zero output, flagged
    c.slot_mapping[0] = -1                      # padding: not written
    c.slot_mapping[6] = c.num_blocks * 16 + 7   # past the pool: flagged, not written
    check(c, max_splits=1)
    c2 = wl.paged_case(46, num_heads=4, kv_num_heads=2, head_size=64, block_size=16,
                       past=[10, 20, 30], new_tokens=[3, 2, 2])
    c2.cu_seqlens[3] = 5                        # last 2 tokens are padding: zero output
    g = run_paged_gpu(c2, max_splits=1)
    r = run_paged_oracle(c2)
    assert (g.out[5:] == 0).all() and g.status == r.status == 0
    assert_f16_close(g.out, r.out, "padded batch, single pass")


def test_one_split_without_combine():
    """One split per sequence but too much work for the single-pass kernel: the split
    kernel writes the output itself and no combine is launched."""
    c = wl.paged_case(49, num_heads=8, kv_num_heads=2, head_size=128, block_size=16,
                      past=[0, 63, 5000, 130], new_tokens=[300, 1, 1, 2])
    B.pkv_profiler_reset()
    B.pkv_profiler_enable(True)
    try:
        check(c, split_policy=B.PKV_SPLIT_FIXED, fixed_splits=1)
        assert B.pkv_profiler_query("combine")[1] == 0
        assert B.pkv_profiler_query("single_pass")[1] == 0
        assert B.pkv_profiler_query("decode_split")[1] == 1
    finally:
        B.pkv_profiler_enable(False)
        B.pkv_profiler_reset()


@pytest.mark.parametrize("splits", [1, 2, 3, 5, 7, 16])
def test_forced_splits_match_unsplit(splits):
    c = wl.paged_case(40, num_heads=8, kv_num_heads=2, head_size=128, block_size=16,
                      past=[0, 63, 64, 130, 1500, 2047], new_tokens=[1, 1, 1, 2, 1, 4])
    check(c, split_policy=B.PKV_SPLIT_FIXED, fixed_splits=splits)


def test_pages_split_policy():
    c = wl.paged_case(41, num_heads=8, kv_num_heads=2, head_size=128, block_size=16,
                      past=[500, 900], new_tokens=[1, 1])
    check(c, split_policy=B.PKV_SPLIT_PAGES)


# rotary_dim 12 keeps rotation pairs across 8-element chunks: the per-chunk fallback path
@pytest.mark.parametrize("rotary_dim,inter", [(128, False), (64, True), (32, False),
                                              (12, False), (12, True)])
def test_rotary_on_append(rotary_dim, inter):
    c = wl.paged_case(42, num_heads=8, kv_num_heads=2, head_size=128, block_size=16,
                      past=[5, 300, 0], new_tokens=[1, 40, 3], rotary_dim=rotary_dim,
                      rotary_interleaved=inter)
    check(c)


# query heads rotated with the keys: decode (stream-K), tensor-core prefill (head 128,
# blocks of 16) and mma.sync prefill (head 64) read the rotated query from the workspace
@pytest.mark.parametrize("D,rotary_dim,inter,packed", [(128, 128, False, False),
                                                       (128, 64, True, True),
                                                       (128, 12, False, False),
                                                       (64, 64, False, True),
                                                       (64, 12, True, False)])
def test_rotary_query(D, rotary_dim, inter, packed):
    c = wl.paged_case(44, num_heads=8, kv_num_heads=2, head_size=D, block_size=16,
                      past=[5, 300, 0, 1000], new_tokens=[1, 40, 130, 1], packed=packed,
                      rotary_dim=rotary_dim, rotary_interleaved=inter)
    check(c, rotary_query=True)


def test_rotary_query_with_slot_padding():
    # a padding slot skips the key write but the token still attends (over the stale row)
    # with its query rotated; the oracle does the same
    c = wl.paged_case(46, num_heads=8, kv_num_heads=2, head_size=128, block_size=16,
                      past=[7, 40], new_tokens=[3, 1], use_slot_mapping=True,
                      rotary_dim=128, extra_blocks=2)
    c.slot_mapping = c.slot_mapping.copy()
    c.slot_mapping[1] = -1
    check(c, rotary_query=True)


def test_rotary_query_position_past_table():
    c = wl.paged_case(45, num_heads=4, kv_num_heads=1, head_size=128, block_size=16,
                      past=[5, 60], new_tokens=[3, 1], rotary_dim=128)
    c.cos_cache = c.cos_cache[:7]     # token 2 of sequence 0 and sequence 1: past the table
    c.sin_cache = c.sin_cache[:7]
    check(c, rotary_query=True)


def test_llama8b_decode_full_size():
    """The benchmark workload at full size (64 sequences, contexts 512..8192), in the
    launch configuration the benchmark times; every output element is compared."""
    c = wl.llama8b_decode()
    check(c)


def test_varlen_mixed_sampled():
    """Mixed prefill + decode batch at full size; the oracle evaluates every decode
    token, the first and last token of every prefill sequence (first tile, diagonal,
    ragged tail) and every 41st token in between."""
    c = wl.varlen_mixed()
    tokens = set()
    for b in range(c.batch):
        lo, hi = int(c.cu_seqlens[b]), int(c.cu_seqlens[b + 1])
        tokens |= {lo, hi - 1} | set(range(lo, hi, 41))
        tokens |= set(range(max(lo, hi - 70), hi))
    check(c, tokens=sorted(tokens))


def test_empty_batch_is_a_no_op():
    c = wl.paged_case(43, num_heads=4, kv_num_heads=2, head_size=64, block_size=16,
                      past=[3, 4], new_tokens=[0, 0])
    g = run_paged_gpu(c)
    assert g.out.shape == (0, 256)
    np.testing.assert_array_equal(g.kc, c.key_cache)


def test_unmapped_block_is_masked_and_flagged():
    c = wl.paged_case(44, num_heads=8, kv_num_heads=2, head_size=128, block_size=16,
                      past=[100, 40], new_tokens=[1, 20])
    c.block_table[0, 2] = -1
    c.block_table[1, 0] = c.num_blocks + 5
    g = check(c)


def test_slot_padding_and_bad_slot():
    c = wl.paged_case(45, num_heads=4, kv_num_heads=2, head_size=64, block_size=16,
                      past=[10, 20], new_tokens=[3, 2], use_slot_mapping=True)
    c.slot_mapping[1] = -1                      # padding: not written
    c.slot_mapping[3] = c.num_blocks * 16 + 7   # past the pool: flagged, not written
    check(c)


def test_invalid_sequence_and_trailing_padding():
    c = wl.paged_case(46, num_heads=4, kv_num_heads=2, head_size=64, block_size=16,
                      past=[10, 20, 30], new_tokens=[3, 2, 2])
    c.past_seqlens[1] = -4                      # invalid sequence: zero output, flagged
    check(c)
    c2 = wl.paged_case(46, num_heads=4, kv_num_heads=2, head_size=64, block_size=16,
                       past=[10, 20, 30], new_tokens=[3, 2, 2])
    c2.cu_seqlens[3] = 5                        # last 2 tokens are padding: zero output
    g = run_paged_gpu(c2)
    r = run_paged_oracle(c2)
    assert (g.out[5:] == 0).all() and g.status == r.status == 0
    assert_f16_close(g.out, r.out, "padded batch")


def test_page_permutation_invariance_on_gpu():
    c = wl.paged_case(47, num_heads=8, kv_num_heads=2, head_size=128, block_size=16,
                      past=[300, 17, 0], new_tokens=[1, 40, 9], extra_blocks=5)
    a = run_paged_gpu(c)
    perm = np.random.default_rng(3).permutation(c.num_blocks)
    inv = np.argsort(perm)
    c.key_cache = c.key_cache[perm]
    c.value_cache = c.value_cache[perm]
    bt = c.block_table.copy()
    bt[bt >= 0] = inv[bt[bt >= 0]]
    c.block_table = bt
    b = run_paged_gpu(c)
    np.testing.assert_array_equal(a.out, b.out)


def test_scatter_pass_alone_is_bit_exact():
    c = wl.paged_case(48, num_heads=4, kv_num_heads=2, head_size=128, block_size=32,
                      past=[0, 33, 100], new_tokens=[40, 1, 7], packed=True)
    kc, vc = dev(c.key_cache), dev(c.value_cache)
    B.pkv_paged_scatter_kv(dev(c.query), None, None, kc, vc, dev(c.cu_seqlens),
                           dev(c.past_seqlens), dev(c.block_table), None,
                           num_heads=4, kv_num_heads=2)
    torch.cuda.synchronize()
    k_new, v_new, _ = orc.split_new_kv(c.query, None, None, 4, 2, 128)
    rk, rv, st = orc.paged_scatter(k_new, v_new, c.key_cache, c.value_cache, c.cu_seqlens,
                                   c.past_seqlens, c.block_table)
    np.testing.assert_array_equal(host(kc), rk)
    np.testing.assert_array_equal(host(vc), rv)


def test_rejects_contract_violations_before_launch():
    c = wl.tiny_decode()
    q, k, v = dev(c.query), dev(c.key), dev(c.value)
    kc, vc = dev(c.key_cache), dev(c.value_cache)
    cu, past, bt = dev(c.cu_seqlens), dev(c.past_seqlens), dev(c.block_table)
    with pytest.raises(B.PagedKVError):
        B.pkv_paged_attention(q, k, None, kc, vc, cu, past, bt, num_heads=4, kv_num_heads=2)
    with pytest.raises(B.PagedKVError):
        B.pkv_paged_attention(q, k, v, kc, vc, cu, past, bt, num_heads=4, kv_num_heads=3)
    with pytest.raises(B.PagedKVError):
        B.pkv_paged_attention(q, k, v, kc, vc, cu, past, bt, num_heads=4, kv_num_heads=2,
                              is_causal=0)
    before = B.pkv_launch_count()
    with pytest.raises(B.PagedKVError):
        B.pkv_paged_attention(q, k, v, kc, vc, cu[:1], past, bt, num_heads=4,
                              kv_num_heads=2)
    assert B.pkv_launch_count() == before
