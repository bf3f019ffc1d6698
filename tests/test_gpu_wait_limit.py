"""The give-up path of the bounded waits in the tensor-core kernels, run on the GPU.

Every wait on an mbarrier in the tcgen05 prefill and in the two block-sparse partial
kernels is bounded; when one gives up, the CTA raises a shared abort flag, every role
unwinds, what the CTA issued is waited for (bounded), its tensor memory is freed and
PKV_DEV_TIMEOUT is reported. Here the testing hook lowers the bound to a few thousand
polls and makes every CTA withhold its first bulk copy, so that a wait runs out with
nothing of that copy in flight. Each test checks that the call returns cleanly with the
timeout bit set, then that a normal call in the same process matches the oracle (the
context and the kernels are still usable).
"""
import numpy as np
import pytest
import torch

from oracle import pagedkv_oracle as orc
from paged_kv_cache_231_gb300 import binding as B
from paged_kv_cache_231_gb300 import workloads as wl

from .gpu_util import (DEV, assert_f16_close, assert_f32_close, compare_caches, dev, host,
                       run_paged_gpu, run_paged_oracle)

pytestmark = pytest.mark.gpu

TIMEOUT = 32
POLLS = 4096


@pytest.fixture
def withheld_copy():
    B.pkv_testing_wait_limit(POLLS, True)
    try:
        yield
    finally:
        B.pkv_testing_wait_limit()


def _prefill_case():
    # head size 128, blocks of 16: the prefill tiles run on the tensor core
    return wl.paged_case(71, num_heads=8, kv_num_heads=2, head_size=128, block_size=16,
                         past=[0, 100, 37], new_tokens=[200, 1, 150])


def test_prefill_wait_gives_up_cleanly(withheld_copy):
    g = run_paged_gpu(_prefill_case())
    assert g.status & TIMEOUT, g.status
    assert g.status & ~TIMEOUT == 0, g.status


def test_prefill_after_a_timeout_matches_the_oracle():
    B.pkv_testing_wait_limit(POLLS, True)
    try:
        g = run_paged_gpu(_prefill_case())
    finally:
        B.pkv_testing_wait_limit()
    assert g.status & TIMEOUT
    c = _prefill_case()
    g = run_paged_gpu(c)
    r = run_paged_oracle(c)
    assert g.status == r.status == 0
    assert_f16_close(g.out, r.out, "prefill after a timeout")
    compare_caches(g, r, False, "caches")


def _sparse(c):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, m, l = B.pkv_sparse_attention_partials(
        dev(c.q), dev(c.k_pages), dev(c.v_pages), dev(c.edge_meta), dev(c.block_tables),
        qhead=c.qhead, block_size=c.block_size, page_size=c.page_size,
        pages_per_block=c.pages_per_block, softmax_scale=c.softmax_scale,
        device_status=status)
    torch.cuda.synchronize()
    return host(o), host(m), host(l), int(status.item())


@pytest.mark.parametrize("dtype", [np.float32, np.float16], ids=["f32", "f16"])
def test_sparse_wait_gives_up_then_recovers(dtype):
    c = wl.block_sparse(72, n_seqs=2, kv_len=512, queries_per_seq=32, hq=16, hkv=4,
                        head_dim=128, pages_per_block=4, blocks_per_query=4, dtype=dtype)
    B.pkv_testing_wait_limit(POLLS, True)
    try:
        *_, st = _sparse(c)
    finally:
        B.pkv_testing_wait_limit()
    assert st & TIMEOUT, st
    go, gm, gl, st = _sparse(c)
    assert st == 0
    ro, rm, rl, rst = orc.sparse_attention_partials(
        c.q, c.k_pages, c.v_pages, c.edge_meta, c.block_tables, qhead=c.qhead, hq=c.hq,
        head_dim=c.head_dim, block_size=c.block_size, page_size=c.page_size,
        pages_per_block=c.pages_per_block, softmax_scale=c.softmax_scale)
    assert rst == 0
    live = rl > 0
    rt = 5e-3 if dtype == np.float16 else None
    assert_f32_close(go[live], ro[live], "o after a timeout", rtol=rt)
    assert_f32_close(gl[live], rl[live], "l after a timeout", scalars=True, rtol=rt)
    assert_f32_close(gm[live], rm[live], "m after a timeout", scalars=True)


def test_hook_rejects_withholding_without_a_bound():
    with pytest.raises(B.PagedKVError):
        B.pkv_testing_wait_limit(0, True)
