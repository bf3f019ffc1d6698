"""GPU parity of pkv_kv_append_rotary (KV append + RoPE into a BNSH cache)."""
import numpy as np
import pytest
import torch

from oracle import pagedkv_oracle as orc
from paged_kv_cache_231_gb300 import binding as B
from paged_kv_cache_231_gb300 import workloads as wl

from .gpu_util import DEV, assert_f16_close, dev, host

pytestmark = pytest.mark.gpu


def run(c, query=None, query_out=None):
    pk, pv = dev(c.present_key), dev(c.present_value)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.pkv_kv_append_rotary(dev(c.source), dev(c.value), dev(c.total_sequence_length),
                           dev(c.key_total_sequence_lengths), pk, pv,
                           num_heads=c.num_heads, kv_num_heads=c.kv_num_heads,
                           batch=c.batch, seq_len=c.seq_len, packed=c.packed,
                           cos_cache=dev(c.cos_cache) if c.rotary_dim else None,
                           sin_cache=dev(c.sin_cache) if c.rotary_dim else None,
                           rotary_dim=c.rotary_dim, interleaved=c.interleaved,
                           device_status=status, query=query, query_out=query_out)
    torch.cuda.synchronize()
    return host(pk), host(pv), int(status.item())


def check_query(c, query=None):
    """With query_out: the rotated query heads against the oracle (unrotated components
    bit-exact), and the cache writes unchanged by the extra output."""
    q_out = torch.full((c.batch * c.seq_len, c.num_heads * c.present_key.shape[3]),
                       float("nan"), dtype=torch.float16, device=DEV)
    gk, gv, gst = run(c, dev(query), q_out)
    ref = orc.append_query_rotary(
        c.source, query, packed=c.packed, num_heads=c.num_heads,
        kv_num_heads=c.kv_num_heads, head_size=c.present_key.shape[3], batch=c.batch,
        seq_len=c.seq_len, total_sequence_length=c.total_sequence_length,
        key_total_sequence_lengths=c.key_total_sequence_lengths, cos_cache=c.cos_cache,
        sin_cache=c.sin_cache, rotary_dim=c.rotary_dim, interleaved=c.interleaved)
    D, R = c.present_key.shape[3], c.rotary_dim
    g = host(q_out).reshape(-1, c.num_heads, D)
    r = ref.reshape(-1, c.num_heads, D)
    np.testing.assert_array_equal(g[:, :, R:], r[:, :, R:].astype(np.float16))
    if R:
        assert_f16_close(g[:, :, :R].astype(np.float64), r[:, :, :R], "rotated queries")
    hk, hv, hst = run(c)
    np.testing.assert_array_equal(gk, hk)
    np.testing.assert_array_equal(gv, hv)
    assert gst == hst


def check(c):
    gk, gv, gst = run(c)
    rk, rv, written, rst = orc.kv_append_rotary(
        c.source, c.value, packed=c.packed, num_heads=c.num_heads,
        kv_num_heads=c.kv_num_heads, head_size=c.present_key.shape[3], batch=c.batch,
        seq_len=c.seq_len, total_sequence_length=c.total_sequence_length,
        key_total_sequence_lengths=c.key_total_sequence_lengths, cos_cache=c.cos_cache,
        sin_cache=c.sin_cache, rotary_dim=c.rotary_dim, interleaved=c.interleaved,
        present_key=c.present_key, present_value=c.present_value)
    assert gst == rst
    # untouched rows and V rows: bit-exact
    np.testing.assert_array_equal(gk[~written], c.present_key[~written])
    np.testing.assert_array_equal(gv, rv.astype(np.float16))
    R = c.rotary_dim
    # components at or past rotary_dim: plain copies
    np.testing.assert_array_equal(gk[written][:, R:], rk[written][:, R:].astype(np.float16))
    if R:
        assert_f16_close(gk[written][:, :R].astype(np.float64), rk[written][:, :R],
                         "rotated keys")
    return written


@pytest.mark.parametrize("mode", ["decode", "prompt"])
@pytest.mark.parametrize("interleaved", [False, True])
def test_append_rotary_workload(mode, interleaved):
    c = wl.append_rotary(2, mode=mode, interleaved=interleaved)
    written = check(c)
    if mode == "prompt":
        assert written[:, :, :512].all() and not written[:, :, 512:].any()


def test_separate_kv_partial_rotary():
    c = wl.append_rotary(3, mode="decode", interleaved=False, batch=3, num_heads=8,
                         kv_num_heads=2, head_size=128, rotary_dim=64, max_cache_seq=512,
                         max_past=400, packed=False)
    check(c)


def test_no_rotary_is_a_bit_copy():
    c = wl.append_rotary(4, mode="prompt", batch=2, num_heads=4, kv_num_heads=2,
                         head_size=64, rotary_dim=0, max_cache_seq=256, prompt_len=37)
    check(c)


def test_position_past_cache_is_skipped_and_flagged():
    c = wl.append_rotary(5, mode="decode", batch=3, num_heads=4, kv_num_heads=2,
                         head_size=64, rotary_dim=64, max_cache_seq=64, max_past=40)
    c.key_total_sequence_lengths[1] = 200      # history 199 >= max_cache_seq
    check(c)


@pytest.mark.parametrize("mode", ["decode", "prompt"])
@pytest.mark.parametrize("interleaved", [False, True])
def test_query_rotation_packed(mode, interleaved):
    c = wl.append_rotary(6, mode=mode, interleaved=interleaved, batch=2, prompt_len=64)
    check_query(c)


# rotary_dim 12: rotation pairs cross 8-element chunks (per-chunk path)
@pytest.mark.parametrize("rotary_dim,interleaved", [(64, False), (12, True), (0, False)])
def test_query_rotation_separate(rotary_dim, interleaved):
    c = wl.append_rotary(7, mode="decode", interleaved=interleaved, batch=3, num_heads=8,
                         kv_num_heads=2, head_size=128, rotary_dim=rotary_dim,
                         max_cache_seq=512, max_past=400, packed=False)
    query = wl.normal_f16(wl.rng_for(8), (3, 8 * 128))
    check_query(c, query)


def test_query_rotation_past_cache_and_table():
    c = wl.append_rotary(9, mode="decode", batch=3, num_heads=4, kv_num_heads=2,
                         head_size=64, rotary_dim=64, max_cache_seq=64, max_past=40)
    c.key_total_sequence_lengths[1] = 200      # history 199: past the cache and the table
    check_query(c)
