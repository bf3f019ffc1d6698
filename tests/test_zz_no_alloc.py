"""The allocation-free paged attention call (pkv_paged_attention_static_workspace).

Some callers may not allocate device memory (an engine plugin whose enqueue step
must not allocate, a framework that owns all device memory through its own pool);
this call takes its scratch from a fixed array inside the library instead of a
workspace argument. The test runs it twice in a row through the C ABI, with a call on
a different shape in between (so the second call finds leftovers that do not match its
own layout in the shared array), and compares each result bit for bit with the
regular call's output: both run the same deterministic kernels on the same GPU. It
then checks that a problem needing more scratch than the array holds is refused.
"""
import ctypes

import numpy as np
import pytest
import torch

from paged_kv_cache_231_gb300 import binding as B
from paged_kv_cache_231_gb300 import workloads as wl

from .gpu_util import DEV, dev, host

pytestmark = pytest.mark.gpu


def _inputs(case):
    return dict(query=dev(case.query), key=dev(case.key), value=dev(case.value),
                key_cache=dev(case.key_cache), value_cache=dev(case.value_cache),
                cumulative_sequence_length=dev(case.cu_seqlens),
                past_seqlens=dev(case.past_seqlens), block_table=dev(case.block_table),
                slot_mapping=dev(case.slot_mapping))


def _static_call(t, case, out):
    """Through the C ABI: fill the argument block and call the entry point."""
    lib = B.load_library()
    fn = lib.pkv_paged_attention_static_workspace
    fn.restype = ctypes.c_int32
    fn.argtypes = [ctypes.POINTER(B.PagedAttentionArgs), ctypes.c_void_p]
    a = B.make_paged_args(t["query"], t["key"], t["value"], t["key_cache"],
                          t["value_cache"], t["cumulative_sequence_length"],
                          t["past_seqlens"], t["block_table"], t["slot_mapping"], out,
                          num_heads=case.num_heads, kv_num_heads=case.kv_num_heads,
                          scale=case.scale)
    return fn(ctypes.byref(a), torch.cuda.current_stream().cuda_stream)


def _case(which):
    if which == "tiny_decode":
        return wl.tiny_decode()
    if which == "mixed":
        return wl.paged_case(61, num_heads=8, kv_num_heads=2, head_size=128, block_size=16,
                             past=[0, 300, 1500, 17], new_tokens=[1, 40, 1, 3],
                             use_slot_mapping=True)
    if which == "other_shape":
        return wl.paged_case(62, num_heads=16, kv_num_heads=2, head_size=64, block_size=32,
                             past=[700, 5, 2000], new_tokens=[2, 70, 1], packed=True)
    return wl.llama8b_decode()


def _regular(case):
    """Output and caches of the regular call (caller-provided workspace)."""
    t = _inputs(case)
    out = B.pkv_paged_attention(**t, num_heads=case.num_heads,
                                kv_num_heads=case.kv_num_heads, scale=case.scale)
    torch.cuda.synchronize()
    return host(out), host(t["key_cache"]), host(t["value_cache"])


def _static_matches(case, ref, what):
    t = _inputs(case)
    out = torch.full((case.num_tokens, case.num_heads * case.head_size), float("nan"),
                     dtype=torch.float16, device=DEV)
    assert _static_call(t, case, out) == B.PKV_OK
    torch.cuda.synchronize()
    got = host(out)
    diff = got.view(np.uint16) != ref[0].view(np.uint16)
    assert not diff.any(), (f"{what}: {int(diff.sum())} elements differ from the regular "
                            f"call; max |diff| "
                            f"{np.abs(got.astype(np.float64) - ref[0]).max():.3e}")
    np.testing.assert_array_equal(host(t["key_cache"]), ref[1])
    np.testing.assert_array_equal(host(t["value_cache"]), ref[2])


@pytest.mark.parametrize("which", ["tiny_decode", "mixed", "llama8b_decode"])
def test_static_workspace_matches_regular_call_twice(which):
    case, other = _case(which), _case("other_shape")
    ref, ref_other = _regular(case), _regular(other)
    _static_matches(case, ref, f"{which}: first static call")
    # a call of another shape in between leaves counters, piece tickets and partials laid
    # out for a different problem in the shared array
    _static_matches(other, ref_other, "other shape in between")
    _static_matches(case, ref, f"{which}: second static call")


def test_static_workspace_refuses_oversized_problem():
    # 2048 decoding sequences x 32 heads x 16 splits of fp32 partials need far more
    # scratch than the fixed array holds: refused before anything is enqueued
    B_, Hq, Hkv, D = 2048, 32, 8, 128
    f16 = dict(dtype=torch.float16, device=DEV)
    q = torch.zeros((B_, Hq * D), **f16)
    k = torch.zeros((B_, Hkv * D), **f16)
    kc = torch.zeros((8, 16, Hkv, D), **f16)
    cu = torch.arange(B_ + 1, dtype=torch.int32, device=DEV)
    past = torch.zeros(B_, dtype=torch.int32, device=DEV)
    bt = torch.zeros((B_, 512), dtype=torch.int32, device=DEV)
    out = torch.zeros((B_, Hq * D), **f16)
    a = B.make_paged_args(q, k, k, kc, kc, cu, past, bt, None, out, num_heads=Hq,
                          kv_num_heads=Hkv)
    assert B.pkv_paged_attention_workspace_size(a) > (32 << 20)
    before = B.pkv_launch_count()
    lib = B.load_library()
    fn = lib.pkv_paged_attention_static_workspace
    fn.restype = ctypes.c_int32
    fn.argtypes = [ctypes.POINTER(B.PagedAttentionArgs), ctypes.c_void_p]
    assert fn(ctypes.byref(a), torch.cuda.current_stream().cuda_stream) == 7
    assert B.pkv_launch_count() == before
