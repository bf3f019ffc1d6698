"""Helpers for the GPU parity tests: move seeded inputs to the device, run the CUDA
library through its C ABI, run the oracle on the same inputs, compare."""
import numpy as np
import torch

from oracle import pagedkv_oracle as orc
from paged_kv_cache_231_gb300 import binding as B

DEV = "cuda:0"

# fp16 outputs and rotated keys: |err| <= 5e-3 + 5e-3 |ref|
F16_ATOL, F16_RTOL = 5e-3, 5e-3
# fp32 block-sparse path: 1e-4 relative to the element, with a floor of 1e-4 times the
# largest magnitude in the same output row (fp32 sums of many terms carry absolute
# error proportional to the row's scale, not to each element)
F32_RTOL = 1e-4


def dev(x):
    return None if x is None else torch.from_numpy(np.ascontiguousarray(x)).to(DEV)


def host(t):
    return t.detach().cpu().numpy()


def assert_f16_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    tol = F16_ATOL + F16_RTOL * np.abs(ref)
    bad = ~(err <= tol)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} elements out of tolerance; max err "
                             f"{err.max():.3e}; first {idx.tolist()} got "
                             f"{got[tuple(idx[0])]} ref {ref[tuple(idx[0])]}")
    return float(err.max()) if err.size else 0.0


def assert_f32_close(got, ref, what="", scalars=False, rtol=None):
    """Rows are the last axis (a 1-D array is one row) unless ``scalars`` is set, in
    which case every element is its own row: then the floor is rtol * max(|ref|, 1),
    the scale of a softmax statistic such as m. rtol defaults to 1e-4 (fp32 inputs)."""
    rtol = F32_RTOL if rtol is None else rtol
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if scalars:
        row_scale = np.maximum(np.abs(ref), 1.0)
    else:
        row_scale = np.max(np.abs(ref), axis=-1, keepdims=True)
    err = np.abs(got - ref)
    tol = rtol * (np.abs(ref) + row_scale) + 1e-30
    bad = ~(err <= tol)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} elements out of tolerance; first "
                             f"{idx.tolist()} got {got[tuple(idx[0])]} ref {ref[tuple(idx[0])]}")
    return float((err / (np.abs(ref) + row_scale + 1e-30)).max()) if err.size else 0.0


def f32_margins(got, ref, what=""):
    """Achieved fp32 error, reported beside the row-scale tolerance: the largest
    element-relative error over elements of at least 1 % of their row's largest
    magnitude, and the largest row-norm relative error ||got - ref|| / ||ref|| (rows are
    the last axis; all-zero reference rows are skipped). Prints both; returns the
    row-norm error."""
    got = np.atleast_2d(np.asarray(got, dtype=np.float64))
    ref = np.atleast_2d(np.asarray(ref, dtype=np.float64))
    rmax = np.max(np.abs(ref), axis=-1, keepdims=True)
    big = (np.abs(ref) >= 0.01 * rmax) & (rmax > 0)
    elem = float((np.abs(got - ref)[big] / np.abs(ref)[big]).max()) if big.any() else 0.0
    norm = np.linalg.norm(ref, axis=-1)
    live = norm > 0
    row = float((np.linalg.norm(got - ref, axis=-1)[live] / norm[live]).max()) \
        if live.any() else 0.0
    print(f"fp32 margin {what}: element-relative (|ref| >= 1% of row max) {elem:.3e}, "
          f"row-norm relative {row:.3e}")
    return row


class PagedRun:
    def __init__(self, out, kc, vc, status):
        self.out, self.kc, self.vc, self.status = out, kc, vc, status


def run_paged_gpu(case, **kw) -> PagedRun:
    kc, vc = dev(case.key_cache), dev(case.value_cache)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = B.pkv_paged_attention(
        dev(case.query), dev(case.key), dev(case.value), kc, vc, dev(case.cu_seqlens),
        dev(case.past_seqlens), dev(case.block_table), dev(case.slot_mapping),
        num_heads=case.num_heads, kv_num_heads=case.kv_num_heads, scale=case.scale,
        device_status=status, cos_cache=dev(case.cos_cache), sin_cache=dev(case.sin_cache),
        rotary_dim=case.rotary_dim, rotary_interleaved=case.rotary_interleaved, **kw)
    torch.cuda.synchronize()
    return PagedRun(host(out), host(kc), host(vc), int(status.item()))


def run_paged_oracle(case, tokens=None, rotary_query=False) -> PagedRun:
    out, kc, vc, st = orc.paged_attention(
        case.query, case.key, case.value, case.key_cache, case.value_cache,
        case.cu_seqlens, case.past_seqlens, case.block_table, case.slot_mapping,
        num_heads=case.num_heads, kv_num_heads=case.kv_num_heads, scale=case.scale,
        cos_cache=case.cos_cache, sin_cache=case.sin_cache, rotary_dim=case.rotary_dim,
        rotary_interleaved=case.rotary_interleaved, tokens=tokens,
        rotary_query=rotary_query)
    return PagedRun(out, kc, vc, st)


def compare_caches(gpu: PagedRun, ref: PagedRun, rotated: bool, what=""):
    """Scatter without rotation is a bit copy; rotated keys are rounded once to fp16 on
    both sides from fp32 (GPU) / fp64 (oracle) math, so they may differ by an ulp."""
    np.testing.assert_array_equal(gpu.vc, ref.vc, err_msg=f"{what}: value cache")
    if rotated:
        diff = gpu.kc != ref.kc
        if diff.any():
            assert_f16_close(gpu.kc[diff], ref.kc[diff], f"{what}: rotated keys")
    else:
        np.testing.assert_array_equal(gpu.kc, ref.kc, err_msg=f"{what}: key cache")
