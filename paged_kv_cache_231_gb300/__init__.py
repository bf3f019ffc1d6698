"""GB300 paged / block-sparse grouped-query attention: C-ABI library + thin binding.

The compute lives in ``libpagedkv.so`` (CUDA kernels for sm_103a); this package only
builds it, loads it and marshals torch tensors into its C argument blocks.
"""
from .binding import (  # noqa: F401
    PKV_SPLIT_AUTO, PKV_SPLIT_FIXED, PKV_SPLIT_PAGES, PagedKVError, load_library,
    make_paged_args, make_sparse_args, pkv_combine_partials, pkv_kv_append_rotary,
    pkv_launch_count, pkv_paged_attention, pkv_paged_attention_plan,
    pkv_paged_attention_workspace_size, pkv_paged_contract_check, pkv_paged_scatter_kv,
    pkv_profiler_enable, pkv_profiler_query, pkv_profiler_reset,
    pkv_sparse_attention_partials, pkv_sparse_attention_partials_workspace_size)
