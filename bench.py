#!/usr/bin/env python
"""Benchmark of the paged attention hot path on one GB300 (or N replicas).

Default workload: Llama-3-8B-shaped paged decode (64 sequences, 32 query heads over
8 kv heads, head size 128, 16-token blocks, contexts uniform in [512, 8192]). One step
is one pkv_paged_attention call: scatter of the 64 new tokens' K/V into the paged
cache, device planning, split-KV attention and the LSE combine.

Prints ONE JSON line. ``value`` is KV+Q+O bytes per step / device time per step (GB/s);
``e2e`` repeats the metric through the public Python call with host buffers (H2D of
the step's inputs and D2H of its output inside the timed region). ``--impl reference``
times the CPU oracle on a bounded sample of the same workload instead.

Other workloads (``--workload llama8b_decode_rope|varlen_mixed|block_sparse|
block_sparse_f16|block_sparse_causal|append_prompt|tiny_decode``) print the same structure
with their own metric; they are not the headline line.
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

os.environ.setdefault("OPENBLAS_NUM_THREADS", str(os.cpu_count() or 1))
os.environ.setdefault("OMP_NUM_THREADS", str(os.cpu_count() or 1))

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attention KV GB/s and % of HBM peak; tokens/s at Llama-8B shape"
L2_BYTES = 129 * 1024 * 1024
WORKLOADS = ["llama8b_decode", "llama8b_decode_rope", "varlen_mixed", "block_sparse",
             "block_sparse_f16", "block_sparse_causal", "append_prompt", "tiny_decode"]
# metric, unit and direction of every workload (shared by both arms of the benchmark)
METRICS = {
    "llama8b_decode": (METRIC, "GB/s", True),
    "llama8b_decode_rope": (METRIC + ", RoPE on new keys and queries", "GB/s", True),
    "varlen_mixed": ("varlen prefill+decode attention TFLOP/s (causal pairs)", "TFLOP/s", True),
    "block_sparse": ("block-sparse partials+combine fp32 TFLOP/s", "TFLOP/s", True),
    "block_sparse_f16": ("block-sparse partials+combine fp16 TFLOP/s", "TFLOP/s", True),
    "block_sparse_causal": ("block-sparse partials+combine fp32 TFLOP/s, right-aligned causal",
                            "TFLOP/s", True),
    "append_prompt": ("KV append+RoPE GB/s (prompt)", "GB/s", True),
    "tiny_decode": ("tiny paged decode latency (2 sequences, scatter + attention), "
                    "microseconds per call", "us", False),
}


# ----------------------------------------------------------------------------- infra
def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama8b_decode",
                    choices=WORKLOADS)
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="CPU work budget of the oracle baseline sample")
    ap.add_argument("--e2e-steps", type=int, default=0, help="0 = same as --steps")
    ap.add_argument("--skip-e2e", action="store_true", help="omit the host-buffer leg")
    ap.add_argument("--oracle-one-core", action="store_true", help=argparse.SUPPRESS)
    return ap.parse_args()


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Largest value over all ranks (the job is as slow as its slowest replica)."""
    if world <= 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return (float(d["hbm_gbs"]), float(d["bf16_tflops"]),
                float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured")
    return 6800.0, 1900.0, 1700.0, "fallback"


CLOCK_PAD_S = 0.5


class ClockSampler:
    """nvidia-smi clock / throttle samples every 50 ms while it runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.rows = []
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4)
                          if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.rows)}


def source_sha(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(summary, sources):
    """DRAM bytes per launch from a committed ncu summary, or None if the summary is
    missing or the kernel's sources changed since it was taken."""
    p = os.path.join(ROOT, "profiles", summary)
    if not os.path.exists(p):
        return None
    text = open(p).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    s = re.search(r"source_sha256:\s*([0-9a-f]+)", text)
    if not m or not s or s.group(1) != source_sha(sources):
        return None
    return int(m.group(1))


def to_dev(x):
    return None if x is None else torch.from_numpy(np.ascontiguousarray(x)).cuda()


def timed_loop(fn, steps, world):
    """Time exactly `steps` calls of fn on the current stream with CUDA events, barrier
    and synchronize on both sides; returns ms per step (max over ranks)."""
    stream = torch.cuda.current_stream()
    barrier(world)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    end.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    ms = start.elapsed_time(end) / steps
    return max_over_ranks(ms, world)


# ----------------------------------------------------------------------------- workloads
ATTN_SOURCES = ["paged_kv_cache_231_gb300/csrc/attention.cu",
                "paged_kv_cache_231_gb300/csrc/device_common.cuh",
                "paged_kv_cache_231_gb300/csrc/scatter_dev.cuh",
                "paged_kv_cache_231_gb300/csrc/tcgen05.cuh",
                "paged_kv_cache_231_gb300/csrc/internal.h"]
SPARSE_SOURCES = ["paged_kv_cache_231_gb300/csrc/sparse.cu",
                  "paged_kv_cache_231_gb300/csrc/device_common.cuh",
                  "paged_kv_cache_231_gb300/csrc/tcgen05.cuh",
                  "paged_kv_cache_231_gb300/csrc/internal.h"]
SPARSE16_SOURCES = ["paged_kv_cache_231_gb300/csrc/sparse16.cu",
                    "paged_kv_cache_231_gb300/csrc/device_common.cuh",
                    "paged_kv_cache_231_gb300/csrc/tcgen05.cuh",
                    "paged_kv_cache_231_gb300/csrc/internal.h"]


def decode_bytes(case):
    """KV bytes of every visible key (K and V, fp16) + Q + O: the step's compulsory
    HBM traffic; partials and block-table reads are overhead and not counted."""
    n = case.context_lengths()
    D, Hkv, Hq, T = case.head_size, case.kv_num_heads, case.num_heads, case.num_tokens
    kv = int(n.sum()) * Hkv * D * 2 * 2
    q = T * Hq * D * 2
    return kv, q, q


def prefill_flops(case):
    """4*D per (query head, visible key) pair, causal pairs only."""
    N = np.diff(case.cu_seqlens.astype(np.int64))
    P = case.past_seqlens.astype(np.int64)
    pairs = int((N * P + N * (N + 1) // 2).sum())
    return 4.0 * case.head_size * case.num_heads * pairs


class Workload:
    pass


def paged_config(name, case):
    """The `config` object of a paged workload (both arms print the same one)."""
    pool = case.key_cache.nbytes + case.value_cache.nbytes
    if name == "tiny_decode":
        kvb, qb, ob = decode_bytes(case)
        return {"workload": name, "batch": case.batch, "tokens": case.num_tokens,
                "num_heads": case.num_heads, "kv_num_heads": case.kv_num_heads,
                "head_size": case.head_size, "block_size": case.block_size,
                "past": [int(x) for x in case.past_seqlens], "bytes_per_step": kvb + qb + ob,
                "l2": "no flush: a latency case (%.0f KB of KV pool, L2-resident)" % (pool / 1e3)}
    if name.startswith("llama8b_decode"):
        kvb, qb, ob = decode_bytes(case)
        return {"workload": name, "batch": case.batch, "tokens": case.num_tokens,
                "num_heads": 32, "kv_num_heads": 8, "head_size": 128, "block_size": 16,
                "context": "U[512,8192]",
                "mean_context": float(case.context_lengths().mean()),
                "kv_bytes_per_step": kvb, "bytes_per_step": kvb + qb + ob,
                "l2": "no flush: the KV pool (%.2f GB) is larger than L2 (129 MB)"
                      % (pool / 1e9)}
    return {"workload": "varlen_mixed", "batch": case.batch, "tokens": case.num_tokens,
            "num_heads": 32, "kv_num_heads": 8, "head_size": 128, "block_size": 32,
            "flops_per_step": prefill_flops(case),
            "l2": "no flush: KV pool %.2f GB > L2" % (pool / 1e9)}


def sparse_keys(c, causal):
    """Keys taking part per edge (block_len clipped; at or before the query if causal)."""
    bl = np.clip(c.edge_meta[:, 4], 0, c.block_size).astype(np.int64)
    if causal:
        qpos = c.query_positions()
        lim = (qpos[c.edge_meta[:, 0]].astype(np.int64)
               - c.edge_meta[:, 2].astype(np.int64) * c.block_size + 1)
        bl = np.clip(np.minimum(bl, lim), 0, None)
    return bl


def sparse_config(name, c):
    P = c.num_edges * c.qhead
    flops = 4.0 * c.head_dim * c.qhead * float(sparse_keys(c, name == "block_sparse_causal").sum())
    compulsory = (c.k_pages.nbytes + c.v_pages.nbytes + c.q.nbytes + P * (c.head_dim + 2) * 4)
    return {"workload": name, "queries": int(c.q.shape[0]), "edges": c.num_edges,
            "partials": P, "hq": c.hq, "hkv": c.hkv, "head_dim": c.head_dim,
            "block": c.block_size, "flops_per_step": flops,
            "partials_compulsory_bytes": compulsory,
            "l2": "no flush: K/V pages %.2f GB > L2" % ((c.k_pages.nbytes + c.v_pages.nbytes) / 1e9)}


def append_config(c):
    byts = c.batch * c.seq_len * c.kv_num_heads * c.head_size * 2 * 4 + c.seq_len * c.rotary_dim * 2
    return {"workload": "append_prompt", "batch": 4, "seq_len": 512, "kv_num_heads": 8,
            "head_size": 128, "rotary_dim": 128, "bytes_per_step": byts,
            "l2": "inputs %.1f MB < L2: numbers include L2 hits" % (byts / 1e6)}


def workload_config(name, case):
    if name in ("block_sparse", "block_sparse_f16", "block_sparse_causal"):
        return sparse_config(name, case)
    if name == "append_prompt":
        return append_config(case)
    return paged_config(name, case)


def setup_paged(name, args):
    from paged_kv_cache_231_gb300 import binding as B
    from paged_kv_cache_231_gb300 import workloads as wl
    lib = B.load_library()
    rope = name == "llama8b_decode_rope"
    case = case_for(name)
    # RoPE variant: new keys and every query head rotated at the token's position
    rot = dict(cos_cache=to_dev(case.cos_cache), sin_cache=to_dev(case.sin_cache),
               rotary_dim=case.rotary_dim, rotary_query=True) if rope else {}
    q, k, v = to_dev(case.query), to_dev(case.key), to_dev(case.value)
    kc, vc = to_dev(case.key_cache), to_dev(case.value_cache)
    cu, past, bt = to_dev(case.cu_seqlens), to_dev(case.past_seqlens), to_dev(case.block_table)
    sm = to_dev(case.slot_mapping)
    out = torch.empty((case.num_tokens, case.num_heads * case.head_size),
                      dtype=torch.float16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = B.make_paged_args(q, k, v, kc, vc, cu, past, bt, sm, out,
                          num_heads=case.num_heads, kv_num_heads=case.kv_num_heads,
                          scale=case.scale, device_status=status, **rot)
    nws = B.pkv_paged_attention_workspace_size(a)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    import ctypes
    aref = ctypes.byref(a)

    def step():
        st = lib.pkv_paged_attention(aref, ws.data_ptr(), nws,
                                     torch.cuda.current_stream().cuda_stream)
        if st != 0:
            raise B.PagedKVError("pkv_paged_attention", st)

    # end-to-end: the public call with pinned host inputs, H2D + call + D2H per step. The
    # step's inputs (query, new K/V, lengths, block table, slots) sit in one pinned host
    # buffer, as a serving loop stages a batch, and move in one copy; the call's device
    # tensors are views into one device buffer. The caches stay resident on the device.
    parts = [case.query, case.key, case.value, case.cu_seqlens, case.past_seqlens,
             case.block_table, case.slot_mapping]
    offs, nbytes = [], 0
    for a in parts:
        offs.append(nbytes)
        nbytes += 0 if a is None else (a.nbytes + 255) // 256 * 256
    h_buf = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d_buf = torch.empty(nbytes, dtype=torch.uint8, device="cuda")

    def view(buf, a, off):
        if a is None:
            return None
        src = torch.from_numpy(np.ascontiguousarray(a))
        return buf[off:off + src.numel() * src.element_size()].view(src.dtype).view(src.shape)

    for a, off in zip(parts, offs):
        if a is not None:
            view(h_buf, a, off).copy_(torch.from_numpy(np.ascontiguousarray(a)))
    eq, ek, ev, ecu, epast, ebt, esm = (view(d_buf, a, off) for a, off in zip(parts, offs))
    h_out = torch.empty(out.shape, dtype=torch.float16).pin_memory()
    h2d = nbytes
    d2h = h_out.numel() * h_out.element_size()

    def e2e_step():
        d_buf.copy_(h_buf, non_blocking=True)
        B.pkv_paged_attention(eq, ek, ev, kc, vc, ecu, epast, ebt, esm,
                              num_heads=case.num_heads, kv_num_heads=case.kv_num_heads,
                              scale=case.scale, output=out, workspace=ws, **rot)
        h_out.copy_(out, non_blocking=True)

    w = Workload()
    w.case, w.step, w.e2e_step, w.h2d, w.d2h = case, step, e2e_step, h2d, d2h
    w.status = status
    w.check = lambda: int(status.item())
    w.metric, w.unit, w.higher = METRICS[name]
    w.config = paged_config(name, case)
    if name == "tiny_decode":
        # latency: one call's device time; the whole call is one single-pass launch
        kvb, qb, ob = decode_bytes(case)
        w.work, w.dtype, w.tokens = None, "f16", case.num_tokens
        w.dominant, w.dom_work, w.bound, w.dom_unit = "single_pass", (kvb + qb + ob) / 1e9, \
            "hbm", "GB/s"
        w.traffic_summary, w.traffic_sources = "single_pass_tiny_decode.md", ATTN_SOURCES
    elif name.startswith("llama8b_decode"):
        kvb, qb, ob = decode_bytes(case)
        w.work, w.dtype = (kvb + qb + ob) / 1e9, "f16"
        w.tokens = case.num_tokens
        # the persistent attention kernel reads K/V and Q and writes O (fused combine)
        w.dominant, w.dom_work, w.bound = "attention", (kvb + qb + ob) / 1e9, "hbm"
        w.dom_unit = "GB/s"
        w.traffic_summary, w.traffic_sources = "attention_llama8b_decode.md", ATTN_SOURCES
        if rope:   # the summary's counters were taken on the unrotated workload
            w.traffic_summary = None
    else:
        fl = prefill_flops(case)
        w.work, w.dtype = fl / 1e12, "f16"
        w.tokens = case.num_tokens
        # prefill tiles run in the tensor-core kernel (decode tokens in the attention one)
        w.dominant, w.dom_work, w.bound, w.dom_unit = "prefill_tc", fl / 1e12, "tensor", "TFLOP/s"
        w.traffic_summary, w.traffic_sources = "prefill_tc_varlen_mixed.md", ATTN_SOURCES
    w.launches_per_step = None
    return w


def setup_sparse(args, f16=False, causal=False):
    from paged_kv_cache_231_gb300 import binding as B
    from paged_kv_cache_231_gb300 import workloads as wl
    import ctypes
    lib = B.load_library()
    name = "block_sparse_causal" if causal else ("block_sparse_f16" if f16 else "block_sparse")
    c = case_for(name)
    q, kp, vp = to_dev(c.q), to_dev(c.k_pages), to_dev(c.v_pages)
    em, bt, so = to_dev(c.edge_meta), to_dev(c.block_tables), to_dev(c.seg_offsets)
    # right-aligned causal: keys after the query's position take no part
    qpos = c.query_positions() if causal else None
    P = c.num_edges * c.qhead
    o = torch.empty((P, c.head_dim), dtype=torch.float32, device="cuda")
    m = torch.empty(P, dtype=torch.float32, device="cuda")
    l = torch.empty(P, dtype=torch.float32, device="cuda")
    nseg = c.seg_offsets.shape[0] - 1
    out = torch.empty((nseg * c.qhead, c.head_dim), dtype=torch.float32, device="cuda")
    a = B.make_sparse_args(q, kp, vp, em, bt, o, m, l, qhead=c.qhead, block_size=c.block_size,
                           page_size=c.page_size, pages_per_block=c.pages_per_block,
                           softmax_scale=c.softmax_scale, query_positions=to_dev(qpos))
    nws = B.pkv_sparse_attention_partials_workspace_size(a)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    ca = B.CombineArgs()
    ca.o, ca.m, ca.l, ca.segment_offsets = o.data_ptr(), m.data_ptr(), l.data_ptr(), so.data_ptr()
    ca.out, ca.lse = out.data_ptr(), None
    ca.num_segments, ca.lanes, ca.head_dim, ca.out_dtype = nseg, c.qhead, c.head_dim, B.PKV_F32

    def step():
        s = torch.cuda.current_stream().cuda_stream
        st = lib.pkv_sparse_attention_partials(ctypes.byref(a), ws.data_ptr(), nws, s)
        st = st or lib.pkv_combine_partials(ctypes.byref(ca), s)
        if st != 0:
            raise B.PagedKVError("sparse step", st)

    w = Workload()
    w.config = sparse_config(name, c)
    flops = w.config["flops_per_step"]
    w.case, w.step, w.e2e_step, w.h2d, w.d2h = c, step, None, 0, 0
    w.check = lambda: 0
    w.metric, w.unit, w.higher = METRICS[name]
    w.work, w.dtype, w.tokens = flops / 1e12, "f16" if f16 else "f32", c.q.shape[0]
    # the partials run on the tensor core (fp32 inputs as three fp16 products of scaled
    # (hi, lo) splits, fp16 inputs as one), so their roofline is HBM: K/V pool read once,
    # Q once, partials (fp32) written once
    compulsory = w.config["partials_compulsory_bytes"]
    w.dominant, w.dom_work, w.bound, w.dom_unit = "sparse_partials", compulsory / 1e9, "hbm", "GB/s"
    w.traffic_summary, w.traffic_sources = "sparse_partials_block_sparse.md", SPARSE_SOURCES
    if f16:
        w.traffic_summary, w.traffic_sources = "sparse_tc16_block_sparse_f16.md", SPARSE16_SOURCES
    if causal:   # the committed counters are for the unmasked workload
        w.traffic_summary = None
    return w


def setup_append(args):
    from paged_kv_cache_231_gb300 import binding as B
    from paged_kv_cache_231_gb300 import workloads as wl
    c = case_for("append_prompt")
    src, pk, pv = to_dev(c.source), to_dev(c.present_key), to_dev(c.present_value)
    ts, kt = to_dev(c.total_sequence_length), to_dev(c.key_total_sequence_lengths)
    cos, sin = to_dev(c.cos_cache), to_dev(c.sin_cache)

    import ctypes
    lib = B.load_library()
    a = B.make_append_args(src, None, ts, kt, pk, pv, num_heads=c.num_heads,
                           kv_num_heads=c.kv_num_heads, batch=c.batch, seq_len=c.seq_len,
                           packed=True, cos_cache=cos, sin_cache=sin,
                           rotary_dim=c.rotary_dim, interleaved=False)
    aref = ctypes.byref(a)

    def step():   # the C entry point with a prebuilt argument block, as for attention
        st = lib.pkv_kv_append_rotary(aref, torch.cuda.current_stream().cuda_stream)
        if st != 0:
            raise B.PagedKVError("pkv_kv_append_rotary", st)

    rows = c.batch * c.seq_len * c.kv_num_heads
    byts = rows * c.head_size * 2 * 4 + c.seq_len * c.rotary_dim * 2
    w = Workload()
    w.case, w.step, w.e2e_step, w.h2d, w.d2h = c, step, None, 0, 0
    w.check = lambda: 0
    w.metric, w.unit, w.higher = METRICS["append_prompt"]
    w.work, w.dtype = byts / 1e9, "f16"
    w.tokens = c.batch * c.seq_len
    w.dominant, w.dom_work, w.bound, w.dom_unit = "append", byts / 1e9, "hbm", "GB/s"
    w.traffic_summary, w.traffic_sources = None, []
    w.config = append_config(c)
    return w


# ----------------------------------------------------------------------------- CPU oracle
_CASES = {}


def case_for(name):
    """The seeded input of a workload, drawn once per process (numpy, host memory)."""
    from paged_kv_cache_231_gb300 import workloads as wl
    if name not in _CASES:
        _CASES[name] = {"llama8b_decode": wl.llama8b_decode,
                        "llama8b_decode_rope": lambda: wl.llama8b_decode(rotary=True),
                        "varlen_mixed": wl.varlen_mixed,
                        "block_sparse": wl.block_sparse,
                        "block_sparse_f16": lambda: wl.block_sparse(dtype=np.float16),
                        "block_sparse_causal": wl.block_sparse,
                        "append_prompt": lambda: wl.append_rotary(2, mode="prompt",
                                                                  interleaved=False),
                        "tiny_decode": wl.tiny_decode}[name]()
    return _CASES[name]


def oracle_sample(name, seconds):
    """Time the CPU oracle on whole sequences (edge batches) of the workload until
    `seconds` of wall time are spent. Returns (value in the workload's unit, tokens/s or
    None, description, effective cores = process CPU time / wall time)."""
    from oracle import pagedkv_oracle as orc
    case = case_for(name)
    cpu0, wall0 = time.process_time(), time.perf_counter()

    def busy():   # cores kept busy since the sample began: CPU time / wall time
        return (time.process_time() - cpu0) / max(time.perf_counter() - wall0, 1e-9)
    if name in ("llama8b_decode", "llama8b_decode_rope", "varlen_mixed", "tiny_decode"):
        D, Hkv, Hq = case.head_size, case.kv_num_heads, case.num_heads
        done_work, done_tok, spent, seqs = 0.0, 0, 0.0, 0
        for b in range(case.batch):
            sub = _subcase(case, b)
            t0 = time.perf_counter()
            orc.paged_attention(sub.query, sub.key, sub.value, sub.key_cache, sub.value_cache,
                                sub.cu_seqlens, sub.past_seqlens, sub.block_table,
                                sub.slot_mapping, num_heads=Hq, kv_num_heads=Hkv,
                                scale=sub.scale, cos_cache=sub.cos_cache,
                                sin_cache=sub.sin_cache, rotary_dim=sub.rotary_dim,
                                rotary_query=sub.rotary_dim > 0)
            spent += time.perf_counter() - t0
            seqs += 1
            done_tok += sub.num_tokens
            if name == "varlen_mixed":
                done_work += prefill_flops(sub) / 1e12
            else:
                kvb, qb, ob = decode_bytes(sub)
                done_work += (kvb + qb + ob) / 1e9
            if spent >= seconds and name != "tiny_decode":
                break
        cores = busy()
        if name == "tiny_decode":   # the whole call, every sequence: microseconds
            return spent * 1e6, done_tok / spent, \
                f"the whole call ({seqs} sequences), {spent * 1e3:.2f} ms", cores
        return done_work / spent, done_tok / spent, \
            f"{seqs} of {case.batch} sequences, whole (scatter + attention), {spent:.1f} s", cores
    if name in ("block_sparse", "block_sparse_f16", "block_sparse_causal"):
        c = case
        qpos = c.query_positions() if name == "block_sparse_causal" else None
        keys = sparse_keys(c, qpos is not None)
        rng = np.random.default_rng(0)
        order = rng.permutation(c.num_edges)
        spent, n, fl = 0.0, 0, 0.0
        t0 = time.perf_counter()
        for i in range(0, c.num_edges, 256):
            edges = order[i:i + 256]
            orc.sparse_attention_partials(
                c.q, c.k_pages, c.v_pages, c.edge_meta, c.block_tables, qhead=c.qhead,
                hq=c.hq, head_dim=c.head_dim, block_size=c.block_size, page_size=c.page_size,
                pages_per_block=c.pages_per_block, softmax_scale=c.softmax_scale, edges=edges,
                query_positions=qpos)
            n += len(edges)
            fl += 4.0 * c.head_dim * c.qhead * float(keys[edges].sum())
            spent = time.perf_counter() - t0
            if spent >= seconds:
                break
        cores = busy()
        return fl / 1e12 / spent, None, f"{n} random edges of {c.num_edges}, {spent:.1f} s", \
            cores
    c = case
    t0 = time.perf_counter()
    orc.kv_append_rotary(c.source, c.value, packed=True, num_heads=c.num_heads,
                         kv_num_heads=c.kv_num_heads, head_size=128, batch=c.batch,
                         seq_len=c.seq_len, total_sequence_length=c.total_sequence_length,
                         key_total_sequence_lengths=c.key_total_sequence_lengths,
                         cos_cache=c.cos_cache, sin_cache=c.sin_cache, rotary_dim=128,
                         interleaved=False, present_key=c.present_key,
                         present_value=c.present_value)
    spent = time.perf_counter() - t0
    cores = busy()
    byts = c.batch * c.seq_len * c.kv_num_heads * 128 * 2 * 4 + c.seq_len * 128 * 2
    return byts / 1e9 / spent, None, f"whole prompt append, {spent:.1f} s", cores


def oracle_single_core(name, seconds):
    """The same oracle sample in a child process confined to one CPU with one BLAS
    thread; None if the child fails."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")

    def pin():   # before the child starts: every thread it creates inherits one CPU
        try:
            os.sched_setaffinity(0, {sorted(os.sched_getaffinity(0))[0]})
        except (AttributeError, OSError):
            pass

    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-one-core",
                            "--workload", name, "--cpu-seconds", str(seconds)],
                           env=env, capture_output=True, text=True, timeout=600,
                           preexec_fn=pin)
        line = [x for x in r.stdout.splitlines() if x.startswith("{")]
        return json.loads(line[-1]) if r.returncode == 0 and line else None
    except (OSError, subprocess.SubprocessError, ValueError):
        return None


def one_core_child(args):
    """Entry of the single-CPU child (started pinned to one CPU): run the sample, print
    JSON."""
    v, tps, desc, cores = oracle_sample(args.workload, args.cpu_seconds)
    print(json.dumps({"value": v, "unit": METRICS[args.workload][1], "cores": 1,
                      "cpu_per_wall": cores, "sample": desc, "tokens_per_s": tps}))


def _subcase(case, b):
    """Sequence b of a paged case as a self-contained case with a compact block pool."""
    from paged_kv_cache_231_gb300 import workloads as wl
    lo, hi = int(case.cu_seqlens[b]), int(case.cu_seqlens[b + 1])
    row = case.block_table[b]
    used = row[row >= 0]
    bt = np.full((1, case.max_blocks), -1, dtype=np.int32)
    bt[0, :used.size] = np.arange(used.size, dtype=np.int32)
    return wl.PagedCase(
        num_heads=case.num_heads, kv_num_heads=case.kv_num_heads, head_size=case.head_size,
        block_size=case.block_size, query=case.query[lo:hi],
        key=None if case.key is None else case.key[lo:hi],
        value=None if case.value is None else case.value[lo:hi],
        key_cache=case.key_cache[used], value_cache=case.value_cache[used],
        cu_seqlens=np.array([0, hi - lo], dtype=np.int32),
        past_seqlens=case.past_seqlens[b:b + 1], block_table=bt,
        slot_mapping=None, scale=case.scale, cos_cache=case.cos_cache,
        sin_cache=case.sin_cache, rotary_dim=case.rotary_dim,
        rotary_interleaved=case.rotary_interleaved)


def cpus_available():
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def cpu_baseline(name, seconds, value=None, desc=None, cores=None, tps=None):
    """cpu_baseline object: the oracle on all host cores (cores = CPU time / wall time of
    the sample, i.e. the cores it kept busy) plus the same sample on one core."""
    if value is None:
        value, tps, desc, cores = oracle_sample(name, seconds)
    out = {"value": value, "unit": METRICS[name][1], "cores": round(cores, 2),
           "cpus_available": cpus_available(), "kind": "oracle", "sample": desc}
    if tps is not None:
        out["tokens_per_s"] = tps
    one = oracle_single_core(name, seconds)
    if one is not None:
        out["single_core"] = one
    return out


# ----------------------------------------------------------------------------- main
def run_reference(args, world, rank):
    if rank != 0:
        return
    metric, unit, higher = METRICS[args.workload]
    # each step is a bounded sample (at least one whole sequence / edge batch); the
    # whole run is kept to about two minutes of CPU work
    per = min(args.cpu_seconds, 120.0 / max(1, args.steps + args.warmup))
    vals, descs, toks, walls, cores = [], [], [], [], []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        v, tps, desc, cr = oracle_sample(args.workload, per)
        if i >= args.warmup:
            walls.append(time.perf_counter() - t0)
            vals.append(v)
            descs.append(desc)
            toks.append(tps)
            cores.append(cr)
    value = statistics.median(vals)
    line = {"impl": "reference", "metric": metric, "value": value, "unit": unit,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * statistics.median(walls), "higher_is_better": higher,
            "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded numpy draws, N(0,1))",
            "config": dict(workload_config(args.workload, case_for(args.workload)),
                           parallelism=f"replicas{world}"),
            "cpu_baseline": {"value": value, "unit": unit,
                             "cores": round(statistics.median(cores), 2),
                             "cpus_available": cpus_available(), "kind": "oracle",
                             "sample": descs[-1]},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    if toks[-1] is not None:
        line["tokens_per_s"] = statistics.median(toks)
    print(json.dumps(line), flush=True)


def run_for(fn, seconds):
    """Untimed steps for about `seconds` of wall time (synchronised every 8 steps)."""
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        for _ in range(8):
            fn()
        torch.cuda.synchronize()


def main():
    args = parse_args()
    if args.oracle_one_core:
        one_core_child(args)
        return
    world, rank, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    from paged_kv_cache_231_gb300 import binding as B
    import __graft_entry__
    if rank == 0 or world == 1:
        __graft_entry__.build()
    barrier(world)
    B.load_library()
    setup = {"llama8b_decode": lambda: setup_paged("llama8b_decode", args),
             "llama8b_decode_rope": lambda: setup_paged("llama8b_decode_rope", args),
             "varlen_mixed": lambda: setup_paged("varlen_mixed", args),
             "block_sparse": lambda: setup_sparse(args),
             "block_sparse_f16": lambda: setup_sparse(args, f16=True),
             "block_sparse_causal": lambda: setup_sparse(args, causal=True),
             "append_prompt": lambda: setup_append(args),
             "tiny_decode": lambda: setup_paged("tiny_decode", args)}[args.workload]
    w = setup()
    hbm, bf16, bf16_sus, peak_kind = measured_peaks()

    for _ in range(max(3, args.warmup)):
        w.step()
    torch.cuda.synchronize()
    assert w.check() == 0, "device status flagged invalid data"

    # timed region: K steps exactly as a caller runs them (no extra events). The clock
    # sampler runs over a window of the same steps around it (half a second before and
    # after), because a timed region of a few milliseconds is shorter than the sampling
    # period of nvidia-smi
    clocks = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    t_win = time.perf_counter()
    run_for(w.step, CLOCK_PAD_S)
    launches0 = B.pkv_launch_count()
    ms = timed_loop(w.step, args.steps, world)
    launches = B.pkv_launch_count() - launches0
    run_for(w.step, CLOCK_PAD_S)
    clk = clocks.stop() if clocks else None
    if clk is not None:
        clk["window_s"] = round(time.perf_counter() - t_win, 3)
        clk["window"] = "the same steps, run continuously before, during and after the timed region"
    # second timed pass of the same K steps with a CUDA event pair around every kernel
    # on its launching stream: per-kernel device time for the roofline (events between
    # kernels stop the prefill kernel's early start, so this pass is not the value)
    B.pkv_profiler_reset()
    B.pkv_profiler_enable(True)
    prof_ms = timed_loop(w.step, args.steps, world)
    B.pkv_profiler_enable(False)
    dom_ms, dom_n = B.pkv_profiler_query(w.dominant)
    kernel_ms = {k: B.pkv_profiler_query(k) for k in
                 ("prologue", "attention", "prefill_tc", "decode_split", "combine",
                  "single_pass", "scatter", "sparse_group", "sparse_qsplit", "sparse_partials",
                  "append")}
    B.pkv_profiler_reset()

    e2e = None
    if w.e2e_step is not None and not args.skip_e2e:
        for _ in range(3):
            w.e2e_step()
        e2e_ms = timed_loop(w.e2e_step, args.e2e_steps or args.steps, world)
        e2e_v = e2e_ms * 1e3 if w.work is None else world * w.work / (e2e_ms / 1e3)
        e2e = {"value": e2e_v, "unit": w.unit,
               "h2d_bytes_per_step": w.h2d, "d2h_bytes_per_step": w.d2h,
               "ms_per_step": e2e_ms}

    # w.work None: a latency workload, value = microseconds per call (max over ranks)
    value = ms * 1e3 if w.work is None else world * w.work / (ms / 1e3)
    dom_avg_ms = dom_ms / max(1, dom_n)
    achieved = w.dom_work / (dom_avg_ms / 1e3) if dom_n else None
    if w.bound == "hbm":
        peak, punit = hbm, "GB/s"
    elif w.bound == "tensor":
        # the prefill kernel is timed alone in sub-millisecond steps: the burst rate
        peak, punit = bf16, "TFLOP/s"
        peak_kind += " dense bf16 burst rate (fp16 has the same dense rate)"
    else:
        sm_mhz = 2070.0
        peak, punit = 152 * 128 * 2 * sm_mhz * 1e6 / 1e12, "TFLOP/s"
        peak_kind = "derived: 152 SMs x 128 fp32 FMA lanes x 2 x 2070 MHz"
    traffic = profiled_traffic(w.traffic_summary, w.traffic_sources) if w.traffic_summary else None

    if rank != 0:
        return
    line = {"metric": w.metric, "value": value, "unit": w.unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": w.higher, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic (seeded numpy draws, N(0,1))",
            "config": dict(w.config, parallelism=f"replicas{world}"),
            "tokens_per_s": world * w.tokens / (ms / 1e3)}
    if w.bound == "hbm" and w.unit == "GB/s":
        line["pct_hbm_peak"] = 100.0 * value / world / hbm
    line["roofline"] = {"bound": w.bound, "kernel": w.dominant, "achieved": achieved,
                        "peak": peak, "unit": punit,
                        "frac": (achieved / peak) if achieved else None,
                        "traffic": traffic, "peak_source": peak_kind,
                        "kernel_ms_avg": dom_avg_ms, "kernel_launches": dom_n}
    line["kernels_ms_per_step"] = {k: v[0] / args.steps for k, v in kernel_ms.items() if v[1]}
    line["profiled_ms_per_step"] = prof_ms
    line["gpu_launches"] = launches
    line["clocks"] = clk
    line["e2e"] = e2e
    if world == 1 and args.cpu_seconds > 0:
        line["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_seconds)
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
