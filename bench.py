#!/usr/bin/env python
"""Decode-step benchmark of the paged, quantized KV store on GB300.

One step = the whole hot path over one batch: block tables from the
ReqToTokenPool rows, the quantizing store of each request's new token, and
paged split-K decode attention (plus its combine), all through the C ABI.

Default workload: INT8 KV (per-token, per-head asymmetric), MHA 32 q / 32 kv
heads, head_dim 128, block size 16, 128 requests at context 4096, K/V drawn
from N(0,1) with 1% of the channels scaled by 8. The pool (4.4 GB) is larger
than L2, so no flush is needed between steps.

Prints one JSON line (rank 0). `--impl reference` times the CPU oracle
instead (the reference arm of this build: there is no reference code to
install), on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import re
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synthetic  # noqa: E402

METRIC = "decode attn tokens/s and HBM GB/s (% of GB300 peak) over paged INT8/INT4 KV"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="cfg3",
                   choices=["cfg1", "cfg2", "cfg3", "cfg4", "cfg5", "cfg4_long_prefix"])
    p.add_argument("--batch", type=int, default=0, help="override the workload's batch (profiling)")
    p.add_argument("--num-splits", type=int, default=0)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-graph", action="store_true", help="launch the step's kernels one by one")
    p.add_argument("--no-extras", action="store_true",
                   help="skip the block copy / swap and extend measurements")
    p.add_argument("--extend-only", action="store_true",
                   help="only the extend (prefill) attention measurement (profiling)")
    p.add_argument("--shared-prefix", choices=["auto", "on", "off"], default="off",
                   help="decode shared prefixes once per group (auto: when the workload has one)")
    p.add_argument("--fused-step", action="store_true",
                   help="time the step as the one cooperative launch of kvq_decode_step")
    p.add_argument("--json-out", default="")
    return p.parse_args()


def make_workload(name: str, batch: int, rank: int):
    kw = {}
    if batch:
        kw["batch"] = batch
    wl = synthetic.by_name(name, **kw)
    if rank:  # each rank serves its own requests: a different seed
        kw["seed"] = wl.seed + 1000 * rank
        wl = synthetic.by_name(name, **kw)
    return wl


def workload_desc(wl) -> dict:
    return {
        "workload": f"{wl.name}: {wl.description}",
        "kv_dtype": wl.kv_dtype, "q_dtype": wl.q_dtype, "batch": wl.batch,
        "q_heads": wl.q_heads, "kv_heads": wl.kv_heads, "head_dim": wl.head_dim,
        "block_size": wl.block_size, "max_context": wl.max_seq_len,
        "mean_context": float(np.mean(wl.seq_lens)),
        "prefill_chunk_tokens": 0 if wl.chunk_slots is None else len(wl.chunk_slots),
    }


def decode_logical_bytes(wl) -> int:
    """KV codes + scale/zero of every context token of every request (a block
    shared by n requests counted n times), Q, the output, the block tables
    and the lengths."""
    kv = int(np.sum(wl.seq_lens, dtype=np.int64)) * wl.kv_token_bytes()
    q = wl.batch * wl.q_heads * wl.head_dim * 2
    nblk = int(np.sum((wl.seq_lens + 15) // 16))
    return kv + 2 * q + 4 * nblk + 4 * wl.batch


def decode_algorithmic_bytes(wl) -> int:
    """Bytes the decode call must move at the least: as above, but every stored
    token once however many requests attend it (shared prefixes). Equal to
    the logical bytes when no block is shared."""
    seen = set()
    kv = 0
    for b in range(wl.batch):
        L = int(wl.seq_lens[b])
        for j in range((L + 15) // 16):
            blk = int(wl.block_tables[b, j])
            if blk in seen:
                continue
            seen.add(blk)
            kv += min(16, L - 16 * j) * wl.kv_token_bytes()
    q = wl.batch * wl.q_heads * wl.head_dim * 2
    nblk = int(np.sum((wl.seq_lens + 15) // 16))
    return kv + 2 * q + 4 * nblk + 4 * wl.batch


def prefix_groups(wl):
    """The requests holding the workload's whole common prefix, as one group
    (what a radix prefix cache knows when it schedules the batch); None when
    the workload shares nothing."""
    if wl.prefix_blocks is None or wl.shared_tokens is None:
        return None
    full = len(wl.prefix_blocks)
    members = [b for b in range(wl.batch) if int(wl.shared_tokens[b]) == 16 * full]
    if len(members) < 2:
        return None
    return members, full


# ---- clocks (NVML through ctypes, read-only) -----------------------------------

class ClockSampler:
    """Polls SM clock and clock-event reasons of one GPU during a region."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}

    def __init__(self, uuid: str, period_s: float = 0.005):
        self.ok = False
        self.samples = []
        self.period = period_s
        self.max_mhz = None
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            if self.nvml.nvmlDeviceGetHandleByUUID(("GPU-" + uuid).encode(),
                                                   ctypes.byref(self.h)) != 0:
                return
            mx = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None)
            self.reason_fn = fn or self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
            self.ok = True
        except OSError:
            pass

    def _poll(self):
        mhz = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self.nvml.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(mhz)) == 0 and \
                    self.reason_fn(self.h, ctypes.byref(rs)) == 0:
                self.samples.append((mhz.value, rs.value))
            time.sleep(self.period)

    def start(self):
        if not self.ok:
            return
        self._stop = threading.Event()
        self._t = threading.Thread(target=self._poll, daemon=True)
        self._t.start()

    def stop(self) -> dict:
        if not self.ok:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvml unavailable"]}
        self._stop.set()
        self._t.join()
        mhz = [m for m, _ in self.samples]
        bits = 0
        for _, r in self.samples:
            bits |= r
        reasons = [name for bit, name in self.REASONS.items() if bits & bit]
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(mhz)}


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


DECODE_SOURCES = ("kvq_decode.cu", "kvq_decode_common.cuh", "kvq_tile.cuh", "kvq_device.cuh",
                  "kvq_ranges.h")
GQA_SOURCES = ("kvq_decode_gqa.cu", "kvq_decode_common.cuh", "kvq_tile.cuh", "kvq_device.cuh",
               "kvq_ranges.h")
STEP_SOURCES = DECODE_SOURCES + ("kvq_store_row.cuh", "kvq_tables_item.cuh")
SPEC_HBM_GBS = 8000.0  # GB300 HBM3e, nominal (~8 TB/s)


def uses_gqa_kernel(wl, fused: bool = False) -> bool:
    """Whether the decode call runs the grouped-query kernel (INT8/INT4 pool,
    fp16 queries, 4 q heads per kv head; not inside the fused step)."""
    return (not fused and wl.kv_dtype in ("int8", "int4") and wl.q_dtype == "f16"
            and wl.q_heads == 4 * wl.kv_heads)


def kernel_source_sha(files=DECODE_SOURCES) -> str:
    """Hash of the decode kernel's source with // comments and blank lines
    removed, so that editing a comment keeps a DRAM-traffic record valid."""
    src = hashlib.sha256()
    for fn in files:
        with open(os.path.join(ROOT, "paged_quantized_kv_store_gb300", "csrc", fn)) as f:
            for line in f:
                code = re.sub(r"\s*//.*$", "", line.rstrip("\n")).rstrip()
                if code:
                    src.update(code.encode() + b"\n")
    return src.hexdigest()[:16]


def traffic_from_profile(workload: str, kind: str = "decode"):
    """DRAM bytes per launch of the decode kernel (kind "decode": the general
    kernel, "gqa": the grouped-query kernel) or of the fused step kernel (kind
    "step") from the committed ncu summary, if it was taken on the current
    kernel source (else None)."""
    sha = kernel_source_sha({"decode": DECODE_SOURCES, "gqa": GQA_SOURCES,
                             "step": STEP_SOURCES}[kind])
    kind = "decode" if kind == "gqa" else kind
    path = os.path.join(ROOT, "profiles", f"{kind}_{workload}_traffic.txt")
    try:
        text = open(path).read()
    except OSError:
        return None, sha
    m_sha = re.search(r"kernel_source_sha:\s*(\w+)", text)
    m_b = re.search(r"dram_bytes_per_launch_full_size:\s*([0-9.eE+]+)", text)
    if not m_sha or not m_b or m_sha.group(1) != sha:
        return None, sha
    return float(m_b.group(1)), sha


def max_over_ranks(x: float, dist, device) -> float:
    """The largest x over all ranks (x itself without a process group). The
    value travels in a tensor on `device`: a CUDA device for NCCL, the CPU for
    gloo."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def copy_bandwidth_gbs(dev, n_bytes: int = 1 << 31, reps: int = 10) -> float:
    """This GPU's device-to-device copy bandwidth right now (read + write bytes),
    best of `reps` copies of a 2 GiB buffer (larger than L2)."""
    import torch
    a = torch.empty(n_bytes // 2, dtype=torch.bfloat16, device=dev)
    b = torch.empty_like(a)
    a.fill_(1.0)
    best = float("inf")
    for _ in range(reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        b.copy_(a)
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    del a, b
    return 2 * n_bytes / (best / 1e3) / 1e9


def measure_block_copy(kvq, pool, wl, dev, peak: float, n_cow: int = 4096, n_swap: int = 1024,
                       reps: int = 20) -> dict:
    """kvq_copy_blocks on the workload's pool geometry: a copy-on-write of n_cow
    random blocks into a second device pool (HBM read + write), and a swap out
    / in of n_swap blocks through a pinned host pool, each against a plain
    copy of the same bytes on the same path (torch copy_)."""
    import torch

    block_bytes = pool.nbytes() // pool.num_blocks
    n_cow = min(n_cow, pool.num_blocks)
    n_swap = min(n_swap, pool.num_blocks)
    ids = torch.from_numpy(synthetic.permutation(wl.seed, 99, pool.num_blocks)
                           .astype(np.int32)).to(dev)

    def timed(fn):
        # 5 warm-up calls, then three batches of `reps` back-to-back calls,
        # each batch bracketed by CUDA events; the median batch's mean
        for _ in range(5):
            fn()
        torch.cuda.synchronize()
        batches = []
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(reps):
                fn()
            e1.record()
            torch.cuda.synchronize()
            batches.append(e0.elapsed_time(e1) / reps)
        return sorted(batches)[1]

    out = {"block_bytes": block_bytes}
    dst = kvq.KVPool.allocate(n_cow, wl.kv_heads, wl.kv_dtype, device=dev)
    seq = torch.arange(n_cow, dtype=torch.int32, device=dev)
    ms = timed(lambda: kvq.kvq_copy_blocks(pool, dst, ids[:n_cow], seq))
    moved = 2 * n_cow * block_bytes  # read + write
    out["cow"] = {"blocks": n_cow, "ms": round(ms, 4), "gbs": round(moved / ms / 1e6, 1),
                  "frac_of_peak": round(moved / ms / 1e6 / peak, 4)}
    del dst
    host = kvq.KVPool.allocate(n_swap, wl.kv_heads, wl.kv_dtype, pinned=True)
    seq = torch.arange(n_swap, dtype=torch.int32, device=dev)
    nbytes = n_swap * block_bytes
    ref_d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    ref_h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    for name, fn, ref in (
            ("swap_out", lambda: kvq.kvq_copy_blocks(pool, host, ids[:n_swap], seq),
             lambda: ref_h.copy_(ref_d, non_blocking=True)),
            ("swap_in", lambda: kvq.kvq_copy_blocks(host, pool, seq, ids[:n_swap]),
             lambda: ref_d.copy_(ref_h, non_blocking=True))):
        if name == "swap_in":  # the blocks swapped out go back where they were
            kvq.kvq_copy_blocks(pool, host, ids[:n_swap], seq)
        ms = timed(fn)
        ms_ref = timed(ref)
        out[name] = {"blocks": n_swap, "ms": round(ms, 4), "gbs": round(nbytes / ms / 1e6, 1),
                     "plain_copy_gbs": round(nbytes / ms_ref / 1e6, 1),
                     "frac_of_plain_copy": round(ms_ref / ms, 4)}
    del host, ref_d, ref_h
    return out


def measure_step_forms(sep_step, fused_step, out_sep, out_fused, reps: int = 50) -> dict:
    """The decode step as three calls (four kernels) and as kvq_decode_step
    (one cooperative kernel when the step carries no prefill chunk), each
    replayed from a CUDA graph, interleaved in
    blocks of ten so that both see the same clocks; the two outputs must agree
    to the decode tolerance."""
    import torch

    graphs = []
    for fn in (sep_step, fused_step):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        graphs.append(g)
    for g in graphs:
        for _ in range(3):
            g.replay()
    torch.cuda.synchronize()
    diff = (out_sep.float() - out_fused.float()).abs()
    tol = 2e-3 + 1e-2 * out_sep.float().abs()
    if not bool((diff <= tol).all()):
        raise RuntimeError("fused step output differs from the three-call step")
    ms = [0.0, 0.0]
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    for blk in range(reps // 10):
        for i, g in enumerate(graphs):
            ev[0].record()
            for _ in range(10):
                g.replay()
            ev[1].record()
            torch.cuda.synchronize()
            ms[i] += ev[0].elapsed_time(ev[1])
    n = (reps // 10) * 10
    return {"three_calls_ms": round(ms[0] / n, 5), "fused_ms": round(ms[1] / n, 5),
            "speedup": round(ms[0] / ms[1], 4), "cuda_graph": True, "reps": n}


def measured_tensor_peak():
    """(bf16 dense TFLOP/s burst, where it came from)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            v = float(json.load(f)["bf16_tflops"])
        if v > 0:
            return v, "measured"
    except (OSError, KeyError, ValueError, TypeError):
        pass
    return 1900.0, "fallback"


def measure_extend(kvq, dev, reps: int = 20) -> dict:
    """paged_extend_attn on the mixed step's prefill chunk alone: one fresh
    4096-token prompt chunk over INT8 KV (GQA 32q/8kv), stored, then attended
    causally. FLOPs: 4 * head_dim * q_heads * sum over queries of (position + 1);
    the products run on fp16 tensor cores (mma.sync), against the measured
    bf16 dense peak. torch's causal scaled_dot_product_attention on the same
    shapes (K/V dequantized to fp16, heads expanded) is timed for context."""
    import torch

    ew = synthetic.cfg5_prefill()
    wl = ew.wl
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}

    def to_dev(bits, dt):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(tdt[dt]).to(dev)

    pool = kvq.KVPool.allocate(wl.num_blocks, wl.kv_heads, wl.kv_dtype, device=dev)
    for slots, k, v in wl.setup_chunks():
        kvq.kv_store_quant(pool, to_dev(k, wl.in_dtype), to_dev(v, wl.in_dtype),
                           torch.from_numpy(slots).to(dev))
    slots, k, v = wl.step_store()
    kvq.kv_store_quant(pool, to_dev(k, wl.in_dtype), to_dev(v, wl.in_dtype),
                       torch.from_numpy(slots).to(dev))
    q = to_dev(ew.q_ext(), wl.q_dtype)
    out = torch.empty_like(q)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
    qo, kl, bt = i32(ew.qo_indptr), i32(ew.kv_lens), i32(wl.block_tables)
    ws = torch.empty(max(kvq.paged_extend_attn_workspace_size(
        wl.batch, ew.total_q, wl.q_heads, wl.kv_heads, wl.max_seq_len), 16),
        dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def timed(fn):
        # 5 warm-up calls, then three batches of `reps` back-to-back calls,
        # each batch bracketed by CUDA events; the median batch's mean
        for _ in range(5):
            fn()
        torch.cuda.synchronize()
        batches = []
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(reps):
                fn()
            e1.record()
            torch.cuda.synchronize()
            batches.append(e0.elapsed_time(e1) / reps)
        return sorted(batches)[1]

    C = ew.total_q
    flops = 4.0 * wl.head_dim * wl.q_heads * (C * (C + 1) / 2)
    peak, kind = measured_tensor_peak()
    res = {"workload": f"prefill chunk of {C} tokens, INT8 KV, GQA {wl.q_heads}q/{wl.kv_heads}kv",
           "flops_per_launch": flops, "peak_tflops": peak,
           "peak_kind": f"{kind} (bf16_tflops)", "default_variant": "tcgen05"}
    for variant in ("tcgen05", "mma_sync"):
        ms = timed(lambda: kvq.paged_extend_attn(pool, q, out, qo, kl, bt, wl.max_seq_len,
                                                 wl.sm_scale, ws, err, variant=variant))
        if kvq.kvq_check_error(err):
            raise RuntimeError("device error word set by the extend measurement")
        res[variant] = {"ms": round(ms, 4), "tflops": round(flops / ms / 1e9, 1),
                        "frac": round(flops / ms / 1e9 / peak, 4)}
    # context: the library's causal attention on dequantized fp16 K/V, same shapes
    try:
        import torch.nn.functional as F
        kd = torch.randn(1, wl.q_heads, C, wl.head_dim, dtype=torch.float16, device=dev)
        vd = torch.randn_like(kd)
        qd = q.view(1, C, wl.q_heads, wl.head_dim).transpose(1, 2).to(torch.float16)
        ms_ref = timed(lambda: F.scaled_dot_product_attention(qd, kd, vd, is_causal=True))
        res["torch_sdpa_fp16_ms"] = round(ms_ref, 4)
        res["torch_sdpa_fp16_tflops"] = round(flops / ms_ref / 1e9, 1)
    except Exception as e:  # noqa: BLE001 - context only
        res["torch_sdpa_fp16"] = f"not measured: {e}"
    del pool, ws
    return res


def store_bytes(wl, n_tokens: int) -> int:
    """HBM bytes of kv_store_quant for n_tokens: the new K and V rows read
    (16-bit), the pool rows and scale/zero pairs written, the slot mapping."""
    row_out = wl.kv_row_bytes() + (4 if wl.quantized else 0)
    return n_tokens * (2 * wl.kv_heads * (2 * wl.head_dim + row_out) + 8)


def time_store(kvq, pool, wl, d_k, d_v, d_slots, dev, peak: float, reps: int = 100) -> dict:
    """kv_store_quant of the given rows alone (graph-replayed), L2 flushed by
    a write of twice its size before every call, outside the CUDA events."""
    import torch

    l2 = int(torch.cuda.get_device_properties(dev).L2_cache_size)
    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    kvq.kv_store_quant(pool, d_k, d_v, d_slots, err)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        kvq.kv_store_quant(pool, d_k, d_v, d_slots, err)
    ms = []
    for i in range(reps + 3):
        flush.fill_(i & 0xFF)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= 3:
            ms.append(e0.elapsed_time(e1))
    if kvq.kvq_check_error(err):
        raise RuntimeError("device error word set by the store measurement")
    n = int(d_slots.numel())
    sb = store_bytes(wl, n)
    m = float(np.mean(ms))
    del flush, g
    return {"tokens": n, "bytes": sb, "ms_mean": round(m, 5),
            "ms_median": round(float(np.median(ms)), 5),
            "gbs": round(sb / (m / 1e3) / 1e9, 1), "frac": round(sb / (m / 1e3) / 1e9 / peak, 4),
            "l2": "flushed before every call", "cuda_graph": True, "reps": reps}


def stored_workload(kvq, wl, dev):
    """The workload's pool with its context and the step's new tokens stored
    through kv_store_quant, its block tables from kvq_block_tables_from_req_to_token,
    and the step's queries and lengths on the device."""
    import torch
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}

    def to_dev(bits, dt):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(tdt[dt]).to(dev)

    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
    pool = kvq.KVPool.allocate(wl.num_blocks, wl.kv_heads, wl.kv_dtype, device=dev)
    for slots, k, v in wl.setup_chunks(max_tokens=1 << 17):
        kvq.kv_store_quant(pool, to_dev(k, wl.in_dtype), to_dev(v, wl.in_dtype),
                           torch.from_numpy(slots).to(dev))
    slots, k_new, v_new = wl.step_store()
    d_slots = torch.from_numpy(slots).to(dev)
    d_k, d_v = to_dev(k_new, wl.in_dtype), to_dev(v_new, wl.in_dtype)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    kvq.kv_store_quant(pool, d_k, d_v, d_slots, err)
    bt = torch.empty((wl.batch, wl.max_blocks_per_seq), dtype=torch.int32, device=dev)
    kvq.kvq_block_tables_from_req_to_token(i32(wl.req_to_token), i32(wl.req_pool_indices),
                                           i32(wl.seq_lens), bt, err)
    return pool, bt, to_dev(wl.q(), wl.q_dtype), i32(wl.seq_lens), err, (d_k, d_v, d_slots)


def replica_pools(kvq, pool, l2: int):
    """The pool and enough copies of it that the copies together hold at least
    3 x L2 (just the pool when it alone is larger): calls rotated over them
    start with a cold L2."""
    nb = pool.nbytes()
    R = 1 if nb > 3 * l2 else -(-3 * l2 // nb)
    pools = [pool]
    for _ in range(R - 1):
        pools.append(kvq.KVPool(pool.k.clone(), pool.v.clone(),
                                None if pool.k_sz is None else pool.k_sz.clone(),
                                None if pool.v_sz is None else pool.v_sz.clone(),
                                pool.num_blocks, pool.kv_heads, pool.kv_dtype))
    return pools


def time_rotated(graphs, reps: int, stream) -> list:
    """CUDA-event times (ms) of `reps` graph replays rotated over `graphs`,
    after a warm-up in the same rotation."""
    import torch
    R = len(graphs)
    for i in range(3 * R):
        graphs[i % R].replay()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    for i, (e0, e1) in enumerate(ev):
        e0.record(stream)
        graphs[i % R].replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return [e0.elapsed_time(e1) for e0, e1 in ev]


def measure_shared_prefix(kvq, dev, peak: float, reps: int = 60) -> dict:
    """The shared-prefix (cascade) decode against the plain decode on the
    same pool and GPU: cfg4's structure with an 8192-token prefix that all 64
    requests hold ("pymllm Runtime Design", KV cache and prefix cache: a
    radix hit shares leading blocks). Both graph-replayed over replica pools
    (cold L2); the two outputs are checked against each other."""
    import torch

    wl = synthetic.cfg4_long_prefix()
    members, shared = prefix_groups(wl)
    pool, bt, q, sl, err, _ = stored_workload(kvq, wl, dev)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
    groups = kvq.SharedPrefixGroups(i32([0, len(members)]), i32(members), i32([shared]), shared)
    ws = torch.empty(max(16, kvq.paged_decode_attn_workspace_size(
        wl.batch, wl.q_heads, wl.kv_heads, wl.max_seq_len, 0)), dtype=torch.uint8, device=dev)
    sp_ws = torch.empty(kvq.paged_decode_attn_shared_prefix_workspace_size(
        wl.batch, wl.q_heads, wl.kv_heads, wl.max_seq_len, shared, 0), dtype=torch.uint8,
        device=dev)
    l2 = int(torch.cuda.get_device_properties(dev).L2_cache_size)
    pools = replica_pools(kvq, pool, l2)
    stream = torch.cuda.current_stream(dev)
    outs, times = {}, {}
    for mode in ("plain", "cascade"):
        out = torch.empty_like(q)
        graphs = []
        for pl in pools:
            if mode == "plain":
                call = (lambda pl=pl: kvq.paged_decode_attn(pl, q, out, bt, sl, wl.max_seq_len,
                                                            wl.sm_scale, 0, ws, err))
            else:
                call = (lambda pl=pl: kvq.paged_decode_attn_shared_prefix(
                    pl, q, out, bt, sl, wl.max_seq_len, wl.sm_scale, groups, 0, sp_ws, err))
            for _ in range(3):
                call()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                call()
            graphs.append(g)
        times[mode] = time_rotated(graphs, reps, stream)
        outs[mode] = out
        del graphs
    if kvq.kvq_check_error(err):
        raise RuntimeError("device error word set by the shared-prefix measurement")
    a, b = outs["plain"].double(), outs["cascade"].double()
    diff = (a - b).abs()
    agree = bool(((diff <= 2e-3) | (diff <= 1e-2 * b.abs())).all().item())
    alg, logical = decode_algorithmic_bytes(wl), decode_logical_bytes(wl)
    mp, mc = float(np.mean(times["plain"])), float(np.mean(times["cascade"]))
    res = {
        "workload": wl.description,
        "members": len(members), "shared_tokens": 16 * shared,
        "unique_bytes": alg, "logical_bytes": logical,
        "plain": {"kernels": "decode_gqa_kernel + combine_kernel", "ms_mean": round(mp, 5),
                  "unique_gbs": round(alg / (mp / 1e3) / 1e9, 1),
                  "logical_gbs": round(logical / (mp / 1e3) / 1e9, 1)},
        "cascade": {"kernels": "prefix_kernel + decode_kernel + combine_kernel",
                    "ms_mean": round(mc, 5), "unique_gbs": round(alg / (mc / 1e3) / 1e9, 1),
                    "frac": round(alg / (mc / 1e3) / 1e9 / peak, 4)},
        "speedup": round(mp / mc, 3),
        "outputs_agree": agree,
        "l2": f"cold: {len(pools)} replica pools rotated ({pool.nbytes() / 1e6:.1f} MB each)",
        "cuda_graph": True, "reps": reps,
    }
    del pools, pool, ws, sp_ws
    torch.cuda.empty_cache()
    return res


def measure_workload(kvq, name: str, dev, peak: float, reps: int = 100) -> dict:
    """One workload's decode call (paged_decode_attn: decode + combine kernels,
    graph-replayed, CUDA events on the launching stream) and its store
    (kv_store_quant of the step's tokens: each request's new token and, for
    the mixed step, the 4096-token prefill chunk).

    The decode is timed with a cold L2: a pool larger than L2 is read anew by
    every call; a pool that fits is replicated R times (R x bytes >= 3 x L2)
    and the calls rotate over the replicas, as the layers of a model would.
    The warm-L2 time (one pool, back to back) is reported beside it. The
    store is timed with L2 flushed (a write larger than L2) before every
    call, outside the timed events."""
    import torch

    wl = synthetic.by_name(name)
    pool, bt, q, sl, err, (d_k, d_v, d_slots) = stored_workload(kvq, wl, dev)
    out = torch.empty_like(q)
    ws = torch.empty(max(16, kvq.paged_decode_attn_workspace_size(
        wl.batch, wl.q_heads, wl.kv_heads, wl.max_seq_len, 0)), dtype=torch.uint8, device=dev)
    l2 = int(torch.cuda.get_device_properties(dev).L2_cache_size)
    alg, logical = decode_algorithmic_bytes(wl), decode_logical_bytes(wl)
    pool_bytes = pool.nbytes()
    pools = replica_pools(kvq, pool, l2)
    R = len(pools)
    graphs = []
    for pl in pools:
        call = (lambda pl=pl: kvq.paged_decode_attn(pl, q, out, bt, sl, wl.max_seq_len,
                                                    wl.sm_scale, 0, ws, err))
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            call()
        graphs.append(g)
    stream = torch.cuda.current_stream(dev)

    def timed(order):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in order]
        for i in range(min(len(order), 3 * R)):  # warm-up in the same rotation
            graphs[order[i]].replay()
        torch.cuda.synchronize()
        for (e0, e1), r in zip(ev, order):
            e0.record(stream)
            graphs[r].replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return [e0.elapsed_time(e1) for e0, e1 in ev]

    cold = timed([i % R for i in range(reps)])
    warm = timed([0] * reps)
    if kvq.kvq_check_error(err):
        raise RuntimeError(f"device error word set by the {name} decode measurement")

    store = time_store(kvq, pool, wl, d_k, d_v, d_slots, dev, peak, reps)
    mc, mw = float(np.mean(cold)), float(np.mean(warm))
    res = {
        "workload": f"{wl.name}: {wl.description}",
        "kernel": ("grouped-query decode kernel + combine" if uses_gqa_kernel(wl)
                   else "decode kernel + combine"),
        "decode_ms_mean": round(mc, 5), "decode_ms_median": round(float(np.median(cold)), 5),
        "decode_ms_min": round(float(np.min(cold)), 5),
        "decode_ms_max": round(float(np.max(cold)), 5),
        "decode_tokens_per_s": round(wl.batch / (mc / 1e3), 1),
        "algorithmic_bytes": alg, "logical_bytes": logical,
        "decode_gbs": round(alg / (mc / 1e3) / 1e9, 1),
        "frac": round(alg / (mc / 1e3) / 1e9 / peak, 4),
        "frac_of_spec_8tbs": round(alg / (mc / 1e3) / 1e9 / SPEC_HBM_GBS, 4),
        "logical_gbs": round(logical / (mc / 1e3) / 1e9, 1),
        "l2": (f"cold: {R} replica pools rotated ({R} x {pool_bytes / 1e6:.1f} MB >= 3 x L2 of "
               f"{l2 / 1e6:.0f} MB)" if R > 1 else
               f"cold: the pool ({pool_bytes / 1e6:.0f} MB) is more than 3 x L2"),
        "warm_l2": {"decode_ms_mean": round(mw, 5),
                    "decode_gbs": round(alg / (mw / 1e3) / 1e9, 1),
                    "frac": round(alg / (mw / 1e3) / 1e9 / peak, 4)},
        "store": store,
        "cuda_graph": True, "reps": reps,
    }
    traffic, sha = traffic_from_profile(wl.name, "gqa" if uses_gqa_kernel(wl) else "decode")
    res["traffic"] = traffic  # ncu DRAM bytes per decode launch, null when taken on other source
    res["traffic_over_algorithmic"] = None if traffic is None else round(traffic / alg, 4)
    res["kernel_source_sha"] = sha
    del graphs, pools, pool, ws
    torch.cuda.empty_cache()
    return res


# ---- our arm ---------------------------------------------------------------------

def run_ours(args, rank: int, world: int, dist):
    import torch

    import paged_quantized_kv_store_gb300 as kvq

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    kvq.load()
    wl = make_workload(args.workload, args.batch, rank)
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}

    def to_dev(bits, dt):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(tdt[dt]).to(dev)

    # ---- setup (untimed): pool, stored context, per-step inputs -------------------
    pool = kvq.KVPool.allocate(wl.num_blocks, wl.kv_heads, wl.kv_dtype, device=dev)
    for slots, k, v in wl.setup_chunks(max_tokens=1 << 17):
        kvq.kv_store_quant(pool, to_dev(k, wl.in_dtype), to_dev(v, wl.in_dtype),
                           torch.from_numpy(slots).to(dev))
    torch.cuda.synchronize()
    slots, k_new, v_new = wl.step_store()
    h_inputs = {
        "q": wl.q().view(np.int16), "k_new": k_new.view(np.int16), "v_new": v_new.view(np.int16),
        "slot_mapping": slots, "seq_lens": wl.seq_lens.astype(np.int32),
        "req_pool_indices": wl.req_pool_indices.astype(np.int32),
    }
    groups = prefix_groups(wl) if args.shared_prefix != "off" else None
    if args.shared_prefix == "on" and groups is None:
        raise SystemExit(f"--shared-prefix on: {wl.name} has no shared prefix")
    if groups is not None:
        # the group description is a per-step input like the lengths
        h_inputs["grp_off"] = np.array([0, len(groups[0])], dtype=np.int32)
        h_inputs["grp_mem"] = np.array(groups[0], dtype=np.int32)
        h_inputs["grp_shared"] = np.array([groups[1]], dtype=np.int32)
    views = {"q": tdt[wl.q_dtype], "k_new": tdt[wl.in_dtype], "v_new": tdt[wl.in_dtype]}

    def typed(raw):
        return {k: (t.view(views[k]) if k in views else t) for k, t in raw.items()}

    d_raw = {k: torch.from_numpy(np.ascontiguousarray(a)).to(dev) for k, a in h_inputs.items()}
    d_in = typed(d_raw)
    r2t = torch.from_numpy(wl.req_to_token).to(dev)
    step = kvq.DecodeStep(pool, wl.batch, wl.q_heads, wl.max_blocks_per_seq, wl.max_seq_len,
                          tdt[wl.q_dtype], num_splits=args.num_splits, device=dev)
    fstep = None
    if groups is None and wl.in_dtype == wl.q_dtype:
        fstep = kvq.DecodeStep(pool, wl.batch, wl.q_heads, wl.max_blocks_per_seq,
                               wl.max_seq_len, tdt[wl.q_dtype], num_splits=args.num_splits,
                               device=dev, fused=True)
    if args.fused_step and fstep is None:
        raise SystemExit("--fused-step: needs no shared prefix and new rows in q's dtype")
    plan = kvq.paged_decode_attn_plan(wl.batch, wl.q_heads, wl.kv_heads, wl.max_seq_len,
                                      args.num_splits)
    stream = torch.cuda.current_stream(dev)

    def pre_step(inp):
        kvq.kvq_block_tables_from_req_to_token(r2t, inp["req_pool_indices"], inp["seq_lens"],
                                               step.block_tables, step.dev_err)
        kvq.kv_store_quant(pool, inp["k_new"], inp["v_new"], inp["slot_mapping"], step.dev_err)

    def fused(inp):
        fstep(r2t, inp["req_pool_indices"], inp["seq_lens"], inp["q"], inp["k_new"],
              inp["v_new"], inp["slot_mapping"], wl.sm_scale)

    if args.fused_step:
        def pre_step(inp):
            pass

        def dec_step(inp):
            fused(inp)

        step = fstep
        if kvq.kvq_decode_step_fused(wl.batch, len(wl.step_store()[0])):
            launches_per_step = 1
            decode_kernels = "kvq_decode_step (step_kernel: tables + store, decode, combine)"
        else:
            launches_per_step = 4
            decode_kernels = ("kvq_decode_step as four kernels (prefill chunk in the step): "
                              "tables, store, decode, combine")
    elif groups is None:
        def dec_step(inp):
            kvq.paged_decode_attn(pool, inp["q"], step.out, step.block_tables, inp["seq_lens"],
                                  wl.max_seq_len, wl.sm_scale, args.num_splits, step.workspace,
                                  step.dev_err)

        launches_per_step = 4  # tables, store, decode, combine
        decode_kernels = "paged_decode_attn (decode_kernel + combine_kernel)"
    else:
        sp_bytes = kvq.paged_decode_attn_shared_prefix_workspace_size(
            wl.batch, wl.q_heads, wl.kv_heads, wl.max_seq_len, groups[1], args.num_splits)
        sp_ws = torch.empty(sp_bytes, dtype=torch.uint8, device=dev)

        def dec_step(inp):
            g = kvq.SharedPrefixGroups(inp["grp_off"], inp["grp_mem"], inp["grp_shared"],
                                       groups[1])
            kvq.paged_decode_attn_shared_prefix(pool, inp["q"], step.out, step.block_tables,
                                                inp["seq_lens"], wl.max_seq_len, wl.sm_scale, g,
                                                args.num_splits, sp_ws, step.dev_err)

        launches_per_step = 5  # tables, store, prefix, decode, combine (+ a memset)
        decode_kernels = ("paged_decode_attn_shared_prefix (prefix_kernel + decode_kernel + "
                          "combine_kernel)")

    for _ in range(max(args.warmup, 1)):
        pre_step(d_in)
        dec_step(d_in)
    torch.cuda.synchronize()
    bits = kvq.kvq_check_error(step.dev_err)
    if bits:
        raise RuntimeError(f"device error word {bits:#x} after warm-up")
    use_graph = not args.no_graph
    if use_graph:
        # the step as two CUDA graphs (a decode step is replayed as a graph in
        # serving runtimes); the decode call is timed between the two replays
        g_dec = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_dec):
            dec_step(d_in)
        run_dec = g_dec.replay
        if args.fused_step:  # nothing runs before the one launch
            def run_pre():
                pass
        else:
            g_pre = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_pre):
                pre_step(d_in)
            run_pre = g_pre.replay
        for _ in range(args.warmup):
            run_pre()
            run_dec()
        torch.cuda.synchronize()
    else:
        def run_pre():
            pre_step(d_in)

        def run_dec():
            dec_step(d_in)

    uuid = str(torch.cuda.get_device_properties(dev).uuid)
    sampler = ClockSampler(uuid)
    K = args.steps
    ev_d0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_d1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    t0.record(stream)
    for i in range(K):
        run_pre()
        ev_d0[i].record(stream)
        run_dec()
        ev_d1[i].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if dist is not None:
        dist.barrier()
    ms_total = t0.elapsed_time(t1)
    decode_ms = [ev_d0[i].elapsed_time(ev_d1[i]) for i in range(K)]
    if dist is not None:
        ms_total = max_over_ranks(ms_total, dist, dev)
    ms_step = ms_total / K
    tokens_per_step = wl.batch * world
    value = tokens_per_step / (ms_step / 1e3)

    # ---- end to end through the public API with host buffers -------------------------
    e2e = None
    if not args.no_e2e:
        pinned = {k: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
                  for k, a in h_inputs.items()}
        out_host = torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory()
        e_raw = {k: torch.empty_like(v) for k, v in d_raw.items()}
        e_in = typed(e_raw)
        h2d = sum(t.numel() * t.element_size() for t in pinned.values())
        d2h = out_host.numel() * out_host.element_size()

        def e2e_body():
            for key, t in pinned.items():
                e_raw[key].copy_(t, non_blocking=True)
            pre_step(e_in)
            dec_step(e_in)
            out_host.copy_(step.out, non_blocking=True)

        if use_graph:
            g_e2e = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_e2e):
                e2e_body()
            e2e_step = g_e2e.replay
        else:
            e2e_step = e2e_body
        for _ in range(max(3, args.warmup)):
            e2e_step()
        torch.cuda.synchronize()
        if not torch.equal(out_host.to(dev), step.out):
            raise RuntimeError("end-to-end output differs from the device-resident step")
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(K):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        ms_e2e = e0.elapsed_time(e1)
        if dist is not None:
            ms_e2e = max_over_ranks(ms_e2e, dist, dev)
        e2e = {"value": tokens_per_step / (ms_e2e / K / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}

    bits = kvq.kvq_check_error(step.dev_err)
    if bits:
        raise RuntimeError(f"device error word {bits:#x} after the timed steps")

    # ---- roofline of the dominant call (decode + combine) ---------------------------
    box_copy = copy_bandwidth_gbs(dev)
    alg = decode_algorithmic_bytes(wl)
    logical = decode_logical_bytes(wl)
    mean_decode_ms = float(np.mean(decode_ms))
    peak, peak_kind = measured_peak()
    achieved = alg / (mean_decode_ms / 1e3) / 1e9
    single = args.fused_step and launches_per_step == 1
    gqa = uses_gqa_kernel(wl, fused=bool(args.fused_step))
    traffic, sha = traffic_from_profile(wl.name, "step" if single else ("gqa" if gqa else "decode"))
    if gqa and groups is None and not args.fused_step:
        decode_kernels = "paged_decode_attn (decode_gqa_kernel + combine_kernel)"
    roofline = {
        "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
        "frac": round(achieved / peak, 4), "traffic": traffic,
        "kernel": decode_kernels,
        "peak_kind": f"{peak_kind} (hbm_gbs)",
        "frac_of_spec_8tbs": round(achieved / SPEC_HBM_GBS, 4),
        "algorithmic_bytes_per_launch": alg, "logical_bytes_per_launch": logical,
        "decode_ms_mean": round(mean_decode_ms, 5),
        "decode_ms_median": round(float(np.median(decode_ms)), 5),
        "decode_ms_min": round(float(np.min(decode_ms)), 5),
        "decode_ms_max": round(float(np.max(decode_ms)), 5),
        "logical_gbs": round(logical / (mean_decode_ms / 1e3) / 1e9, 1),
        "kernel_source_sha": sha,
        "copy_gbs_this_gpu": round(box_copy, 1),
        "frac_of_this_gpu_copy": round(achieved / box_copy, 4),
    }

    # the step's store (each request's new token, and a prefill chunk if the
    # step has one) alone, L2 flushed before each call
    store = time_store(kvq, pool, wl, d_in["k_new"], d_in["v_new"], d_in["slot_mapping"], dev,
                       peak, reps=50)
    l2_bytes = int(torch.cuda.get_device_properties(dev).L2_cache_size)
    pool_bytes = pool.nbytes()
    l2_note = (f"no flush: the pool ({pool_bytes / 1e6:.0f} MB) is more than 3 x L2 "
               f"({l2_bytes / 1e6:.0f} MB); every step reads it anew" if pool_bytes > 3 * l2_bytes
               else f"warm L2: the pool ({pool_bytes / 1e6:.0f} MB) fits in L2 "
                    f"({l2_bytes / 1e6:.0f} MB); the cold-L2 figure of this workload is in "
                    f"extras.workloads")

    extras = None
    if not args.no_extras:
        extras = {"workloads": {}}
        for name in ("cfg2", "cfg4", "cfg5"):
            if name != wl.name:
                extras["workloads"][name] = measure_workload(kvq, name, dev, peak)
        extras["kvq_copy_blocks"] = measure_block_copy(kvq, pool, wl, dev, peak)
        extras["paged_extend_attn"] = measure_extend(kvq, dev)
        extras["shared_prefix"] = measure_shared_prefix(kvq, dev, peak)
        if fstep is not None:
            sep = kvq.DecodeStep(pool, wl.batch, wl.q_heads, wl.max_blocks_per_seq,
                                 wl.max_seq_len, tdt[wl.q_dtype], num_splits=args.num_splits,
                                 device=dev)

            def sep_call():
                sep(r2t, d_in["req_pool_indices"], d_in["seq_lens"], d_in["q"], d_in["k_new"],
                    d_in["v_new"], d_in["slot_mapping"], wl.sm_scale)

            extras["kvq_decode_step"] = measure_step_forms(sep_call, lambda: fused(d_in),
                                                           sep.out, fstep.out)
            extras["kvq_decode_step"]["single_launch"] = kvq.kvq_decode_step_fused(
                wl.batch, int(d_in["slot_mapping"].numel()))
            if kvq.kvq_check_error(sep.dev_err) or kvq.kvq_check_error(fstep.dev_err):
                raise RuntimeError("device error word set by the step-form measurement")
        bits = kvq.kvq_check_error(step.dev_err)
        if bits:
            raise RuntimeError(f"device error word {bits:#x} after the copy measurement")

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"int8": "u8", "int4": "u4", "f16": "f16", "bf16": "bf16"}[wl.kv_dtype],
        "data": "synthetic (seeded counter-based generator; no dataset)",
        "config": {**workload_desc(wl), "l2": l2_note,
                   "cuda_graph": use_graph, "fused_step": bool(args.fused_step),
                   "shared_prefix": None if groups is None else
                   {"groups": 1, "members": len(groups[0]), "shared_blocks": groups[1]},
                   "plan": plan, "parallelism": f"replicas x{world} (no data-path collective)"},
        "roofline": roofline, "store": store, "clocks": clocks, "e2e": e2e,
        "gpu_launches": launches_per_step * K,
        "decode_hbm_gbs": round(achieved, 1),
        "extras": extras,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(wl, budget_s=20.0)
    return result


# ---- the oracle as the CPU baseline / reference arm ---------------------------------

def _oracle_sample(wl, n_req: int):
    """Compact oracle pools of the first n_req requests, context stored (setup)."""
    import oracle
    reqs = []
    for b in range(n_req):
        L = int(wl.seq_lens[b])
        nblk = max(1, (L + 15) // 16)
        pool = oracle.Pool(nblk, wl.kv_heads, wl.head_dim, wl.kv_dtype)
        if L > 1:
            k = wl.ctx_rows("k", b, 0, L - 1)
            v = wl.ctx_rows("v", b, 0, L - 1)
            oracle.kv_store(pool, k, v, wl.in_dtype, np.arange(L - 1, dtype=np.int64))
        r2t = np.arange(max(L, 16), dtype=np.int32)[None]
        reqs.append((b, L, pool, r2t))
    return reqs


def _oracle_step(wl, reqs, q, k_new, v_new):
    """One step of the oracle over the sampled requests: block table, store of
    the new token, decode of every q head."""
    import oracle
    outs = []
    for b, L, pool, r2t in reqs:
        nblk = max(1, (L + 15) // 16)
        bt, err = oracle.block_tables(r2t, np.array([0], np.int32), np.array([L], np.int32),
                                      nblk)
        if L > 0:
            oracle.kv_store(pool, k_new[b:b + 1], v_new[b:b + 1], wl.in_dtype,
                            np.array([L - 1], np.int64))
        outs.append(oracle.paged_decode(pool, q[b:b + 1], wl.q_dtype, bt,
                                        np.array([L], np.int32), wl.sm_scale))
    return outs


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine)."""
    import platform
    import subprocess
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip().lower() == "model name":
                return f"{line.split(':', 1)[1].strip()} ({platform.machine()})"
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu model", "hardware"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def _oracle_store_rate(wl, budget_s: float) -> dict:
    """The oracle's quantizing store of the step's tokens (each request's new
    token, and the prefill chunk if the step has one), one host core, on as
    many of them as fit the time budget."""
    import oracle
    slots, k, v = wl.step_store()
    n = len(slots)
    pool = oracle.Pool(wl.num_blocks, wl.kv_heads, wl.head_dim, wl.kv_dtype)
    t = time.perf_counter()
    oracle.kv_store(pool, k[:1], v[:1], wl.in_dtype, slots[:1])
    per_tok = max(time.perf_counter() - t, 1e-7)
    m = int(max(1, min(n, budget_s / per_tok)))
    t = time.perf_counter()
    oracle.kv_store(pool, k[:m], v[:m], wl.in_dtype, slots[:m])
    dt = time.perf_counter() - t
    sb = store_bytes(wl, m)
    return {"tokens": m, "of_tokens": n, "s": round(dt, 4),
            "tokens_per_s": round(m / dt, 1), "gbs": round(sb / dt / 1e9, 4)}


def cpu_baseline(wl, budget_s: float = 20.0, n_req: int = 0) -> dict:
    """The oracle, single-threaded, on a bounded sample of the workload: the
    decode of a sample of requests (block table, store of the new token, fp64
    attention of every q head) gives the line's value; the store of the
    step's tokens is timed on its own beside it."""
    q = wl.q()
    k_new, v_new = wl.new_rows("k"), wl.new_rows("v")
    if n_req <= 0:
        probe = _oracle_sample(wl, 1)
        t = time.perf_counter()
        _oracle_step(wl, probe, q, k_new, v_new)
        per_req = time.perf_counter() - t
        n_req = int(max(1, min(wl.batch, budget_s / max(per_req, 1e-6))))
    reqs = _oracle_sample(wl, n_req)
    t = time.perf_counter()
    _oracle_step(wl, reqs, q, k_new, v_new)
    dt = time.perf_counter() - t
    store = _oracle_store_rate(wl, budget_s=min(5.0, budget_s / 4))
    return {"value": round(n_req / dt, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{n_req} of the {wl.batch} requests of one step (block table, store of "
                      f"the new token, fp64 decode of all {wl.q_heads} q heads), "
                      f"{dt:.1f} s on one host core",
            "decode": {"requests": n_req, "s": round(dt, 3),
                       "requests_per_s": round(n_req / dt, 3)},
            "store": store, "nproc": os.cpu_count(), "cpu_model": cpu_model()}


def run_reference(args, rank: int):
    if rank != 0:
        return None
    wl = make_workload(args.workload, args.batch, 0)
    q = wl.q()
    k_new, v_new = wl.new_rows("k"), wl.new_rows("v")
    probe = _oracle_sample(wl, 1)
    t = time.perf_counter()
    _oracle_step(wl, probe, q, k_new, v_new)
    per_req = time.perf_counter() - t
    budget = 150.0 / max(1, args.steps + args.warmup)  # whole run within a few minutes
    n_req = int(max(1, min(wl.batch, budget / max(per_req, 1e-6))))
    reqs = _oracle_sample(wl, n_req)
    for _ in range(args.warmup):
        _oracle_step(wl, reqs, q, k_new, v_new)
    times = []
    for _ in range(args.steps):
        t = time.perf_counter()
        _oracle_step(wl, reqs, q, k_new, v_new)
        times.append(time.perf_counter() - t)
    ms = float(np.mean(times)) * 1e3
    value = n_req / (ms / 1e3)
    sample = (f"{n_req} of the {wl.batch} requests per step (block table, store of the new "
              f"token, fp64 decode of all {wl.q_heads} q heads)")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
        "n_gpus": 0, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded counter-based generator; no dataset)",
        "config": {**workload_desc(wl), "reference": "CPU oracle (oracle/kvq_oracle.cpp), "
                   "single-threaded; the pages ship no code to install"},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample, "nproc": os.cpu_count(), "cpu_model": cpu_model()},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as tdist
        backend = "gloo" if args.impl == "reference" else "nccl"
        if backend == "nccl":
            import torch
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        tdist.init_process_group(backend=backend)
        dist = tdist
    if args.extend_only:
        import torch

        import paged_quantized_kv_store_gb300 as kvq
        kvq.load()
        res = {"paged_extend_attn": measure_extend(kvq, torch.device("cuda"))}
    elif args.impl == "reference":
        res = run_reference(args, rank)
    else:
        res = run_ours(args, rank, world, dist)
    if rank == 0 and res is not None:
        line = json.dumps(res)
        print(line, flush=True)
        if args.json_out:
            with open(args.json_out, "w") as f:
                f.write(line + "\n")
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
