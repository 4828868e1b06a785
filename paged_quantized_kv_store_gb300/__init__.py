"""Python binding of libkvq: paged, quantized KV store + paged decode attention.

A thin ctypes layer over the C ABI declared in ``include/kvq.h``. Functions
keep the C names; they take torch tensors (device memory) and pass raw
pointers, sizes and the current CUDA stream. Every step of the computation
runs in libkvq's CUDA kernels; this module only marshals arguments. If the
shared library is missing or cannot be loaded, ``load()`` raises: there is no
fallback.

Pages followed (see the header for details): "pymllm Runtime Design"
(ReqToTokenPool / KVPool / store_cache) and the LMDeploy article on
devpress.csdn.net (§2.2 blocked KV cache, §2.4 online INT8/INT4 KV
quantization, §3.2 and §4.2 paged decode attention).
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

from . import _build

LIB_PATH = _build.LIB_PATH

KVQ_F16, KVQ_BF16, KVQ_INT4, KVQ_INT8 = 0, 1, 4, 8
DTYPE_CODES = {"f16": KVQ_F16, "bf16": KVQ_BF16, "int4": KVQ_INT4, "int8": KVQ_INT8}
BLOCK_SIZE = 16
HEAD_DIM = 128

DEV_ERR_BITS = {
    "req_slot": 1, "length": 2, "kv_index": 4, "not_blocked": 8, "slot": 16, "block_id": 32,
    "timeout": 64, "prefix": 128,
}

_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported configuration", 3: "CUDA error",
           4: "device reported an out-of-range index or length", 5: "workspace"}

_lib = None


class KvqError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {_STATUS.get(status, status)} (status {status})")
        self.status = status


class _Pool(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("k_sz", ctypes.c_void_p),
                ("v_sz", ctypes.c_void_p), ("num_blocks", ctypes.c_int64),
                ("block_size", ctypes.c_int32), ("kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("kv_dtype", ctypes.c_int32)]


class _Plan(ctypes.Structure):
    _fields_ = [("min_blocks_per_warp", ctypes.c_int32), ("warps", ctypes.c_int32),
                ("head_groups", ctypes.c_int32), ("heads_per_group", ctypes.c_int32),
                ("num_sms", ctypes.c_int32), ("max_ctas_per_sm", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_size_t)]


EXPORTED = ["kv_store_quant", "kvq_block_tables_from_req_to_token", "paged_decode_attn_plan",
            "paged_decode_attn_workspace_size", "paged_decode_attn", "kvq_check_error",
            "kvq_status_string", "kvq_version", "paged_decode_attn_noalloc",
            "paged_decode_attn_shared_prefix_workspace_size", "paged_decode_attn_shared_prefix",
            "kvq_copy_blocks", "paged_extend_attn_workspace_size", "paged_extend_attn",
            "kvq_decode_step_workspace_size", "kvq_decode_step", "kvq_decode_step_fused"]


def load(build_if_missing: bool = False):
    """Load libkvq.so (optionally building it first). Raises when unavailable."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing:
        _build.build()
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libkvq is not built ({LIB_PATH} missing); run "
                          "__graft_entry__.build() or paged_quantized_kv_store_gb300._build")
    lib = ctypes.CDLL(LIB_PATH)
    P, I64, I32, SZ, F = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t,
                          ctypes.c_float)
    lib.kv_store_quant.argtypes = [ctypes.POINTER(_Pool), P, P, I32, P, I64, P, P]
    lib.kv_store_quant.restype = ctypes.c_int
    lib.kvq_block_tables_from_req_to_token.argtypes = [P, I32, I32, P, P, I32, I32, P, P, P]
    lib.kvq_block_tables_from_req_to_token.restype = ctypes.c_int
    lib.paged_decode_attn_plan.argtypes = [I32, I32, I32, I32, I32, I32, I32,
                                           ctypes.POINTER(_Plan)]
    lib.paged_decode_attn_plan.restype = ctypes.c_int
    lib.paged_decode_attn_workspace_size.argtypes = [I32, I32, I32, I32, I32, I32]
    lib.paged_decode_attn_workspace_size.restype = SZ
    lib.paged_decode_attn.argtypes = [ctypes.POINTER(_Pool), P, I32, P, P, I32, P, I32, I32, I32,
                                      F, I32, P, SZ, P, P]
    lib.paged_decode_attn.restype = ctypes.c_int
    lib.paged_decode_attn_noalloc.argtypes = [ctypes.POINTER(_Pool), P, I32, P, P, I32, P, I32,
                                              I32, I32, F, I32, P, P]
    lib.paged_decode_attn_noalloc.restype = ctypes.c_int
    lib.paged_decode_attn_shared_prefix_workspace_size.argtypes = [I32, I32, I32, I32, I32, I32,
                                                                   I32, ctypes.POINTER(SZ)]
    lib.paged_decode_attn_shared_prefix_workspace_size.restype = ctypes.c_int
    lib.paged_decode_attn_shared_prefix.argtypes = [ctypes.POINTER(_Pool), P, I32, P, P, I32, P,
                                                    I32, I32, I32, F, P, P, P, I32, I32, I32,
                                                    I32, P, SZ, P, P]
    lib.paged_decode_attn_shared_prefix.restype = ctypes.c_int
    lib.paged_extend_attn_workspace_size.argtypes = [I32, I32, I32, I32, I32, I32,
                                                     ctypes.POINTER(SZ)]
    lib.paged_extend_attn_workspace_size.restype = ctypes.c_int
    lib.paged_extend_attn.argtypes = [ctypes.POINTER(_Pool), P, I32, P, P, P, P, I32, I32, I32,
                                      I32, I32, F, I32, P, SZ, P, P]
    lib.paged_extend_attn.restype = ctypes.c_int
    lib.kvq_decode_step_workspace_size.argtypes = [I32, I32, I32, I32, I32, I32,
                                                   ctypes.POINTER(SZ)]
    lib.kvq_decode_step_workspace_size.restype = ctypes.c_int
    lib.kvq_decode_step.argtypes = [ctypes.POINTER(_Pool), P, I32, I32, P, P, I32, P, I32, P, P,
                                    P, I64, P, I32, P, I32, I32, F, I32, P, SZ, P, P]
    lib.kvq_decode_step.restype = ctypes.c_int
    lib.kvq_decode_step_fused.argtypes = [I32, I64]
    lib.kvq_decode_step_fused.restype = I32
    lib.kvq_selftest_step_barrier.argtypes = [P, I32, I32, P, P]
    lib.kvq_selftest_step_barrier.restype = ctypes.c_int
    lib.kvq_copy_blocks.argtypes = [ctypes.POINTER(_Pool), ctypes.POINTER(_Pool), P, P, I64, P, P]
    lib.kvq_copy_blocks.restype = ctypes.c_int
    lib.kvq_check_error.argtypes = [P, ctypes.POINTER(ctypes.c_uint32), P]
    lib.kvq_check_error.restype = ctypes.c_int
    lib.kvq_status_string.argtypes = [ctypes.c_int]
    lib.kvq_status_string.restype = ctypes.c_char_p
    lib.kvq_version.argtypes = []
    lib.kvq_version.restype = I32
    _lib = lib
    return lib


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    h = getattr(stream, "cuda_stream", stream)
    return h or None


def _check(status: int, where: str):
    if status != 0:
        raise KvqError(status, where)


@dataclass
class KVPool:
    """One layer's KV pool on the device (KVPool of "pymllm Runtime Design").

    k, v: uint8/int16 tensors [num_blocks, 16, kv_heads, row] where row is
    head_dim 16-bit elements (f16/bf16), head_dim bytes (int8) or head_dim/2
    bytes (int4); k_sz, v_sz: int32 [num_blocks, kv_heads, 16] holding fp16
    (scale, zero) pairs, or None for f16/bf16 pools.
    """

    k: object
    v: object
    k_sz: object
    v_sz: object
    num_blocks: int
    kv_heads: int
    kv_dtype: str
    head_dim: int = HEAD_DIM

    @staticmethod
    def allocate(num_blocks: int, kv_heads: int, kv_dtype: str, device="cuda",
                 head_dim: int = HEAD_DIM, pinned: bool = False) -> "KVPool":
        """Zero-filled pool tensors (allocation is the caller's side of the ABI).
        pinned: a host pool in page-locked memory the GPU addresses directly
        (the swap target of kvq_copy_blocks)."""
        import torch
        row = {"f16": 2 * head_dim, "bf16": 2 * head_dim, "int8": head_dim,
               "int4": head_dim // 2}[kv_dtype]
        shape = (num_blocks, BLOCK_SIZE, kv_heads, row)
        kw = dict(device="cpu", pin_memory=True) if pinned else dict(device=device)
        k = torch.zeros(shape, dtype=torch.uint8, **kw)
        v = torch.zeros(shape, dtype=torch.uint8, **kw)
        if kv_dtype in ("int8", "int4"):
            szs = (num_blocks, kv_heads, BLOCK_SIZE)
            k_sz = torch.zeros(szs, dtype=torch.int32, **kw)
            v_sz = torch.zeros(szs, dtype=torch.int32, **kw)
        else:
            k_sz = v_sz = None
        return KVPool(k, v, k_sz, v_sz, num_blocks, kv_heads, kv_dtype, head_dim)

    def c_struct(self) -> _Pool:
        return _Pool(_ptr(self.k), _ptr(self.v), _ptr(self.k_sz), _ptr(self.v_sz),
                     self.num_blocks, BLOCK_SIZE, self.kv_heads, self.head_dim,
                     DTYPE_CODES[self.kv_dtype])

    def nbytes(self) -> int:
        n = self.k.numel() + self.v.numel()
        if self.k_sz is not None:
            n += 4 * (self.k_sz.numel() + self.v_sz.numel())
        return n


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return KVQ_F16
    if t.dtype == torch.bfloat16:
        return KVQ_BF16
    raise TypeError(f"expected float16 or bfloat16 tensor, got {t.dtype}")


def kv_store_quant(pool: KVPool, k_new, v_new, slot_mapping, dev_err=None, stream=None):
    """Store new K/V rows [N, Hkv, D] at slot_mapping (int64 [N]); see kvq.h."""
    lib = load()
    ps = pool.c_struct()
    st = lib.kv_store_quant(ctypes.byref(ps), _ptr(k_new), _ptr(v_new), _dtype_code(k_new),
                            _ptr(slot_mapping), int(slot_mapping.numel()), _ptr(dev_err),
                            _stream(stream))
    _check(st, "kv_store_quant")


def kvq_block_tables_from_req_to_token(req_to_token, req_pool_indices, seq_lens, block_tables,
                                       dev_err=None, stream=None):
    """Fill block_tables [B, max_blocks] (int32) from ReqToTokenPool rows; see kvq.h."""
    lib = load()
    st = lib.kvq_block_tables_from_req_to_token(
        _ptr(req_to_token), int(req_to_token.shape[0]), int(req_to_token.shape[1]),
        _ptr(req_pool_indices), _ptr(seq_lens), int(seq_lens.numel()),
        int(block_tables.shape[1]), _ptr(block_tables), _ptr(dev_err), _stream(stream))
    _check(st, "kvq_block_tables_from_req_to_token")


def paged_decode_attn_plan(batch, q_heads, kv_heads, max_seq_len, num_splits=0, num_sms=0,
                           head_dim=HEAD_DIM) -> dict:
    """Host-side launch plan (no device access when num_sms > 0)."""
    lib = load()
    p = _Plan()
    st = lib.paged_decode_attn_plan(batch, q_heads, kv_heads, head_dim, max_seq_len, num_splits,
                                    num_sms, ctypes.byref(p))
    _check(st, "paged_decode_attn_plan")
    return {f: getattr(p, f) for f, _ in _Plan._fields_}


def paged_decode_attn_workspace_size(batch, q_heads, kv_heads, max_seq_len, num_splits=0,
                                     head_dim=HEAD_DIM) -> int:
    return int(load().paged_decode_attn_workspace_size(batch, q_heads, kv_heads, head_dim,
                                                       max_seq_len, num_splits))


def paged_decode_attn(pool: KVPool, q, out, block_tables, seq_lens, max_seq_len, sm_scale,
                      num_splits=0, workspace=None, dev_err=None, stream=None):
    """out[b, h] = softmax(sm_scale q[b, h] . K_b) V_b over the paged pool; see kvq.h."""
    lib = load()
    ps = pool.c_struct()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.paged_decode_attn(ctypes.byref(ps), _ptr(q), _dtype_code(q), _ptr(out),
                               _ptr(block_tables), int(block_tables.shape[1]), _ptr(seq_lens),
                               int(q.shape[0]), int(q.shape[1]), int(max_seq_len),
                               float(sm_scale), int(num_splits), _ptr(workspace), ws_bytes,
                               _ptr(dev_err), _stream(stream))
    _check(st, "paged_decode_attn")


def paged_decode_attn_noalloc(pool: KVPool, q, out, block_tables, seq_lens, max_seq_len,
                              sm_scale, num_splits=0, dev_err=None, stream=None):
    """paged_decode_attn without a caller workspace, for callers that cannot
    allocate device memory: the scratch is a fixed array inside libkvq
    (shared by all calls; overlapping calls race). See kvq.h."""
    lib = load()
    ps = pool.c_struct()
    st = lib.paged_decode_attn_noalloc(ctypes.byref(ps), _ptr(q), _dtype_code(q), _ptr(out),
                                       _ptr(block_tables), int(block_tables.shape[1]),
                                       _ptr(seq_lens), int(q.shape[0]), int(q.shape[1]),
                                       int(max_seq_len), float(sm_scale), int(num_splits),
                                       _ptr(dev_err), _stream(stream))
    _check(st, "paged_decode_attn_noalloc")


def kvq_decode_step_workspace_size(batch, q_heads, kv_heads, max_seq_len, num_splits=0,
                                   head_dim=HEAD_DIM) -> int:
    n = ctypes.c_size_t(0)
    st = load().kvq_decode_step_workspace_size(batch, q_heads, kv_heads, head_dim, max_seq_len,
                                               num_splits, ctypes.byref(n))
    _check(st, "kvq_decode_step_workspace_size")
    return int(n.value)


def kvq_decode_step_fused(batch: int, num_tokens: int) -> bool:
    """Whether kvq_decode_step runs as one launch for this many requests and
    stored tokens (else as four kernels); see kvq.h."""
    return bool(load().kvq_decode_step_fused(int(batch), int(num_tokens)))


def kvq_decode_step(pool: KVPool, req_to_token, req_pool_indices, seq_lens, block_tables, k_new,
                    v_new, slot_mapping, q, out, max_seq_len, sm_scale, num_splits=0,
                    workspace=None, dev_err=None, stream=None):
    """One decode step in one launch: block_tables [B, max_blocks] from the
    ReqToTokenPool rows, the store of k_new/v_new [N, Hkv, D] (q's dtype) at
    slot_mapping, then out[b, h] = attention of q[b, h] over the pool; see
    kvq.h."""
    if k_new.dtype != q.dtype or v_new.dtype != q.dtype or out.dtype != q.dtype:
        raise ValueError("kvq_decode_step: k_new, v_new and out must have q's dtype")
    lib = load()
    ps = pool.c_struct()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.kvq_decode_step(
        ctypes.byref(ps), _ptr(req_to_token), int(req_to_token.shape[0]),
        int(req_to_token.shape[1]), _ptr(req_pool_indices), _ptr(seq_lens),
        int(seq_lens.numel()), _ptr(block_tables), int(block_tables.shape[1]), _ptr(k_new),
        _ptr(v_new), _ptr(slot_mapping), int(slot_mapping.numel()), _ptr(q), _dtype_code(q),
        _ptr(out), int(q.shape[1]), int(max_seq_len), float(sm_scale), int(num_splits),
        _ptr(workspace), ws_bytes, _ptr(dev_err), _stream(stream))
    _check(st, "kvq_decode_step")


def paged_decode_attn_shared_prefix_workspace_size(batch, q_heads, kv_heads, max_seq_len,
                                                   max_shared_blocks, num_splits=0,
                                                   head_dim=HEAD_DIM) -> int:
    n = ctypes.c_size_t(0)
    st = load().paged_decode_attn_shared_prefix_workspace_size(
        batch, q_heads, kv_heads, head_dim, max_seq_len, num_splits, max_shared_blocks,
        ctypes.byref(n))
    _check(st, "paged_decode_attn_shared_prefix_workspace_size")
    return int(n.value)


@dataclass
class SharedPrefixGroups:
    """Requests that share leading blocks, as paged_decode_attn_shared_prefix
    takes them: group G's members are members[offsets[G]:offsets[G + 1]] and
    share their first shared_blocks[G] blocks (device int32 tensors)."""

    offsets: object
    members: object
    shared_blocks: object
    max_shared_blocks: int

    @property
    def num_groups(self) -> int:
        return int(self.shared_blocks.numel())

    @property
    def num_members(self) -> int:
        return int(self.members.numel())

    @classmethod
    def from_lists(cls, groups, device="cuda"):
        """groups: iterable of (member request indices, shared block count)."""
        import torch
        offsets, members, shared = [0], [], []
        for mem, sb in groups:
            members.extend(int(b) for b in mem)
            offsets.append(len(members))
            shared.append(int(sb))

        def t(x):
            return torch.tensor(x, dtype=torch.int32, device=device)

        return cls(t(offsets), t(members), t(shared), max(shared, default=0))

    @classmethod
    def detect(cls, block_tables, seq_lens, min_members=2, min_shared_blocks=1, device="cuda"):
        """Host-side grouping of a batch by common leading blocks (numpy
        arrays): requests with the same first block form a candidate group;
        its shared count s is chosen to maximise (members sharing s blocks)
        x s, and members sharing fewer stay outside (decoded on their own).
        Only full blocks are shared (16 s <= length)."""
        import numpy as np
        bt = np.asarray(block_tables)
        lens = np.asarray(seq_lens)
        by_first = {}
        for b in range(bt.shape[0]):
            if int(lens[b]) // 16 >= 1:
                by_first.setdefault(int(bt[b, 0]), []).append(b)
        groups = []
        for cand in by_first.values():
            if len(cand) < min_members:
                continue
            lead = cand[0]
            lcp = {}
            for b in cand:
                n = min(int(lens[b]) // 16, int(lens[lead]) // 16)
                eq = bt[b, :n] == bt[lead, :n]
                lcp[b] = n if eq.all() else int(np.argmin(eq))
            best, best_s = 0, 0
            for s_ in sorted(set(lcp.values())):
                if s_ < min_shared_blocks:
                    continue
                k = sum(1 for v in lcp.values() if v >= s_)
                if k >= min_members and k * s_ > best:
                    best, best_s = k * s_, s_
            if best_s > 0:
                groups.append(([b for b in cand if lcp[b] >= best_s], best_s))
        return cls.from_lists(groups, device=device)


def paged_decode_attn_shared_prefix(pool: KVPool, q, out, block_tables, seq_lens, max_seq_len,
                                    sm_scale, groups: SharedPrefixGroups, num_splits=0,
                                    workspace=None, dev_err=None, stream=None):
    """paged_decode_attn computed as a cascade over shared leading blocks; see kvq.h."""
    lib = load()
    ps = pool.c_struct()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.paged_decode_attn_shared_prefix(
        ctypes.byref(ps), _ptr(q), _dtype_code(q), _ptr(out), _ptr(block_tables),
        int(block_tables.shape[1]), _ptr(seq_lens), int(q.shape[0]), int(q.shape[1]),
        int(max_seq_len), float(sm_scale), _ptr(groups.offsets),
        _ptr(groups.members) if groups.num_members else None, _ptr(groups.shared_blocks),
        groups.num_groups, groups.num_members, int(groups.max_shared_blocks), int(num_splits),
        _ptr(workspace), ws_bytes, _ptr(dev_err), _stream(stream))
    _check(st, "paged_decode_attn_shared_prefix")


def paged_extend_attn_workspace_size(batch, total_q, q_heads, kv_heads, max_kv_len,
                                     head_dim=HEAD_DIM) -> int:
    n = ctypes.c_size_t(0)
    st = load().paged_extend_attn_workspace_size(batch, total_q, q_heads, kv_heads, head_dim,
                                                 max_kv_len, ctypes.byref(n))
    _check(st, "paged_extend_attn_workspace_size")
    return int(n.value)


EXTEND_VARIANTS = {"auto": 0, "mma_sync": 1, "tcgen05": 2}


def paged_extend_attn(pool: KVPool, q, out, qo_indptr, kv_lens, block_tables, max_kv_len,
                      sm_scale, workspace=None, dev_err=None, stream=None, variant="auto"):
    """Extend (chunked prefill) attention: q rows qo_indptr[b]..qo_indptr[b+1]-1
    are the last tokens of request b and attend causally; variant: "auto",
    "mma_sync" or "tcgen05" (see kvq.h)."""
    lib = load()
    ps = pool.c_struct()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.paged_extend_attn(ctypes.byref(ps), _ptr(q), _dtype_code(q), _ptr(out),
                               _ptr(qo_indptr), _ptr(kv_lens), _ptr(block_tables),
                               int(block_tables.shape[1]), int(kv_lens.numel()),
                               int(q.shape[0]), int(q.shape[1]), int(max_kv_len),
                               float(sm_scale), EXTEND_VARIANTS[variant], _ptr(workspace),
                               ws_bytes, _ptr(dev_err), _stream(stream))
    _check(st, "paged_extend_attn")


def kvq_copy_blocks(src: KVPool, dst: KVPool, src_ids, dst_ids, dev_err=None, stream=None):
    """Copy blocks src_ids[i] of src to dst_ids[i] of dst (int32 tensors the GPU
    can address); either pool may be in pinned host memory. See kvq.h."""
    lib = load()
    sp, dp = src.c_struct(), dst.c_struct()
    n = int(src_ids.numel())
    if int(dst_ids.numel()) != n:
        raise ValueError("src_ids and dst_ids differ in length")
    st = lib.kvq_copy_blocks(ctypes.byref(sp), ctypes.byref(dp), _ptr(src_ids), _ptr(dst_ids), n,
                             _ptr(dev_err), _stream(stream))
    _check(st, "kvq_copy_blocks")


def kvq_check_error(dev_err, stream=None) -> int:
    """Synchronize, read and clear the device error word; returns its bits."""
    lib = load()
    bits = ctypes.c_uint32(0)
    st = lib.kvq_check_error(_ptr(dev_err), ctypes.byref(bits), _stream(stream))
    if st not in (0, 4):
        _check(st, "kvq_check_error")
    return int(bits.value)


def kvq_selftest_step_barrier(counter, dev_err, grid_ctas=0, limit_us=5000, stream=None):
    """The fused step's bounded grid barrier made to wait for one CTA more
    than the grid has (a self-test of its timeout); see kvq.h."""
    lib = load()
    st = lib.kvq_selftest_step_barrier(_ptr(counter), int(grid_ctas), int(limit_us),
                                       _ptr(dev_err), _stream(stream))
    _check(st, "kvq_selftest_step_barrier")


def kvq_status_string(status: int) -> str:
    return load().kvq_status_string(status).decode()


def kvq_version() -> int:
    return int(load().kvq_version())


class DecodeStep:
    """One decode step of a layer through the C ABI: block tables, store, attention.

    Holds the per-step device buffers (block tables, workspace, error word) so
    the call itself allocates nothing. fused=True runs the step as the one
    cooperative launch of kvq_decode_step; otherwise as its three calls.
    """

    def __init__(self, pool: KVPool, batch: int, q_heads: int, max_blocks_per_seq: int,
                 max_seq_len: int, q_dtype, num_splits: int = 0, device="cuda",
                 fused: bool = False):
        import torch
        self.pool = pool
        self.batch = batch
        self.q_heads = q_heads
        self.max_seq_len = max_seq_len
        self.num_splits = num_splits
        self.fused = fused
        self.block_tables = torch.empty((batch, max_blocks_per_seq), dtype=torch.int32,
                                        device=device)
        ws = paged_decode_attn_workspace_size(batch, q_heads, pool.kv_heads, max_seq_len,
                                              num_splits)
        if fused:
            ws = max(ws, kvq_decode_step_workspace_size(batch, q_heads, pool.kv_heads,
                                                        max_seq_len, num_splits))
        self.workspace = torch.empty(max(ws, 16), dtype=torch.uint8, device=device)
        self.dev_err = torch.zeros(1, dtype=torch.int32, device=device)
        self.out = torch.empty((batch, q_heads, pool.head_dim), dtype=q_dtype, device=device)

    def __call__(self, req_to_token, req_pool_indices, seq_lens, q, k_new, v_new, slot_mapping,
                 sm_scale, stream=None):
        if self.fused:
            kvq_decode_step(self.pool, req_to_token, req_pool_indices, seq_lens,
                            self.block_tables, k_new, v_new, slot_mapping, q, self.out,
                            self.max_seq_len, sm_scale, self.num_splits, self.workspace,
                            self.dev_err, stream)
            return self.out
        kvq_block_tables_from_req_to_token(req_to_token, req_pool_indices, seq_lens,
                                           self.block_tables, self.dev_err, stream)
        kv_store_quant(self.pool, k_new, v_new, slot_mapping, self.dev_err, stream)
        paged_decode_attn(self.pool, q, self.out, self.block_tables, seq_lens, self.max_seq_len,
                          sm_scale, self.num_splits, self.workspace, self.dev_err, stream)
        return self.out
