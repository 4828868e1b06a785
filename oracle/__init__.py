"""CPU oracle for the paged, quantized KV store and paged decode attention.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg import this package. The product path
(``paged_quantized_kv_store_gb300``) never imports it and shares no code with
it. The arithmetic lives in ``kvq_oracle.cpp`` (plain single-threaded C++,
IEEE fp32 quantizer, fp64 attention); this file only marshals numpy arrays.

What it computes, and the passages it follows:

* ``quantize_rows`` -- per-token, per-head asymmetric min/max quantization to
  INT8/INT4 with fp16 scale and zero (LMDeploy article on devpress.csdn.net,
  §2.4 "KV Cache 在线量化").
* ``kv_store`` -- scatter of new K/V rows into pool slots given by a slot
  mapping ("pymllm Runtime Design", section "KV cache 与 prefix cache":
  KVPool written by store_cache; LMDeploy article §2.2 for the
  [num_blocks, block_size, kv_heads, head_dim] layout).
* ``block_tables`` -- per-request tables of physical block ids from
  ReqToTokenPool rows ("pymllm Runtime Design", same section; LMDeploy
  article §2.2, block size 16).
* ``paged_decode`` / ``decode_one`` -- single-token attention for a batch of
  requests through their block tables (LMDeploy article §3.2 item 3, indirect
  buffer pointers; §4.2, the separate decoding kernel), evaluated in fp64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "kvq_oracle.cpp")
LIB_PATH = os.path.join(HERE, "libkvq_oracle.so")

DTYPES = {"f16": 0, "bf16": 1, "int4": 4, "int8": 8}
BLOCK_SIZE = 16

_lib = None

_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_int = ctypes.c_int
_dbl = ctypes.c_double


def build(force: bool = False) -> str:
    """Compile the oracle (g++ -O2 -ffp-contract=off, no fast-math)."""
    if force or not os.path.exists(LIB_PATH) or os.path.getmtime(LIB_PATH) < os.path.getmtime(SRC):
        tmp = LIB_PATH + ".tmp%d" % os.getpid()
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-ffp-contract=off",
                               "-fno-fast-math", "-shared", "-fPIC", "-o", tmp, SRC])
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(LIB_PATH)
        sig = {
            "oracle_f16_to_f32": ([ctypes.c_uint16], ctypes.c_float),
            "oracle_f32_to_f16": ([ctypes.c_float], ctypes.c_uint16),
            "oracle_bf16_to_f32": ([ctypes.c_uint16], ctypes.c_float),
            "oracle_f32_to_f16_array": ([_p, _p, _i64], None),
            "oracle_f16_to_f32_array": ([_p, _p, _i64], None),
            "oracle_quantize_row": ([_p, _int, _int, _p, _p, _p], None),
            "oracle_quantize_rows": ([_p, _i64, _int, _int, _p, _p, _p], None),
            "oracle_dequant": ([_int, ctypes.c_uint16, ctypes.c_uint16], _dbl),
            "oracle_kv_store": ([_p, _p, _p, _p, _i64, _int, _int, _int, _p, _p, _int, _p, _i64],
                                _i64),
            "oracle_block_tables": ([_p, _i32, _i32, _p, _p, _i32, _i32, _p], _int),
            "oracle_decode_one": ([_p, _p, _p, _p, _i64, _int, _int, _int, _p, _int, _p, _i32,
                                   _i32, _dbl, _p, _p], _int),
            "oracle_paged_decode": ([_p, _p, _p, _p, _i64, _int, _int, _int, _p, _int, _p, _i32,
                                     _p, _i32, _i32, _dbl, _p], _int),
            "oracle_copy_blocks": ([_p, _p, _p, _p, _i64, _p, _p, _p, _p, _i64, _int, _int,
                                    _int, _p, _p, _i64], _i64),
            "oracle_paged_extend": ([_p, _p, _p, _p, _i64, _int, _int, _int, _p, _int, _p, _p,
                                     _i32, _p, _i32, _i32, _dbl, _p], _int),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


# ---- conversions -----------------------------------------------------------

def f32_to_f16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_f32_to_f16_array(_ptr(x), _ptr(out), x.size)
    return out


def f16_to_f32(h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float32)
    _load().oracle_f16_to_f32_array(_ptr(h), _ptr(out), h.size)
    return out


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32)


def to_f32(bits: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_to_f32(bits) if dtype == "bf16" else f16_to_f32(bits)


# ---- quantizer -------------------------------------------------------------

def quantize_rows(x: np.ndarray, bits: int):
    """x float32 [..., n] -> (codes uint8 [..., n], scale uint16 [...], zero uint16 [...])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    n = x.shape[-1]
    rows = x.size // n
    codes = np.empty(x.shape, dtype=np.uint8)
    sb = np.empty(x.shape[:-1], dtype=np.uint16)
    zb = np.empty(x.shape[:-1], dtype=np.uint16)
    _load().oracle_quantize_rows(_ptr(x), rows, n, bits, _ptr(codes), _ptr(sb), _ptr(zb))
    return codes, sb, zb


def dequant(code: int, scale_bits: int, zero_bits: int) -> float:
    return _load().oracle_dequant(int(code), int(scale_bits), int(zero_bits))


# ---- pool ------------------------------------------------------------------

class Pool:
    """Host copy of one layer's KV pool, laid out like the device pool.

    k, v: uint8 [num_blocks, 16, Hkv, row_bytes]; k_sz, v_sz: uint16
    [num_blocks, Hkv, 16, 2] (scale, zero) or None for fp16/bf16 pools.
    """

    def __init__(self, num_blocks: int, kv_heads: int, head_dim: int, kv_dtype: str):
        self.num_blocks = int(num_blocks)
        self.kv_heads = kv_heads
        self.head_dim = head_dim
        self.kv_dtype = kv_dtype
        row = {"f16": 2 * head_dim, "bf16": 2 * head_dim, "int8": head_dim,
               "int4": head_dim // 2}[kv_dtype]
        shape = (self.num_blocks, BLOCK_SIZE, kv_heads, row)
        self.k = np.zeros(shape, dtype=np.uint8)
        self.v = np.zeros(shape, dtype=np.uint8)
        if kv_dtype in ("int8", "int4"):
            self.k_sz = np.zeros((self.num_blocks, kv_heads, BLOCK_SIZE, 2), dtype=np.uint16)
            self.v_sz = np.zeros((self.num_blocks, kv_heads, BLOCK_SIZE, 2), dtype=np.uint16)
        else:
            self.k_sz = None
            self.v_sz = None

    def _args(self):
        return (_ptr(self.k), _ptr(self.v), _ptr(self.k_sz), _ptr(self.v_sz), self.num_blocks,
                self.kv_heads, self.head_dim, DTYPES[self.kv_dtype])


def kv_store(pool: Pool, k_new: np.ndarray, v_new: np.ndarray, in_dtype: str,
             slot_mapping: np.ndarray) -> int:
    """Store rows k_new/v_new (uint16 [N, Hkv, D]) at slot_mapping (int64 [N]).

    Returns the number of tokens skipped because their slot is past the pool.
    """
    k_new = np.ascontiguousarray(k_new, dtype=np.uint16)
    v_new = np.ascontiguousarray(v_new, dtype=np.uint16)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    return _load().oracle_kv_store(*pool._args(), _ptr(k_new), _ptr(v_new), DTYPES[in_dtype],
                                   _ptr(sm), sm.size)


def block_tables(req_to_token: np.ndarray, req_pool_indices: np.ndarray, seq_lens: np.ndarray,
                 max_blocks_per_seq: int):
    """(block_tables int32 [B, max_blocks_per_seq], error bit mask)."""
    r2t = np.ascontiguousarray(req_to_token, dtype=np.int32)
    rpi = np.ascontiguousarray(req_pool_indices, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    out = np.empty((sl.size, max_blocks_per_seq), dtype=np.int32)
    err = _load().oracle_block_tables(_ptr(r2t), r2t.shape[0], r2t.shape[1], _ptr(rpi), _ptr(sl),
                                      sl.size, max_blocks_per_seq, _ptr(out))
    return out, err


def paged_decode(pool: Pool, q: np.ndarray, q_dtype: str, block_tables_: np.ndarray,
                 seq_lens: np.ndarray, sm_scale: float) -> np.ndarray:
    """fp64 attention output [B, Hq, D] for q (uint16 [B, Hq, D])."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    bt = np.ascontiguousarray(block_tables_, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, Hq, D = q.shape
    out = np.empty((B, Hq, D), dtype=np.float64)
    rc = _load().oracle_paged_decode(*pool._args(), _ptr(q), DTYPES[q_dtype], _ptr(bt),
                                     bt.shape[1], _ptr(sl), B, Hq, sm_scale, _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_paged_decode failed ({rc})")
    return out


def decode_one(pool: Pool, q_row: np.ndarray, q_dtype: str, bt_row: np.ndarray, seq_len: int,
               h_kv: int, sm_scale: float):
    """(out fp64 [D], softmax weights fp64 [seq_len]) for one (request, q head)."""
    q_row = np.ascontiguousarray(q_row, dtype=np.uint16)
    bt = np.ascontiguousarray(bt_row, dtype=np.int32)
    out = np.empty(pool.head_dim, dtype=np.float64)
    probs = np.empty(max(1, seq_len), dtype=np.float64)
    rc = _load().oracle_decode_one(*pool._args(), _ptr(q_row), DTYPES[q_dtype], _ptr(bt),
                                   int(seq_len), int(h_kv), sm_scale, _ptr(out), _ptr(probs))
    if rc != 0:
        raise ValueError(f"oracle_decode_one failed ({rc})")
    return out, probs[:seq_len]


def paged_extend(pool: Pool, q: np.ndarray, q_dtype: str, qo_indptr: np.ndarray,
                 block_tables_: np.ndarray, kv_lens: np.ndarray, sm_scale: float) -> np.ndarray:
    """fp64 extend (chunked prefill) attention [total_q, Hq, D]: chunk query i of
    request b sits at position kv_lens[b] - C_b + i and attends positions 0 ..
    that position through the block table ("pymllm Runtime Design", forward
    stage, extend; LMDeploy article §2.3, prefills split into chunks)."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    qi = np.ascontiguousarray(qo_indptr, dtype=np.int32)
    bt = np.ascontiguousarray(block_tables_, dtype=np.int32)
    kl = np.ascontiguousarray(kv_lens, dtype=np.int32)
    T, Hq, D = q.shape
    assert qi.size == kl.size + 1 and qi[-1] == T
    out = np.empty((T, Hq, D), dtype=np.float64)
    rc = _load().oracle_paged_extend(*pool._args(), _ptr(q), DTYPES[q_dtype], _ptr(qi), _ptr(bt),
                                     bt.shape[1], _ptr(kl), kl.size, Hq, sm_scale, _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_paged_extend failed ({rc})")
    return out


def copy_blocks(src: Pool, dst: Pool, src_ids: np.ndarray, dst_ids: np.ndarray) -> int:
    """Copy whole blocks src_ids[i] of src to dst_ids[i] of dst, in order (LMDeploy
    article §4.4, the cache engine's swap map). Returns the pairs skipped for an
    id outside its pool."""
    assert (src.kv_dtype, src.kv_heads, src.head_dim) == (dst.kv_dtype, dst.kv_heads,
                                                          dst.head_dim)
    si = np.ascontiguousarray(src_ids, dtype=np.int32)
    di = np.ascontiguousarray(dst_ids, dtype=np.int32)
    assert si.size == di.size
    return int(_load().oracle_copy_blocks(
        _ptr(src.k), _ptr(src.v), _ptr(src.k_sz), _ptr(src.v_sz), src.num_blocks,
        _ptr(dst.k), _ptr(dst.v), _ptr(dst.k_sz), _ptr(dst.v_sz), dst.num_blocks,
        src.kv_heads, src.head_dim, DTYPES[src.kv_dtype], _ptr(si), _ptr(di), si.size))


def run_workload(wl, with_step: bool = True, pool: Optional[Pool] = None):
    """Build the pool for a synthetic workload and decode it.

    Returns (pool, out fp64 [B, Hq, D]). The step's own stores (prefill chunk
    and the new tokens) are applied when with_step is true.
    """
    if pool is None:
        pool = Pool(wl.num_blocks, wl.kv_heads, wl.head_dim, wl.kv_dtype)
        for slots, k, v in wl.setup_chunks():
            bad = kv_store(pool, k, v, wl.in_dtype, slots)
            assert bad == 0
    if with_step:
        slots, k, v = wl.step_store()
        assert kv_store(pool, k, v, wl.in_dtype, slots) == 0
    out = paged_decode(pool, wl.q(), wl.q_dtype, wl.block_tables, wl.seq_lens, wl.sm_scale)
    return pool, out
