"""Seeded synthetic workloads for the paged, quantized KV store.

Input generation only. This module builds the inputs that the CPU oracle and
the GPU path both consume: Q/K/V rows from the counter-based generator in
``kvqgen.c``, request lengths, block tables, ReqToTokenPool rows and slot
mappings. It holds none of the method's arithmetic (no quantization, no
attention). Every value is a pure function of (seed, stream, index), so any
row can be regenerated alone.

Workloads (one layer each, head_dim 128, block size 16):

* ``cfg1``  fp16 KV, 4 requests with lengths {17, 33, 64, 100}, 16 q / 8 kv
  heads, a 64-block pool whose tables are the first 16 ids of a random
  permutation.
* ``cfg2``  bf16 KV, 32 requests, lengths uniform in [512, 4096], 16 q / 8 kv
  heads, values scaled by 0.5, pool sized to fit exactly, ids permuted.
* ``cfg3``  INT8 KV, 128 requests of length 4096, 32 q / 32 kv heads, 1 % of
  the K and V channels (41 of 4096) scaled by 8.
* ``cfg4``  INT4 KV, 64 requests, lengths lognormal (median 2048, sigma 0.5)
  clipped to [128, 8192], 32 q / 8 kv heads; every request shares the full
  blocks of a common 1024-token prefix (64 physical blocks).
* ``cfg5``  INT8 KV, 32 q / 8 kv heads: a 4096-token prefill chunk stored
  into 256 blocks popped from a shuffled free list, plus 256 decode requests
  with lengths uniform in [256, 2048].

Lengths count the token stored in the step (its K/V row is the one at
position length - 1).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, field
from typing import Iterator, Optional

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkvqgen.so")

HEAD_DIM = 128
BLOCK_SIZE = 16
# positions per request in the generator's index space
_POS_STRIDE = 1 << 14

# generator streams
S_Q, S_K_CTX, S_V_CTX, S_K_PREFIX, S_V_PREFIX, S_K_CHUNK, S_V_CHUNK = 1, 2, 3, 4, 5, 6, 7
S_LENS, S_PERM, S_OUT_K, S_OUT_V, S_FREE, S_REQSLOT = 16, 17, 18, 19, 20, 21
S_Q_EXT = 22

_DT = {"f32": 0, "f16": 1, "bf16": 2}

_lib = None


def build(force: bool = False) -> str:
    """Compile the generator into a shared library next to its source."""
    src = os.path.join(HERE, "kvqgen.c")
    if force or not os.path.exists(LIB_PATH) or os.path.getmtime(LIB_PATH) < os.path.getmtime(src):
        tmp = LIB_PATH + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread",
                               "-o", tmp, src])
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(LIB_PATH)
        lib.kvqgen_normal.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                      ctypes.c_uint64, ctypes.c_double, ctypes.c_void_p,
                                      ctypes.c_uint64, ctypes.c_int, ctypes.c_void_p,
                                      ctypes.c_int]
        lib.kvqgen_normal.restype = ctypes.c_int
        lib.kvqgen_base.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        lib.kvqgen_base.restype = ctypes.c_uint64
        _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def normal(seed: int, stream: int, start: int, count: int, scale: float = 1.0,
           chan_scale: Optional[np.ndarray] = None, dtype: str = "f16",
           nthreads: Optional[int] = None) -> np.ndarray:
    """Elements start..start+count of a generator stream.

    Returns uint16 bit patterns for 'f16'/'bf16', float32 for 'f32'.
    """
    lib = _load()
    out = np.empty(count, dtype=np.float32 if dtype == "f32" else np.uint16)
    cs = None
    period = 0
    if chan_scale is not None:
        cs = np.ascontiguousarray(chan_scale, dtype=np.float32)
        period = cs.size
    rc = lib.kvqgen_normal(seed, stream, start, count, scale,
                           None if cs is None else cs.ctypes.data, period, _DT[dtype],
                           out.ctypes.data if count else None,
                           nthreads or default_threads())
    if rc != 0:
        raise ValueError("kvqgen_normal rejected its arguments")
    return out


def _splitmix64(x: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = x + np.uint64(0x9E3779B97F4A7C15)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        return z ^ (z >> np.uint64(31))


def uniform_u64(seed: int, stream: int, n: int) -> np.ndarray:
    """n 64-bit draws: splitmix64(base(seed, stream) + i)."""
    base = np.uint64(_load().kvqgen_base(seed, stream))
    with np.errstate(over="ignore"):
        return _splitmix64(base + np.arange(n, dtype=np.uint64))


def randint(seed: int, stream: int, n: int, lo: int, hi: int) -> np.ndarray:
    """n integers uniform in [lo, hi] (inclusive)."""
    span = np.uint64(hi - lo + 1)
    return (uniform_u64(seed, stream, n) % span).astype(np.int64) + lo


def permutation(seed: int, stream: int, n: int) -> np.ndarray:
    """Fisher-Yates shuffle of 0..n-1 driven by the generator."""
    u = uniform_u64(seed, stream, n)
    p = np.arange(n, dtype=np.int64)
    for i in range(n - 1, 0, -1):
        j = int(u[i] % np.uint64(i + 1))
        p[i], p[j] = p[j], p[i]
    return p


@dataclass
class Workload:
    """One layer's synthetic decode step (plus setup) for the KV store."""

    name: str
    kv_dtype: str            # 'f16' | 'bf16' | 'int8' | 'int4'
    in_dtype: str            # dtype of new K/V rows: 'f16' | 'bf16'
    q_dtype: str             # 'f16' | 'bf16'
    batch: int
    q_heads: int
    kv_heads: int
    seed: int
    seq_lens: np.ndarray                 # int32 [B], includes the new token
    num_blocks: int
    block_tables: np.ndarray             # int32 [B, max_blocks_per_seq], -1 padded
    req_to_token: np.ndarray             # int32 [num_req_slots, max_context_len]
    req_pool_indices: np.ndarray         # int32 [B]
    value_scale: float = 1.0
    k_chan_scale: Optional[np.ndarray] = None   # float32 [Hkv * D]
    v_chan_scale: Optional[np.ndarray] = None
    shared_tokens: Optional[np.ndarray] = None  # int32 [B]: leading positions from the prefix
    prefix_blocks: Optional[np.ndarray] = None  # int32 physical ids of the shared prefix
    chunk_slots: Optional[np.ndarray] = None    # int64 [n]: prefill chunk slots (cfg5)
    head_dim: int = HEAD_DIM
    block_size: int = BLOCK_SIZE
    description: str = ""

    # ---- shapes -----------------------------------------------------------
    @property
    def group(self) -> int:
        return self.q_heads // self.kv_heads

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.batch else 0

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def quantized(self) -> bool:
        return self.kv_dtype in ("int8", "int4")

    @property
    def gen_dtype(self) -> str:
        return self.in_dtype

    # ---- generator index space -------------------------------------------
    def _ctx_stream(self, which: str) -> int:
        return S_K_CTX if which == "k" else S_V_CTX

    def _prefix_stream(self, which: str) -> int:
        return S_K_PREFIX if which == "k" else S_V_PREFIX

    def _chan(self, which: str) -> Optional[np.ndarray]:
        return self.k_chan_scale if which == "k" else self.v_chan_scale

    def ctx_rows(self, which: str, b: int, p0: int, p1: int,
                 nthreads: Optional[int] = None) -> np.ndarray:
        """K or V of request b at positions p0..p1-1 as uint16 [n, Hkv, D]."""
        hd = self.kv_heads * self.head_dim
        out = np.empty((p1 - p0, hd), dtype=np.uint16)
        shared = int(self.shared_tokens[b]) if self.shared_tokens is not None else 0
        cs = self._chan(which)
        if p0 < shared:
            e = min(p1, shared)
            out[: e - p0] = normal(self.seed, self._prefix_stream(which), p0 * hd,
                                   (e - p0) * hd, self.value_scale, cs, self.gen_dtype,
                                   nthreads).reshape(e - p0, hd)
        s = max(p0, shared)
        if s < p1:
            start = (b * _POS_STRIDE + s) * hd
            out[s - p0:] = normal(self.seed, self._ctx_stream(which), start, (p1 - s) * hd,
                                  self.value_scale, cs, self.gen_dtype,
                                  nthreads).reshape(p1 - s, hd)
        return out.reshape(p1 - p0, self.kv_heads, self.head_dim)

    def q(self) -> np.ndarray:
        """Queries as uint16 [B, Hq, D] (dtype q_dtype)."""
        n = self.batch * self.q_heads * self.head_dim
        return normal(self.seed, S_Q, 0, n, self.value_scale, None,
                      self.q_dtype).reshape(self.batch, self.q_heads, self.head_dim)

    def slot(self, b: int, p: int) -> int:
        return int(self.block_tables[b, p // self.block_size]) * self.block_size + p % self.block_size

    def new_slots(self) -> np.ndarray:
        """Slot of each request's new token (position length - 1), int64 [B]."""
        return np.array([self.slot(b, int(self.seq_lens[b]) - 1) if self.seq_lens[b] > 0 else -1
                         for b in range(self.batch)], dtype=np.int64)

    def new_rows(self, which: str) -> np.ndarray:
        """K or V rows of each request's new token, uint16 [B, Hkv, D]."""
        out = np.zeros((self.batch, self.kv_heads, self.head_dim), dtype=np.uint16)
        for b in range(self.batch):
            L = int(self.seq_lens[b])
            if L > 0:
                out[b] = self.ctx_rows(which, b, L - 1, L)[0]
        return out

    def chunk_rows(self, which: str) -> np.ndarray:
        """Prefill-chunk K or V rows, uint16 [n, Hkv, D] (cfg5)."""
        n = 0 if self.chunk_slots is None else len(self.chunk_slots)
        hd = self.kv_heads * self.head_dim
        s = S_K_CHUNK if which == "k" else S_V_CHUNK
        return normal(self.seed, s, 0, n * hd, self.value_scale, self._chan(which),
                      self.gen_dtype).reshape(n, self.kv_heads, self.head_dim)

    def step_store(self):
        """Tokens stored inside the timed step: (slots int64, K rows, V rows).

        The prefill chunk (if any) comes first, then each request's new token.
        """
        slots = [self.new_slots()]
        ks = [self.new_rows("k")]
        vs = [self.new_rows("v")]
        if self.chunk_slots is not None:
            slots.insert(0, self.chunk_slots.astype(np.int64))
            ks.insert(0, self.chunk_rows("k"))
            vs.insert(0, self.chunk_rows("v"))
        return np.concatenate(slots), np.concatenate(ks), np.concatenate(vs)

    def setup_chunks(self, max_tokens: int = 1 << 16,
                     nthreads: Optional[int] = None) -> Iterator[tuple]:
        """Context stored before the step, in chunks of at most max_tokens.

        Yields (slots int64 [n], K uint16 [n, Hkv, D], V uint16 [n, Hkv, D]).
        Positions 0..length-2 of every request; shared prefix blocks once.
        """
        if self.prefix_blocks is not None and self.shared_tokens is not None:
            npfx = len(self.prefix_blocks) * self.block_size
            for p0 in range(0, npfx, max_tokens):
                p1 = min(npfx, p0 + max_tokens)
                pos = np.arange(p0, p1)
                slots = (self.prefix_blocks[pos // self.block_size].astype(np.int64)
                         * self.block_size + pos % self.block_size)
                # the prefix stream does not depend on the request: use request 0's view
                hd = self.kv_heads * self.head_dim
                k = normal(self.seed, S_K_PREFIX, p0 * hd, (p1 - p0) * hd, self.value_scale,
                           self.k_chan_scale, self.gen_dtype, nthreads)
                v = normal(self.seed, S_V_PREFIX, p0 * hd, (p1 - p0) * hd, self.value_scale,
                           self.v_chan_scale, self.gen_dtype, nthreads)
                yield (slots, k.reshape(-1, self.kv_heads, self.head_dim),
                       v.reshape(-1, self.kv_heads, self.head_dim))
        pend_s, pend_k, pend_v, pend_n = [], [], [], 0
        for b in range(self.batch):
            L = int(self.seq_lens[b])
            start = int(self.shared_tokens[b]) if self.shared_tokens is not None else 0
            p = start
            while p < L - 1:
                e = min(L - 1, p + max_tokens - pend_n)
                pos = np.arange(p, e)
                bt = self.block_tables[b]
                pend_s.append(bt[pos // self.block_size].astype(np.int64) * self.block_size
                              + pos % self.block_size)
                pend_k.append(self.ctx_rows("k", b, p, e, nthreads))
                pend_v.append(self.ctx_rows("v", b, p, e, nthreads))
                pend_n += e - p
                p = e
                if pend_n >= max_tokens:
                    yield (np.concatenate(pend_s), np.concatenate(pend_k), np.concatenate(pend_v))
                    pend_s, pend_k, pend_v, pend_n = [], [], [], 0
        if pend_n:
            yield (np.concatenate(pend_s), np.concatenate(pend_k), np.concatenate(pend_v))

    # ---- bytes --------------------------------------------------------------
    def kv_row_bytes(self) -> int:
        """Bytes of one (token, kv head) row of K (or V) in the pool."""
        return {"f16": 2 * self.head_dim, "bf16": 2 * self.head_dim,
                "int8": self.head_dim, "int4": self.head_dim // 2}[self.kv_dtype]

    def kv_token_bytes(self) -> int:
        """Pool bytes read per token for K+V and scale/zero, all kv heads."""
        sz = 4 if self.quantized else 0
        return 2 * self.kv_heads * (self.kv_row_bytes() + sz)


def _tables_from_ids(lens: np.ndarray, ids: np.ndarray, bs: int = BLOCK_SIZE):
    nblk = (lens + bs - 1) // bs
    mb = int(max(1, nblk.max()))
    bt = np.full((len(lens), mb), -1, dtype=np.int32)
    k = 0
    for b, n in enumerate(nblk):
        bt[b, :n] = ids[k:k + n]
        k += n
    return bt


def _req_to_token(bt: np.ndarray, lens: np.ndarray, seed: int, extra_slots: int = 3,
                  bs: int = BLOCK_SIZE):
    """ReqToTokenPool rows consistent with the block tables.

    Request b lives in request slot req_pool_indices[b] (a shuffled choice of
    B + extra_slots slots); unused entries hold -1.
    """
    B = len(lens)
    n_slots = B + extra_slots
    rpi = permutation(seed, S_REQSLOT, n_slots)[:B].astype(np.int32)
    max_ctx = int(max(bs, ((lens.max() + bs - 1) // bs) * bs)) if B else bs
    r2t = np.full((n_slots, max_ctx), -1, dtype=np.int32)
    for b in range(B):
        L = int(lens[b])
        pos = np.arange(L)
        r2t[rpi[b], :L] = bt[b, pos // bs] * bs + pos % bs
    return r2t, rpi


def _finish(name, kv_dtype, in_dtype, q_dtype, Hq, Hkv, seed, lens, num_blocks, bt, **kw):
    lens = np.asarray(lens, dtype=np.int32)
    r2t, rpi = _req_to_token(bt, lens, seed)
    return Workload(name=name, kv_dtype=kv_dtype, in_dtype=in_dtype, q_dtype=q_dtype,
                    batch=len(lens), q_heads=Hq, kv_heads=Hkv, seed=seed, seq_lens=lens,
                    num_blocks=int(num_blocks), block_tables=bt, req_to_token=r2t,
                    req_pool_indices=rpi, **kw)


def cfg1(seed: int = 0) -> Workload:
    lens = np.array([17, 33, 64, 100], dtype=np.int32)
    perm = permutation(seed, S_PERM, 64)
    bt = _tables_from_ids(lens, perm)
    return _finish("cfg1", "f16", "f16", "f16", 16, 8, seed, lens, 64, bt,
                   description="fp16 KV, 4 requests {17,33,64,100}, 16q/8kv, 64-block pool")


def cfg2(seed: int = 1, batch: int = 32, lo: int = 512, hi: int = 4096) -> Workload:
    lens = randint(seed, S_LENS, batch, lo, hi).astype(np.int32)
    nblk = (lens + BLOCK_SIZE - 1) // BLOCK_SIZE
    total = int(nblk.sum())
    perm = permutation(seed, S_PERM, total)
    bt = _tables_from_ids(lens, perm)
    return _finish("cfg2", "bf16", "bf16", "bf16", 16, 8, seed, lens, total, bt,
                   value_scale=0.5,
                   description=f"bf16 KV, {batch} requests U[{lo},{hi}], 16q/8kv, x0.5")


def _outliers(seed: int, stream: int, n_chan: int, frac: float = 0.01) -> np.ndarray:
    k = int(round(frac * n_chan))
    scale = np.ones(n_chan, dtype=np.float32)
    scale[permutation(seed, stream, n_chan)[:k]] = 8.0
    return scale


def cfg3(seed: int = 2, batch: int = 128, length: int = 4096, heads: int = 32) -> Workload:
    lens = np.full(batch, length, dtype=np.int32)
    nblk = (length + BLOCK_SIZE - 1) // BLOCK_SIZE
    total = batch * nblk
    perm = permutation(seed, S_PERM, total)
    bt = _tables_from_ids(lens, perm)
    nc = heads * HEAD_DIM
    return _finish("cfg3", "int8", "f16", "f16", heads, heads, seed, lens, total, bt,
                   k_chan_scale=_outliers(seed, S_OUT_K, nc),
                   v_chan_scale=_outliers(seed, S_OUT_V, nc),
                   description=f"INT8 KV, MHA {heads}/{heads}, {batch} requests x {length}, "
                               "1% channels x8")


def cfg4(seed: int = 3, batch: int = 64, median: int = 2048, sigma: float = 0.5,
         lo: int = 128, hi: int = 8192, prefix_blocks: int = 64) -> Workload:
    z = normal(seed, S_LENS, 0, batch, 1.0, None, "f32").astype(np.float64)
    lens = np.clip(np.rint(median * np.exp(sigma * z)), lo, hi).astype(np.int32)
    # request b shares k_b = min(prefix_blocks, (L_b - 1) // 16) full prefix
    # blocks; the block holding its newest token is always private
    k = np.minimum(prefix_blocks, (lens - 1) // BLOCK_SIZE).astype(np.int32)
    nblk = (lens + BLOCK_SIZE - 1) // BLOCK_SIZE
    n_private = int((nblk - k).sum())
    total = prefix_blocks + n_private
    perm = permutation(seed, S_PERM, total)
    pfx = perm[:prefix_blocks].astype(np.int32)
    mb = int(nblk.max())
    bt = np.full((batch, mb), -1, dtype=np.int32)
    c = prefix_blocks
    for b in range(batch):
        bt[b, :k[b]] = pfx[:k[b]]
        n = int(nblk[b] - k[b])
        bt[b, k[b]:nblk[b]] = perm[c:c + n]
        c += n
    return _finish("cfg4", "int4", "f16", "f16", 32, 8, seed, lens, total, bt,
                   shared_tokens=(k * BLOCK_SIZE).astype(np.int32), prefix_blocks=pfx,
                   description=f"INT4 KV, 32q/8kv, {batch} requests lognormal(median {median}, "
                               f"sigma {sigma}) in [{lo},{hi}], shared {prefix_blocks}-block prefix")


def cfg4_long_prefix(seed: int = 3, batch: int = 64) -> Workload:
    """cfg4's structure (INT4 KV, 32q/8kv, one shared prefix) with an
    8192-token (512-block) prefix that every request holds, lengths in
    [8208, 9216]: the prefix is most of each request's context, so a
    cascade that attends it once per group has most of the work to save."""
    return cfg4(seed=seed, batch=batch, median=8704, sigma=0.05, lo=8208, hi=9216,
                prefix_blocks=512)


def cfg5(seed: int = 4, batch: int = 256, lo: int = 256, hi: int = 2048,
         chunk: int = 4096, slack_blocks: int = 256) -> Workload:
    lens = randint(seed, S_LENS, batch, lo, hi).astype(np.int32)
    nblk = (lens + BLOCK_SIZE - 1) // BLOCK_SIZE
    chunk_blocks = (chunk + BLOCK_SIZE - 1) // BLOCK_SIZE
    total = int(nblk.sum()) + chunk_blocks + slack_blocks
    free = permutation(seed, S_FREE, total)       # shuffled free list
    bt = _tables_from_ids(lens, free)             # decode requests pop first
    used = int(nblk.sum())
    cblk = free[used:used + chunk_blocks]         # then the prefill chunk
    pos = np.arange(chunk)
    chunk_slots = cblk[pos // BLOCK_SIZE].astype(np.int64) * BLOCK_SIZE + pos % BLOCK_SIZE
    return _finish("cfg5", "int8", "f16", "f16", 32, 8, seed, lens, total, bt,
                   chunk_slots=chunk_slots,
                   description=f"INT8 KV, 32q/8kv, {chunk}-token prefill chunk + {batch} "
                               f"decode requests U[{lo},{hi}]")


def shared_prefix(name: str, kv_dtype: str, lens, q_heads: int, kv_heads: int,
                  prefix_blocks: int, seed: int = 11, in_dtype: str = "f16",
                  q_dtype: Optional[str] = None, extra_blocks: int = 3) -> Workload:
    """Small workload with cfg4's structure for any pool type and head counts:
    request b's first k_b = min(prefix_blocks, (L_b - 1) // 16) blocks are
    the common prefix's (same physical blocks, same rows); the rest are
    private random blocks."""
    lens = np.asarray(lens, dtype=np.int32)
    k = np.maximum(np.minimum(prefix_blocks, (lens - 1) // BLOCK_SIZE), 0).astype(np.int32)
    nblk = (lens + BLOCK_SIZE - 1) // BLOCK_SIZE
    total = prefix_blocks + int((nblk - k).sum()) + extra_blocks
    perm = permutation(seed, S_PERM, total)
    pfx = perm[:prefix_blocks].astype(np.int32)
    bt = np.full((len(lens), max(int(nblk.max()), 1)), -1, dtype=np.int32)
    c = prefix_blocks
    for b in range(len(lens)):
        bt[b, :k[b]] = pfx[:k[b]]
        n = int(nblk[b] - k[b])
        bt[b, k[b]:nblk[b]] = perm[c:c + n]
        c += n
    if q_dtype is None:
        q_dtype = kv_dtype if kv_dtype in ("f16", "bf16") else in_dtype
    if kv_dtype in ("f16", "bf16"):
        in_dtype = kv_dtype
    return _finish(name, kv_dtype, in_dtype, q_dtype, q_heads, kv_heads, seed, lens, total, bt,
                   shared_tokens=(k * BLOCK_SIZE).astype(np.int32), prefix_blocks=pfx,
                   description=f"{kv_dtype} KV, {q_heads}q/{kv_heads}kv, {len(lens)} requests, "
                               f"shared {prefix_blocks}-block prefix")


@dataclass
class ExtendWorkload:
    """Chunked-prefill (extend) attention input: the pool holds kv_lens[b]
    tokens of request b (its prefix, then its chunk, stored like a decode
    workload's context), and the last chunk_lens[b] of them have queries,
    packed as rows qo_indptr[b] .. qo_indptr[b + 1] - 1 of q_ext()."""

    wl: Workload
    chunk_lens: np.ndarray

    @property
    def qo_indptr(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.chunk_lens)]).astype(np.int32)

    @property
    def total_q(self) -> int:
        return int(self.chunk_lens.sum())

    @property
    def kv_lens(self) -> np.ndarray:
        return self.wl.seq_lens

    def q_ext(self) -> np.ndarray:
        """Queries as uint16 [total_q, Hq, D] (dtype q_dtype)."""
        w = self.wl
        n = self.total_q * w.q_heads * w.head_dim
        return normal(w.seed, S_Q_EXT, 0, n, w.value_scale, None,
                      w.q_dtype).reshape(self.total_q, w.q_heads, w.head_dim)


def extend(name: str, kv_dtype: str, kv_lens, chunk_lens, q_heads: int, kv_heads: int,
           seed: int = 31, in_dtype: str = "f16", q_dtype: Optional[str] = None,
           outliers: bool = False) -> ExtendWorkload:
    """Requests with kv_lens[b] tokens in the pool whose last chunk_lens[b]
    tokens are the chunk being prefilled (chunk_lens[b] == kv_lens[b]: a fresh
    prefill; < kv_lens[b]: an extend over a cached prefix)."""
    kv_lens = np.asarray(kv_lens, dtype=np.int32)
    chunk_lens = np.asarray(chunk_lens, dtype=np.int32)
    assert kv_lens.shape == chunk_lens.shape and (chunk_lens <= kv_lens).all()
    wl = custom(name, kv_dtype, kv_lens, q_heads, kv_heads, seed=seed, in_dtype=in_dtype,
                q_dtype=q_dtype, outliers=outliers)
    return ExtendWorkload(wl, chunk_lens)


def cfg5_prefill(seed: int = 4, chunk: int = 4096) -> ExtendWorkload:
    """The mixed step's prefill chunk on its own: one fresh 4096-token prompt
    chunk (max_prefill_token_num) over INT8 KV, GQA 32q/8kv, attended
    causally after it is stored."""
    return extend("cfg5_prefill", "int8", [chunk], [chunk], 32, 8, seed=seed)


def by_name(name: str, **kw) -> Workload:
    return {"cfg1": cfg1, "cfg2": cfg2, "cfg3": cfg3, "cfg4": cfg4, "cfg5": cfg5,
            "cfg4_long_prefix": cfg4_long_prefix}[name](**kw)


def custom(name: str, kv_dtype: str, lens, q_heads: int, kv_heads: int, seed: int = 7,
           in_dtype: str = "f16", q_dtype: Optional[str] = None, value_scale: float = 1.0,
           extra_blocks: int = 5, outliers: bool = False) -> Workload:
    """Small ad-hoc workload: random distinct blocks for each request.

    outliers: scale 1 % of the K and of the V channels by 8, as in cfg3.
    """
    lens = np.asarray(lens, dtype=np.int32)
    nblk = (lens + BLOCK_SIZE - 1) // BLOCK_SIZE
    total = int(nblk.sum()) + extra_blocks
    perm = permutation(seed, S_PERM, total)
    bt = _tables_from_ids(lens, perm)
    if q_dtype is None:
        q_dtype = kv_dtype if kv_dtype in ("f16", "bf16") else in_dtype
    if kv_dtype in ("f16", "bf16"):
        in_dtype = kv_dtype
    kw = {}
    if outliers:
        nc = kv_heads * HEAD_DIM
        kw = dict(k_chan_scale=_outliers(seed, S_OUT_K, nc), v_chan_scale=_outliers(seed, S_OUT_V, nc))
    return _finish(name, kv_dtype, in_dtype, q_dtype, q_heads, kv_heads, seed, lens, total, bt,
                   value_scale=value_scale, **kw)
