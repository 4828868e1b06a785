"""Runs a synthetic workload through the C ABI on the GPU (tests only).

Inputs come from ``synthetic`` (the same generator the oracle reads); every
compute step runs in libkvq through ``paged_quantized_kv_store_gb300``.
"""
from __future__ import annotations

import numpy as np
import torch

import paged_quantized_kv_store_gb300 as kvq

TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16}

# tolerance on attention outputs: an element passes if it is within ATOL of
# the oracle or within RTOL of the oracle's magnitude
ATOL = 2e-3
RTOL = 1e-2


def to_dev(bits: np.ndarray, dtype: str, device="cuda"):
    """uint16 bit patterns -> device tensor of the 16-bit float dtype."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(TORCH_DT[dtype]).to(device)


def i32(a, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def i64(a, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int64)).to(device)


def fill_pool(wl, pool=None, dev_err=None, max_tokens=1 << 16):
    """Allocate the pool and store the workload's setup context through the ABI."""
    if pool is None:
        pool = kvq.KVPool.allocate(wl.num_blocks, wl.kv_heads, wl.kv_dtype)
    for slots, k, v in wl.setup_chunks(max_tokens=max_tokens):
        kvq.kv_store_quant(pool, to_dev(k, wl.in_dtype), to_dev(v, wl.in_dtype), i64(slots),
                           dev_err)
    return pool


def run_step(wl, pool, num_splits=0, dev_err=None, block_tables=None):
    """The decode step: block tables, store of the step's tokens, attention."""
    if dev_err is None:
        dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if block_tables is None:
        bt = torch.empty((wl.batch, wl.max_blocks_per_seq), dtype=torch.int32, device="cuda")
        kvq.kvq_block_tables_from_req_to_token(i32(wl.req_to_token), i32(wl.req_pool_indices),
                                               i32(wl.seq_lens), bt, dev_err)
    else:
        bt = i32(block_tables)
    slots, k, v = wl.step_store()
    kvq.kv_store_quant(pool, to_dev(k, wl.in_dtype), to_dev(v, wl.in_dtype), i64(slots), dev_err)
    out = decode(wl, pool, bt, num_splits, dev_err)
    return out, bt, dev_err


def decode(wl, pool, bt, num_splits=0, dev_err=None, q=None, seq_lens=None, max_seq_len=None):
    q = to_dev(wl.q(), wl.q_dtype) if q is None else q
    sl = i32(wl.seq_lens) if seq_lens is None else seq_lens
    msl = wl.max_seq_len if max_seq_len is None else max_seq_len
    out = torch.empty_like(q)
    ws = kvq.paged_decode_attn_workspace_size(wl.batch, wl.q_heads, wl.kv_heads, msl, num_splits)
    workspace = torch.empty(max(ws, 16), dtype=torch.uint8, device="cuda")
    kvq.paged_decode_attn(pool, q, out, bt, sl, msl, wl.sm_scale, num_splits, workspace, dev_err)
    return out


def pool_to_host(pool):
    """Device pool -> dict of numpy arrays shaped like oracle.Pool's."""
    d = {"k": pool.k.cpu().numpy(), "v": pool.v.cpu().numpy()}
    if pool.k_sz is not None:
        d["k_sz"] = pool.k_sz.cpu().numpy().view(np.uint16).reshape(pool.k_sz.shape + (2,))
        d["v_sz"] = pool.v_sz.cpu().numpy().view(np.uint16).reshape(pool.v_sz.shape + (2,))
    return d


def out_to_f64(out):
    return out.float().cpu().numpy().astype(np.float64)


def assert_close(got: np.ndarray, ref: np.ndarray, atol=ATOL, rtol=RTOL):
    """Element-wise: |got - ref| <= atol or <= rtol |ref|. Returns the largest
    absolute and relative errors (both are reported on failure)."""
    err = np.abs(got - ref)
    rel = err / np.maximum(np.abs(ref), 1e-30)
    ok = (err <= atol) | (err <= rtol * np.abs(ref))
    if not ok.all():
        idx = np.unravel_index(np.argmax(np.where(ok, 0, err)), err.shape)
        raise AssertionError(
            f"{(~ok).sum()} of {ok.size} elements out of tolerance; worst at {idx}: "
            f"got {got[idx]!r} ref {ref[idx]!r}; max abs err {err.max():.3e}, "
            f"max rel err {rel.max():.3e}")
    return float(err.max()), float(rel.max())


def oracle_request(wl, b):
    """Oracle pool and fp64 output [Hq, D] for request b alone.

    The request's blocks are renumbered 0..n-1 in a compact pool (attention
    does not depend on physical ids); every position, the step's new token
    included, is stored through the oracle.
    """
    import oracle
    L = int(wl.seq_lens[b])
    nblk = max(1, (L + 15) // 16)
    pool = oracle.Pool(nblk, wl.kv_heads, wl.head_dim, wl.kv_dtype)
    if L > 0:
        k = wl.ctx_rows("k", b, 0, L)
        v = wl.ctx_rows("v", b, 0, L)
        oracle.kv_store(pool, k, v, wl.in_dtype, np.arange(L, dtype=np.int64))
    bt = np.arange(nblk, dtype=np.int32)[None]
    out = oracle.paged_decode(pool, wl.q()[b:b + 1], wl.q_dtype, bt,
                              np.array([L], np.int32), wl.sm_scale)
    return pool, out[0]


def gpu_request_rows(wl, pool, b):
    """Pool rows (and scale/zero pairs) of request b's positions, copied to the host."""
    L = int(wl.seq_lens[b])
    pos = np.arange(L)
    slots = wl.block_tables[b, pos // 16].astype(np.int64) * 16 + pos % 16
    idx = torch.from_numpy(slots).cuda()
    nb = pool.num_blocks
    res = {}
    for name in ("k", "v"):
        t = getattr(pool, name)
        res[name] = t.view(nb * 16, *t.shape[2:])[idx].cpu().numpy()
        sz = getattr(pool, name + "_sz")
        if sz is not None:
            blk = idx // 16
            off = idx % 16
            res[name + "_sz"] = sz[blk, :, off].cpu().numpy().view(np.uint16).reshape(L, -1, 2)
    return res


def oracle_request_rows(opool, L):
    res = {}
    for name in ("k", "v"):
        a = getattr(opool, name)
        res[name] = a.reshape(-1, *a.shape[2:])[:L]
        sz = getattr(opool, name + "_sz")
        if sz is not None:
            pos = np.arange(L)
            res[name + "_sz"] = sz[pos // 16, :, pos % 16]
    return res
