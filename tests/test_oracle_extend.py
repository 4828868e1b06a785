"""Pins for the oracle's extend (chunked prefill) attention.

"pymllm Runtime Design", forward stage (extend / prefill over the KV cache);
LMDeploy article §2.3 (a long prefill is split into chunks). Chunk query i of
request b sits at position kv_len - C + i and attends positions 0 .. itself.
The oracle is pinned to
* dense causal softmax attention (numpy, fp64) over the dequantized rows read
  out of the pool arrays by plain [block, offset, head] indexing,
* a chunk of one query being exactly the decode of that request,
* causality: rows past a query's position do not change its output,
* invariance, bit for bit, under a permutation of physical block ids.
"""
import numpy as np
import pytest

import oracle
import synthetic


def _rows(pool, wl, b, which):
    """Dequantized [L, Hkv, D] (fp64) of request b, read from the pool arrays."""
    L = int(wl.seq_lens[b])
    arr = pool.k if which == "k" else pool.v
    szs = pool.k_sz if which == "k" else pool.v_sz
    out = np.zeros((L, wl.kv_heads, wl.head_dim))
    for t in range(L):
        blk, off = int(wl.block_tables[b, t // 16]), t % 16
        row = arr[blk, off]
        if wl.kv_dtype in ("f16", "bf16"):
            out[t] = oracle.to_f32(row.view(np.uint16), wl.kv_dtype)
            continue
        if wl.kv_dtype == "int8":
            codes = row.astype(np.float64)
        else:
            codes = np.empty((wl.kv_heads, wl.head_dim))
            codes[:, 0::2] = row & 0xF
            codes[:, 1::2] = row >> 4
        S = oracle.f16_to_f32(szs[blk, :, off, 0]).astype(np.float64)
        Z = oracle.f16_to_f32(szs[blk, :, off, 1]).astype(np.float64)
        out[t] = codes * S[:, None] + Z[:, None]
    return out


def _dense_causal(q, K, V, sm_scale, group, first_pos):
    """q [C, Hq, D], K/V [L, Hkv, D] -> [C, Hq, D]: softmax(s q K^T + mask) V with
    query i allowed keys 0 .. first_pos + i."""
    C, Hq, _ = q.shape
    L = K.shape[0]
    out = np.zeros_like(q)
    for h in range(Hq):
        s = sm_scale * (q[:, h, :] @ K[:, h // group, :].T)       # [C, L]
        mask = np.arange(L)[None, :] > (first_pos + np.arange(C))[:, None]
        s = np.where(mask, -np.inf, s)
        w = np.exp(s - s.max(axis=1, keepdims=True))
        w /= w.sum(axis=1, keepdims=True)
        out[:, h, :] = w @ V[:, h // group, :]
    return out


def _run(ew):
    wl = ew.wl
    pool, _ = oracle.run_workload(wl)
    out = oracle.paged_extend(pool, ew.q_ext(), wl.q_dtype, ew.qo_indptr, wl.block_tables,
                              ew.kv_lens, wl.sm_scale)
    return pool, out


@pytest.mark.parametrize("kv_dtype,Hq,Hkv", [("int8", 8, 4), ("int4", 8, 2), ("f16", 4, 4),
                                             ("bf16", 6, 2)])
def test_extend_matches_dense_causal_attention(kv_dtype, Hq, Hkv):
    ew = synthetic.extend("e", kv_dtype, [40, 77, 16, 33], [40, 20, 16, 1], Hq, Hkv, seed=41)
    wl = ew.wl
    pool, out = _run(ew)
    q = oracle.to_f32(ew.q_ext(), wl.q_dtype).astype(np.float64)
    ip = ew.qo_indptr
    for b in range(wl.batch):
        K, V = _rows(pool, wl, b, "k"), _rows(pool, wl, b, "v")
        C = int(ew.chunk_lens[b])
        ref = _dense_causal(q[ip[b]:ip[b + 1]], K, V, wl.sm_scale, wl.group,
                            int(wl.seq_lens[b]) - C)
        np.testing.assert_allclose(out[ip[b]:ip[b + 1]], ref, rtol=0, atol=1e-12)


def test_chunk_of_one_is_the_decode():
    ew = synthetic.extend("e1", "int4", [70, 5, 129], [1, 1, 1], 8, 2, seed=42)
    wl = ew.wl
    pool, out = _run(ew)
    dec = oracle.paged_decode(pool, ew.q_ext(), wl.q_dtype, wl.block_tables, wl.seq_lens,
                              wl.sm_scale)
    assert np.array_equal(out, dec)


def test_later_rows_do_not_reach_earlier_queries():
    ew = synthetic.extend("ec", "int8", [50], [30], 4, 2, seed=43)
    wl = ew.wl
    pool, out = _run(ew)
    # overwrite the last stored token (position 49, seen only by the last query)
    blk, off = int(wl.block_tables[0, 49 // 16]), 49 % 16
    pool.k[blk, off] ^= 0x5A
    pool.v[blk, off] ^= 0x3C
    out2 = oracle.paged_extend(pool, ew.q_ext(), wl.q_dtype, ew.qo_indptr, wl.block_tables,
                               ew.kv_lens, wl.sm_scale)
    assert np.array_equal(out[:-1], out2[:-1])
    assert not np.array_equal(out[-1], out2[-1])


def test_block_permutation_invariance():
    ew = synthetic.extend("ep", "int4", [90, 45], [60, 45], 8, 4, seed=44)
    wl = ew.wl
    pool, out = _run(ew)
    perm = synthetic.permutation(9, 88, wl.num_blocks).astype(np.int32)
    p2 = oracle.Pool(wl.num_blocks, wl.kv_heads, wl.head_dim, wl.kv_dtype)
    src = np.arange(wl.num_blocks, dtype=np.int32)
    assert oracle.copy_blocks(pool, p2, src, perm) == 0
    bt = np.where(wl.block_tables >= 0, perm[np.maximum(wl.block_tables, 0)], -1)
    out2 = oracle.paged_extend(p2, ew.q_ext(), wl.q_dtype, ew.qo_indptr, bt, ew.kv_lens,
                               wl.sm_scale)
    assert np.array_equal(out, out2)
