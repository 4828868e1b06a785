"""Pins for the oracle's paged decode attention.

LMDeploy article §2.2 (block tables, block size 16) and §3.2 item 3 (attention
through indirect pointers into a non-contiguous KV layout). The paged oracle
is pinned to
* dense brute-force attention (numpy, fp64) over an unpaged, contiguous cache
  built straight from the generator or read out of the pool arrays by plain
  [block, offset, head] indexing,
* softmax weights that are non-negative and sum to 1,
* uniform K (a constant row quantizes to scale 0): output = mean of V,
* zero query: output = mean of V,
* one key far above the others: output = its V,
* length 1: output = the one V row,
* invariance, bit for bit, under a permutation of physical block ids,
* GQA: q-head h reads kv head h // (Hq / Hkv).
"""
import numpy as np
import pytest

import oracle
import synthetic


def _dense_attention(q, K, V, sm_scale, group):
    """q [Hq, D], K/V [L, Hkv, D] (fp64) -> [Hq, D]; textbook softmax attention."""
    Hq = q.shape[0]
    out = np.zeros_like(q)
    for h in range(Hq):
        k = K[:, h // group, :]
        v = V[:, h // group, :]
        s = sm_scale * (k @ q[h])
        w = np.exp(s - s.max())
        w /= w.sum()
        out[h] = w @ v
    return out


def _pool_contiguous(pool, wl, b, which):
    """Dequantized [L, Hkv, D] of request b read from the pool arrays by index."""
    L = int(wl.seq_lens[b])
    arr = pool.k if which == "k" else pool.v
    szs = pool.k_sz if which == "k" else pool.v_sz
    out = np.zeros((L, wl.kv_heads, wl.head_dim))
    for t in range(L):
        blk = int(wl.block_tables[b, t // 16])
        off = t % 16
        row = arr[blk, off]  # [Hkv, row_bytes]
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


def test_fp16_paged_matches_dense_from_generator():
    wl = synthetic.cfg1()
    pool, out = oracle.run_workload(wl)
    q = oracle.to_f32(wl.q(), wl.q_dtype).astype(np.float64)
    for b in range(wl.batch):
        L = int(wl.seq_lens[b])
        K = oracle.to_f32(wl.ctx_rows("k", b, 0, L), "f16").astype(np.float64)
        V = oracle.to_f32(wl.ctx_rows("v", b, 0, L), "f16").astype(np.float64)
        ref = _dense_attention(q[b], K, V, wl.sm_scale, wl.group)
        np.testing.assert_allclose(out[b], ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("kv_dtype,Hq,Hkv", [("int8", 8, 8), ("int4", 8, 2), ("bf16", 4, 1),
                                             ("int8", 6, 3)])
def test_quantized_paged_matches_dense_from_pool(kv_dtype, Hq, Hkv):
    wl = synthetic.custom(f"dense_{kv_dtype}", kv_dtype, [1, 15, 16, 17, 70, 129], Hq, Hkv,
                          seed=21)
    pool, out = oracle.run_workload(wl)
    q = oracle.to_f32(wl.q(), wl.q_dtype).astype(np.float64)
    for b in range(wl.batch):
        K = _pool_contiguous(pool, wl, b, "k")
        V = _pool_contiguous(pool, wl, b, "v")
        ref = _dense_attention(q[b], K, V, wl.sm_scale, wl.group)
        np.testing.assert_allclose(out[b], ref, rtol=0, atol=1e-12)


def test_weights_sum_to_one():
    wl = synthetic.custom("w", "int4", [5, 100, 333], 4, 2, seed=22)
    pool, _ = oracle.run_workload(wl)
    q = wl.q()
    for b in range(wl.batch):
        for h in range(wl.q_heads):
            _, p = oracle.decode_one(pool, q[b, h], wl.q_dtype, wl.block_tables[b],
                                     int(wl.seq_lens[b]), h // wl.group, wl.sm_scale)
            assert (p >= 0).all()
            assert abs(p.sum() - 1) < 1e-12


def _manual_pool(kv_dtype, k_rows, v_rows, in_dtype="f16"):
    """Pool holding one request whose rows are given (uint16 [L, Hkv, D])."""
    L, Hkv, D = k_rows.shape
    nblk = (L + 15) // 16
    pool = oracle.Pool(nblk + 2, Hkv, D, kv_dtype)
    bt = np.arange(nblk, dtype=np.int32)[::-1].copy() + 2  # non-trivial ids
    pos = np.arange(L)
    slots = bt[pos // 16].astype(np.int64) * 16 + pos % 16
    oracle.kv_store(pool, k_rows, v_rows, in_dtype, slots)
    return pool, bt


def _f16(x):
    return np.asarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


@pytest.mark.parametrize("kv_dtype", ["int8", "int4", "f16"])
def test_uniform_k_gives_mean_of_v(kv_dtype):
    L, Hkv, D = 37, 1, 128
    k = _f16(np.full((L, Hkv, D), 0.3))
    v_bits = synthetic.normal(5, 100, 0, L * Hkv * D).reshape(L, Hkv, D)
    pool, bt = _manual_pool(kv_dtype, k, v_bits)
    q = synthetic.normal(5, 101, 0, D)
    out, p = oracle.decode_one(pool, q, "f16", bt, L, 0, 1 / np.sqrt(D))
    vhat = _pool_rows(pool, bt, L, kv_dtype, "v")
    np.testing.assert_allclose(p, np.full(L, 1 / L), rtol=1e-12)
    np.testing.assert_allclose(out, vhat.mean(axis=0), rtol=0, atol=1e-12)


def _pool_rows(pool, bt, L, kv_dtype, which):
    class W:  # minimal view for _pool_contiguous
        pass
    w = W()
    w.seq_lens = np.array([L])
    w.block_tables = bt[None]
    w.kv_heads = pool.kv_heads
    w.head_dim = pool.head_dim
    w.kv_dtype = kv_dtype
    return _pool_contiguous(pool, w, 0, which)[:, 0, :]


def test_zero_query_gives_mean_of_v():
    L, D = 50, 128
    k = synthetic.normal(6, 100, 0, L * D).reshape(L, 1, D)
    v = synthetic.normal(6, 101, 0, L * D).reshape(L, 1, D)
    pool, bt = _manual_pool("int8", k, v)
    out, _ = oracle.decode_one(pool, np.zeros(D, np.uint16), "f16", bt, L, 0, 0.088)
    np.testing.assert_allclose(out, _pool_rows(pool, bt, L, "int8", "v").mean(0), atol=1e-12)


def test_dominant_key_selects_its_value():
    L, D = 40, 128
    q = np.ones(D, dtype=np.float32)
    k = np.zeros((L, 1, D), dtype=np.float32)
    k[23, 0, :] = 4.0  # score 128*4/sqrt(128) ~ 45 above the rest
    v = synthetic.normal(7, 101, 0, L * D).reshape(L, 1, D)
    pool, bt = _manual_pool("f16", _f16(k), v)
    out, p = oracle.decode_one(pool, _f16(q), "f16", bt, L, 0, 1 / np.sqrt(D))
    assert p[23] > 1 - 1e-15
    np.testing.assert_allclose(out, oracle.f16_to_f32(v[23, 0]), atol=1e-15)


@pytest.mark.parametrize("kv_dtype", ["int4", "bf16"])
def test_length_one_returns_the_value(kv_dtype):
    D = 128
    k = synthetic.normal(8, 100, 0, D, dtype="bf16").reshape(1, 1, D)
    v = synthetic.normal(8, 101, 0, D, dtype="bf16").reshape(1, 1, D)
    pool, bt = _manual_pool(kv_dtype, k, v, in_dtype="bf16")
    q = synthetic.normal(8, 102, 0, D, dtype="bf16")
    out, p = oracle.decode_one(pool, q, "bf16", bt, 1, 0, 0.1)
    assert p[0] == 1.0
    np.testing.assert_allclose(out, _pool_rows(pool, bt, 1, kv_dtype, "v")[0], atol=0)


def test_empty_request_gives_zeros():
    wl = synthetic.custom("empty", "int8", [0, 20], 2, 2, seed=23)
    _, out = oracle.run_workload(wl)
    assert (out[0] == 0).all()
    assert np.abs(out[1]).sum() > 0


@pytest.mark.parametrize("kv_dtype", ["int8", "int4", "f16"])
def test_block_permutation_invariance(kv_dtype):
    wl = synthetic.custom("perm", kv_dtype, [3, 40, 97, 160], 4, 2, seed=24)
    pool, out = oracle.run_workload(wl)
    perm = synthetic.permutation(99, 5, wl.num_blocks)  # new physical id of each block
    pool2 = oracle.Pool(wl.num_blocks, wl.kv_heads, wl.head_dim, wl.kv_dtype)
    pool2.k[perm] = pool.k
    pool2.v[perm] = pool.v
    if pool.k_sz is not None:
        pool2.k_sz[perm] = pool.k_sz
        pool2.v_sz[perm] = pool.v_sz
    bt2 = np.where(wl.block_tables >= 0, perm[np.maximum(wl.block_tables, 0)], -1).astype(np.int32)
    out2 = oracle.paged_decode(pool2, wl.q(), wl.q_dtype, bt2, wl.seq_lens, wl.sm_scale)
    assert np.array_equal(out, out2)


def test_gqa_mapping_uses_consecutive_groups():
    # kv head j holds the constant value j in V; q-head h must read kv head h // g
    L, Hkv, D, Hq = 20, 4, 128, 8
    k = synthetic.normal(9, 100, 0, L * Hkv * D).reshape(L, Hkv, D)
    v = _f16(np.broadcast_to(np.arange(Hkv, dtype=np.float32)[None, :, None], (L, Hkv, D)))
    pool, bt = _manual_pool("f16", k, v)
    q = synthetic.normal(9, 101, 0, Hq * D).reshape(1, Hq, D)
    out = oracle.paged_decode(pool, q, "f16", bt[None], np.array([L], np.int32), 0.1)
    for h in range(Hq):
        np.testing.assert_allclose(out[0, h], h // (Hq // Hkv), atol=1e-12)
