"""Pins of the oracle's block copy / swap (LMDeploy article §4.4: the cache
engine moves whole blocks between caches by a swap map).

What fixes the result independently of the copy itself: attention reads KV
only through the block tables, so moving a request's blocks to other ids (in
the same pool or another) and renumbering its table must leave its output
bit-for-bit unchanged; swapping blocks out and back in is the identity; ids
outside a pool change nothing.
"""
import numpy as np
import pytest

import oracle
import synthetic


def _pool_and_workload(kv_dtype):
    wl = synthetic.custom("cp", kv_dtype, [40, 97, 16, 130], 16, 4, seed=13)
    pool, out = oracle.run_workload(wl)
    return wl, pool, out


@pytest.mark.parametrize("kv_dtype", ["int4", "int8", "f16", "bf16"])
def test_moved_blocks_give_bitwise_identical_attention(kv_dtype):
    wl, pool, out = _pool_and_workload(kv_dtype)
    # a second pool, larger, with the blocks of every request at new ids
    dst = oracle.Pool(wl.num_blocks + 40, wl.kv_heads, wl.head_dim, kv_dtype)
    nblk = (wl.seq_lens + 15) // 16
    used = np.concatenate([wl.block_tables[b, :nblk[b]] for b in range(wl.batch)])
    new_ids = synthetic.permutation(3, 77, dst.num_blocks)[:used.size].astype(np.int32)
    assert oracle.copy_blocks(pool, dst, used, new_ids) == 0
    remap = dict(zip(used.tolist(), new_ids.tolist()))
    bt = np.full_like(wl.block_tables, -1)
    for b in range(wl.batch):
        bt[b, :nblk[b]] = [remap[int(x)] for x in wl.block_tables[b, :nblk[b]]]
    out2 = oracle.paged_decode(dst, wl.q(), wl.q_dtype, bt, wl.seq_lens, wl.sm_scale)
    assert np.array_equal(out, out2)


@pytest.mark.parametrize("kv_dtype", ["int4", "f16"])
def test_swap_out_and_in_is_the_identity(kv_dtype):
    wl, pool, _ = _pool_and_workload(kv_dtype)
    before = {k: getattr(pool, k).copy() for k in ("k", "v", "k_sz", "v_sz")
              if getattr(pool, k) is not None}
    ids = np.array([2, 5, 7], dtype=np.int32)
    host = oracle.Pool(8, wl.kv_heads, wl.head_dim, kv_dtype)
    slots = np.array([6, 0, 3], dtype=np.int32)
    assert oracle.copy_blocks(pool, host, ids, slots) == 0
    for k in before:  # clobber the swapped-out blocks, then bring them back
        getattr(pool, k)[ids] = 0xA5 if getattr(pool, k).dtype == np.uint8 else 0x1234
    assert oracle.copy_blocks(host, pool, slots, ids) == 0
    for k, v in before.items():
        assert np.array_equal(getattr(pool, k), v), k


def test_ids_outside_a_pool_are_skipped_and_counted():
    wl, pool, _ = _pool_and_workload("int8")
    dst = oracle.Pool(4, wl.kv_heads, wl.head_dim, "int8")
    n = oracle.copy_blocks(pool, dst, np.array([1, -1, wl.num_blocks, 2], np.int32),
                           np.array([0, 1, 2, 4], np.int32))
    assert n == 3  # src -1, src past the pool, dst past the pool
    assert np.array_equal(dst.k[0], pool.k[1])
    assert not dst.k[1:].any() and not dst.k_sz[1:].any()


def test_pairs_apply_in_order():
    wl, pool, _ = _pool_and_workload("int4")
    dst = oracle.Pool(2, wl.kv_heads, wl.head_dim, "int4")
    oracle.copy_blocks(pool, dst, np.array([3, 5], np.int32), np.array([1, 1], np.int32))
    assert np.array_equal(dst.k[1], pool.k[5]) and np.array_equal(dst.v_sz[1], pool.v_sz[5])
