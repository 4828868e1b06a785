"""GPU parity of the block copy / swap kernel against the oracle's copy
(LMDeploy article §4.4: blocks move by a swap map between the GPU and the
CPU cache). Every copied byte must be equal: codes, elements, scale/zero."""
import numpy as np
import pytest
import torch

import oracle
import synthetic

pytestmark = pytest.mark.gpu

from gpu_harness import decode, fill_pool, i32, out_to_f64, pool_to_host  # noqa: E402


def _kvq():
    import paged_quantized_kv_store_gb300 as kvq
    return kvq


def _host_view(pool):
    """Pool tensors (device or pinned host) as numpy arrays shaped like oracle.Pool's."""
    d = {"k": pool.k.cpu().numpy(), "v": pool.v.cpu().numpy()}
    if pool.k_sz is not None:
        d["k_sz"] = pool.k_sz.cpu().numpy().view(np.uint16).reshape(pool.k_sz.shape + (2,))
        d["v_sz"] = pool.v_sz.cpu().numpy().view(np.uint16).reshape(pool.v_sz.shape + (2,))
    return d


def _oracle_pool_from(view, kv_dtype, kv_heads):
    op = oracle.Pool(view["k"].shape[0], kv_heads, 128, kv_dtype)
    op.k[...] = view["k"]
    op.v[...] = view["v"]
    if op.k_sz is not None:
        op.k_sz[...] = view["k_sz"]
        op.v_sz[...] = view["v_sz"]
    return op


def _assert_pool_equals(pool, opool):
    g = _host_view(pool)
    for key in ("k", "v", "k_sz", "v_sz"):
        o = getattr(opool, key)
        if o is not None:
            assert np.array_equal(g[key], o), key


def _filled(kv_dtype, hkv=8):
    wl = synthetic.custom("cp", kv_dtype, [200, 77, 300, 45], 4 * hkv, hkv, seed=29,
                          extra_blocks=40)
    return wl, fill_pool(wl)


@pytest.mark.parametrize("kv_dtype", ["int4", "int8", "f16", "bf16"])
@pytest.mark.parametrize("where", ["device", "to_host", "from_host"])
def test_copy_matches_oracle(gpu, kv_dtype, where):
    kvq = _kvq()
    wl, pool = _filled(kv_dtype)
    hkv = wl.kv_heads
    other = kvq.KVPool.allocate(37, hkv, kv_dtype, pinned=(where == "to_host"))
    if where == "from_host":  # a host pool holding the device pool's blocks
        host = kvq.KVPool.allocate(wl.num_blocks, hkv, kv_dtype, pinned=True)
        for key in ("k", "v", "k_sz", "v_sz"):
            if getattr(pool, key) is not None:
                getattr(host, key).copy_(getattr(pool, key))
        src, dst = host, pool
    elif where == "to_host":
        src, dst = pool, other
    else:  # copy-on-write inside one pool: into the free tail blocks
        src, dst = pool, pool
    n = 21
    used = wl.num_blocks - 40
    sids = synthetic.permutation(5, 81, used)[:n].astype(np.int32)
    dst_range = dst.num_blocks if dst is not pool else wl.num_blocks
    first = 0 if dst is not pool else used
    dids = (first + synthetic.permutation(6, 82, dst_range - first)[:n]).astype(np.int32)
    osrc = _oracle_pool_from(_host_view(src), kv_dtype, hkv)
    odst = osrc if src is dst else _oracle_pool_from(_host_view(dst), kv_dtype, hkv)
    assert oracle.copy_blocks(osrc, odst, sids, dids) == 0
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.kvq_copy_blocks(src, dst, i32(sids), i32(dids), dev_err)
    assert gpu.kvq_check_error(dev_err) == 0
    _assert_pool_equals(dst, odst)


def test_ids_outside_a_pool_are_skipped_and_reported(gpu):
    kvq = _kvq()
    wl, pool = _filled("int8")
    dst = kvq.KVPool.allocate(4, wl.kv_heads, "int8")
    sids = np.array([1, -1, wl.num_blocks, 2], np.int32)
    dids = np.array([0, 1, 2, 4], np.int32)
    odst = oracle.Pool(4, wl.kv_heads, 128, "int8")
    osrc = _oracle_pool_from(_host_view(pool), "int8", wl.kv_heads)
    assert oracle.copy_blocks(osrc, odst, sids, dids) == 3
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.kvq_copy_blocks(pool, dst, i32(sids), i32(dids), dev_err)
    assert gpu.kvq_check_error(dev_err) == kvq.DEV_ERR_BITS["block_id"]
    _assert_pool_equals(dst, odst)


def test_swap_out_and_back_keeps_attention_bitwise(gpu):
    """Swap a batch's blocks to a pinned host pool, clobber them, swap them back
    to other ids with the tables renumbered: decode gives the same bits."""
    kvq = _kvq()
    wl, pool = _filled("int4")
    bt = i32(wl.block_tables)
    ref = decode(wl, pool, bt)
    nblk = (wl.seq_lens + 15) // 16
    used = np.concatenate([wl.block_tables[b, :nblk[b]] for b in range(wl.batch)])
    host = kvq.KVPool.allocate(used.size, wl.kv_heads, "int4", pinned=True)
    slots = np.arange(used.size, dtype=np.int32)
    kvq.kvq_copy_blocks(pool, host, i32(used), i32(slots))
    for key in ("k", "v", "k_sz", "v_sz"):
        getattr(pool, key).zero_()
    new_ids = synthetic.permutation(8, 83, wl.num_blocks)[:used.size].astype(np.int32)
    kvq.kvq_copy_blocks(host, pool, i32(slots), i32(new_ids))
    remap = dict(zip(used.tolist(), new_ids.tolist()))
    bt2 = np.full_like(wl.block_tables, -1)
    for b in range(wl.batch):
        bt2[b, :nblk[b]] = [remap[int(x)] for x in wl.block_tables[b, :nblk[b]]]
    got = decode(wl, pool, i32(bt2))
    assert torch.equal(got, ref)


def test_empty_map_is_a_no_op(gpu):
    kvq = _kvq()
    wl, pool = _filled("f16")
    before = pool_to_host(pool)
    e = torch.empty(0, dtype=torch.int32, device="cuda")
    kvq.kvq_copy_blocks(pool, pool, e, e)
    torch.cuda.synchronize()
    after = pool_to_host(pool)
    assert all(np.array_equal(before[k], after[k]) for k in before)
