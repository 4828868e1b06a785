"""bench.py's cold-L2 method for pools that fit in L2: enough replicas that
their total holds at least 3 x L2 (none when the pool alone is larger), each
a copy of the pool in its own storage, rotated so that a call never finds
its pool in L2. Host-side (CPU tensors)."""
import torch

import bench
import paged_quantized_kv_store_gb300 as kvq


def _pool(blocks, kv_dtype="int8"):
    p = kvq.KVPool.allocate(blocks, 2, kv_dtype, device="cpu")
    g = torch.Generator().manual_seed(blocks)
    p.k.copy_(torch.randint(0, 256, p.k.shape, dtype=torch.uint8, generator=g))
    return p


def test_pool_larger_than_three_l2_has_no_replica():
    p = _pool(8)
    pools = bench.replica_pools(kvq, p, l2=p.nbytes() // 3 - 1)
    assert len(pools) == 1 and pools[0] is p


def test_replicas_hold_three_l2_and_copy_the_pool():
    p = _pool(4, "int4")
    l2 = 5 * p.nbytes() + 7
    pools = bench.replica_pools(kvq, p, l2=l2)
    r = len(pools)
    assert r * p.nbytes() >= 3 * l2 and (r - 1) * p.nbytes() < 3 * l2
    for q in pools[1:]:
        assert q.k.data_ptr() != p.k.data_ptr() and torch.equal(q.k, p.k)
        assert torch.equal(q.k_sz, p.k_sz) and q.k_sz.data_ptr() != p.k_sz.data_ptr()
        assert (q.num_blocks, q.kv_heads, q.kv_dtype) == (p.num_blocks, p.kv_heads, p.kv_dtype)
