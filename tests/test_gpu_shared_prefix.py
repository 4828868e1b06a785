"""GPU parity of the shared-prefix (cascade) decode against the CPU oracle.

The cascade is an exact reordering of the attention sum (the shared blocks'
part is computed once per group and merged by log-sum-exp), so its oracle is
the plain paged attention over each request's whole block table. Every output
element must be within 2e-3 absolute or 1e-2 relative of it.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic

pytestmark = pytest.mark.gpu

from gpu_harness import (assert_close, decode, fill_pool, i32, i64, oracle_request,  # noqa: E402
                         out_to_f64, to_dev)


def _kvq():
    import paged_quantized_kv_store_gb300 as kvq
    return kvq


def _full_group(wl):
    """One group: the requests holding the whole common prefix."""
    full = len(wl.prefix_blocks)
    members = [b for b in range(wl.batch) if wl.shared_tokens[b] == 16 * full]
    return [(members, full)]


def _run_shared(wl, pool, bt, groups, num_splits=0, dev_err=None):
    kvq = _kvq()
    if dev_err is None:
        dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q = to_dev(wl.q(), wl.q_dtype)
    out = torch.full_like(q, float("nan"))
    g = groups if isinstance(groups, kvq.SharedPrefixGroups) else \
        kvq.SharedPrefixGroups.from_lists(groups)
    ws = kvq.paged_decode_attn_shared_prefix_workspace_size(
        wl.batch, wl.q_heads, wl.kv_heads, wl.max_seq_len, g.max_shared_blocks, num_splits)
    workspace = torch.empty(max(ws, 16), dtype=torch.uint8, device="cuda")
    kvq.paged_decode_attn_shared_prefix(pool, q, out, bt, i32(wl.seq_lens), wl.max_seq_len,
                                        wl.sm_scale, g, num_splits, workspace, dev_err)
    return out, dev_err


def _stored(wl):
    """GPU pool with the workload's context and step tokens stored, its block
    tables, and the oracle's output for the whole batch."""
    pool = fill_pool(wl)
    slots, k, v = wl.step_store()
    _kvq().kv_store_quant(pool, to_dev(k, wl.in_dtype), to_dev(v, wl.in_dtype), i64(slots))
    _, oout = oracle.run_workload(wl)
    return pool, i32(wl.block_tables), oout


LENS = [12 * 16 + 1, 17, 300, 193, 500, 1000, 12 * 16 + 16, 260, 777]

CASES = [
    # kv dtype, q dtype, q heads, kv heads
    ("int4", "f16", 32, 8),
    ("int4", "bf16", 32, 8),
    ("int8", "f16", 32, 8),
    ("int8", "bf16", 16, 8),
    ("int8", "f16", 8, 8),
    ("int8", "f16", 24, 8),
    ("int4", "f16", 64, 4),
    ("f16", "f16", 16, 8),
    ("bf16", "bf16", 16, 8),
]


@pytest.mark.parametrize("kv_dtype,q_dtype,hq,hkv", CASES)
def test_shared_prefix_matches_oracle(gpu, kv_dtype, q_dtype, hq, hkv):
    wl = synthetic.shared_prefix("sp", kv_dtype, LENS, hq, hkv, prefix_blocks=12,
                                 q_dtype=q_dtype)
    pool, bt, oout = _stored(wl)
    out, dev_err = _run_shared(wl, pool, bt, _full_group(wl))
    assert gpu.kvq_check_error(dev_err) == 0
    got = out_to_f64(out)
    assert_close(got, oout)
    # and against the plain decode of the same pool
    assert_close(got, out_to_f64(decode(wl, pool, bt)))


@pytest.mark.parametrize("splits", [1, 2, 4, 0])
def test_shared_prefix_split_counts(gpu, splits):
    wl = synthetic.shared_prefix("sp", "int4", LENS, 32, 8, prefix_blocks=12)
    pool, bt, oout = _stored(wl)
    out, dev_err = _run_shared(wl, pool, bt, _full_group(wl), num_splits=splits)
    assert gpu.kvq_check_error(dev_err) == 0
    assert_close(out_to_f64(out), oout)


def test_detected_and_nested_groups(gpu):
    wl = synthetic.shared_prefix("sp", "int8", LENS + [40, 33], 32, 8, prefix_blocks=12)
    pool, bt, oout = _stored(wl)
    det = _kvq().SharedPrefixGroups.detect(wl.block_tables, wl.seq_lens)
    assert det.num_groups >= 1
    out, dev_err = _run_shared(wl, pool, bt, det)
    assert gpu.kvq_check_error(dev_err) == 0
    assert_close(out_to_f64(out), oout)
    # two groups: the full-prefix holders, and the short requests sharing
    # their one or two leading blocks
    full = _full_group(wl)[0][0]
    short = [b for b in range(wl.batch) if b not in full and wl.shared_tokens[b] >= 16]
    s_short = int(min(wl.shared_tokens[b] for b in short)) // 16
    out, dev_err = _run_shared(wl, pool, bt, [(full, 12), (short, s_short)])
    assert gpu.kvq_check_error(dev_err) == 0
    assert_close(out_to_f64(out), oout)


def test_long_prefix_many_members(gpu):
    # lognormal lengths around a 64-block prefix (the INT4 GQA-4 workload's
    # shape at a quarter of its batch)
    wl = synthetic.cfg4(batch=16)
    pool, bt, oout = _stored(wl)
    out, dev_err = _run_shared(wl, pool, bt, _full_group(wl))
    assert gpu.kvq_check_error(dev_err) == 0
    assert_close(out_to_f64(out), oout)


def _pool_pair(kv_dtype, num_blocks, kv_heads, seed=21):
    """The same random rows stored in every slot of a GPU pool and an oracle pool."""
    kvq = _kvq()
    n = num_blocks * 16
    k = synthetic.normal(seed, 901, 0, n * kv_heads * 128).reshape(n, kv_heads, 128)
    v = synthetic.normal(seed, 902, 0, n * kv_heads * 128).reshape(n, kv_heads, 128)
    pool = kvq.KVPool.allocate(num_blocks, kv_heads, kv_dtype)
    kvq.kv_store_quant(pool, to_dev(k, "f16"), to_dev(v, "f16"), i64(np.arange(n)))
    opool = oracle.Pool(num_blocks, kv_heads, 128, kv_dtype)
    assert oracle.kv_store(opool, k, v, "f16", np.arange(n)) == 0
    return pool, opool


def _shared_call(pool, q, bt, lens, groups, max_seq_len, dev_err):
    kvq = _kvq()
    B, Hq, _ = q.shape
    g = kvq.SharedPrefixGroups.from_lists(groups)
    ws = kvq.paged_decode_attn_shared_prefix_workspace_size(B, Hq, pool.kv_heads, max_seq_len,
                                                            g.max_shared_blocks)
    workspace = torch.empty(max(ws, 16), dtype=torch.uint8, device="cuda")
    out = torch.full_like(q, float("nan"))
    kvq.paged_decode_attn_shared_prefix(pool, q, out, bt, lens, max_seq_len, 128 ** -0.5, g, 0,
                                        workspace, dev_err)
    return out


@pytest.mark.parametrize("kv_dtype", ["int4", "int8"])
def test_members_with_no_own_blocks(gpu, kv_dtype):
    # requests 0 and 1 consist of the 3 shared blocks only; request 2 adds
    # two private blocks; request 3 is in no group
    pool, opool = _pool_pair(kv_dtype, 12, 8)
    bt = np.array([[4, 9, 2, -1, -1], [4, 9, 2, -1, -1], [4, 9, 2, 7, 0], [5, 6, -1, -1, -1]],
                  dtype=np.int32)
    lens = np.array([48, 48, 70, 20], dtype=np.int32)
    qbits = synthetic.normal(5, 903, 0, 4 * 32 * 128).reshape(4, 32, 128)
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = _shared_call(pool, to_dev(qbits, "f16"), i32(bt), i32(lens), [([0, 1, 2], 3)], 80,
                       dev_err)
    assert gpu.kvq_check_error(dev_err) == 0
    ref = oracle.paged_decode(opool, qbits, "f16", bt, lens, 128 ** -0.5)
    assert_close(out_to_f64(out), ref)


def test_group_errors_are_reported(gpu):
    pool, _ = _pool_pair("int4", 12, 8)
    bt = np.array([[4, 9, 2, 1], [4, 9, 3, 1], [4, 9, 2, 8], [4, 9, 2, 10]], dtype=np.int32)
    lens = np.array([60, 60, 60, 20], dtype=np.int32)
    q = to_dev(synthetic.normal(5, 904, 0, 4 * 32 * 128).reshape(4, 32, 128), "f16")
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    prefix = _kvq().DEV_ERR_BITS["prefix"]
    cases = [
        [([0, 1], 3)],             # tables differ in block 2
        [([0, 3], 3)],             # request 3 is shorter than the shared part
        [([0, 2], 3), ([2], 1)],   # request 2 listed twice
        [([0, 7], 2)],             # member out of range
    ]
    for groups in cases:
        _shared_call(pool, q, i32(bt), i32(lens), groups, 64, dev_err)
        bits = gpu.kvq_check_error(dev_err)
        assert bits & prefix, groups
    # valid groups set nothing
    _shared_call(pool, q, i32(bt), i32(lens), [([0, 2, 3], 1), ([1], 2)], 64, dev_err)
    assert gpu.kvq_check_error(dev_err) == 0


@pytest.mark.slow
def test_full_size_int4_shared_prefix_sampled(gpu):
    wl = synthetic.cfg4()
    pool = fill_pool(wl)
    slots, k, v = wl.step_store()
    _kvq().kv_store_quant(pool, to_dev(k, wl.in_dtype), to_dev(v, wl.in_dtype), i64(slots))
    bt = i32(wl.block_tables)
    out, dev_err = _run_shared(wl, pool, bt, _full_group(wl))
    assert gpu.kvq_check_error(dev_err) == 0
    got = out_to_f64(out)
    assert_close(got, out_to_f64(decode(wl, pool, bt)))
    lens = wl.seq_lens
    for b in sorted({0, wl.batch - 1, int(lens.argmax()), int(lens.argmin()), wl.batch // 2}):
        _, oout = oracle_request(wl, b)
        assert_close(got[b], oout)


def test_block_id_outside_the_pool_in_the_shared_part(gpu):
    """A bad id among the shared blocks: reported, no fault, finite outputs."""
    import paged_quantized_kv_store_gb300 as kvq
    pool, _ = _pool_pair("int4", 12, 8)
    bt = np.array([[4, 99, 2, 1], [4, 99, 2, 7], [4, 99, 2, 8]], dtype=np.int32)
    lens = np.array([60, 60, 55], dtype=np.int32)
    q = to_dev(synthetic.normal(5, 905, 0, 3 * 32 * 128).reshape(3, 32, 128), "f16")
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = _shared_call(pool, q, i32(bt), i32(lens), [([0, 1, 2], 3)], 64, dev_err)
    assert gpu.kvq_check_error(dev_err) & kvq.DEV_ERR_BITS["block_id"]
    assert torch.isfinite(out.float()).all()


@pytest.mark.slow
def test_cascade_with_the_balanced_tail(gpu):
    """Long contexts behind a shared prefix: the members' own blocks give
    per-warp shares above 128 blocks, so the decode hands out tail chunks and
    the combine merges tail pieces with the prefix records. Same outputs as
    the plain decode over whole block tables, and as the oracle on the
    shortest request."""
    wl = synthetic.shared_prefix("sp_tail", "int8", [49152, 40000, 49152, 33333], 48, 48,
                                 prefix_blocks=512, seed=59)
    pool = fill_pool(wl)
    slots, k, v = wl.step_store()
    _kvq().kv_store_quant(pool, to_dev(k, wl.in_dtype), to_dev(v, wl.in_dtype), i64(slots))
    bt = i32(wl.block_tables)
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    plain = decode(wl, pool, bt, dev_err=dev_err)
    out, dev_err = _run_shared(wl, pool, bt, _full_group(wl), dev_err=dev_err)
    assert _kvq().kvq_check_error(dev_err) == 0
    assert_close(out_to_f64(out), out_to_f64(plain))
    b = int(np.argmin(wl.seq_lens))
    _, oout = oracle_request(wl, b)
    assert_close(out_to_f64(out)[b], oout)
