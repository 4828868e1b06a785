"""GPU parity of extend (chunked prefill) attention against the CPU oracle.

"pymllm Runtime Design", forward stage (extend / prefill); LMDeploy article
§2.3 (prefills split into chunks). Every output element must be within 2e-3
absolute or 1e-2 relative of the oracle's fp64 result on the same stored
values; both the direct path (enough query tiles) and the split-context path
(a short chunk over a long prefix: parts merged by a combine kernel) are run.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic

pytestmark = pytest.mark.gpu

from gpu_harness import assert_close, fill_pool, i32, i64, out_to_f64, to_dev  # noqa: E402


def _kvq():
    import paged_quantized_kv_store_gb300 as kvq
    return kvq


def _stored_pool(wl):
    pool = fill_pool(wl)
    slots, k, v = wl.step_store()
    _kvq().kv_store_quant(pool, to_dev(k, wl.in_dtype), to_dev(v, wl.in_dtype), i64(slots))
    return pool


def _gpu_extend(ew, pool, dev_err=None, q=None, variant="auto"):
    kvq = _kvq()
    wl = ew.wl
    if dev_err is None:
        dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q = to_dev(ew.q_ext(), wl.q_dtype) if q is None else q
    out = torch.full_like(q, float("nan"))
    ws = kvq.paged_extend_attn_workspace_size(wl.batch, ew.total_q, wl.q_heads, wl.kv_heads,
                                              wl.max_seq_len)
    workspace = torch.empty(max(ws, 16), dtype=torch.uint8, device="cuda")
    kvq.paged_extend_attn(pool, q, out, i32(ew.qo_indptr), i32(ew.kv_lens),
                          i32(wl.block_tables), wl.max_seq_len, wl.sm_scale, workspace, dev_err,
                          variant=variant)
    return out, dev_err


def _oracle(ew):
    wl = ew.wl
    opool, _ = oracle.run_workload(wl)
    return oracle.paged_extend(opool, ew.q_ext(), wl.q_dtype, ew.qo_indptr, wl.block_tables,
                               ew.kv_lens, wl.sm_scale)


CASES = [
    # kv dtype, q dtype, q heads, kv heads
    ("int8", "f16", 32, 8),
    ("int8", "bf16", 16, 8),
    ("int4", "f16", 32, 8),
    ("int4", "bf16", 8, 8),
    ("f16", "f16", 16, 8),
    ("bf16", "bf16", 16, 8),
    ("int8", "f16", 24, 8),   # 3 q heads per kv head: tiles straddle queries
    ("int4", "f16", 64, 2),   # 32 q heads per kv head: a query spans two tiles
]

# fresh prefills, extends over a cached prefix, a one-token chunk
KV_LENS = [300, 100, 517, 16, 40]
CHUNKS = [300, 37, 200, 16, 1]


@pytest.mark.parametrize("variant", ["mma_sync", "tcgen05"])
@pytest.mark.parametrize("kv_dtype,q_dtype,hq,hkv", CASES)
def test_extend_matches_oracle(gpu, kv_dtype, q_dtype, hq, hkv, variant):
    if variant == "tcgen05" and kv_dtype == "bf16":
        pytest.skip("the tcgen05 kernel takes INT8, INT4 and fp16 pools")
    ew = synthetic.extend("ext", kv_dtype, KV_LENS, CHUNKS, hq, hkv, q_dtype=q_dtype)
    pool = _stored_pool(ew.wl)
    out, dev_err = _gpu_extend(ew, pool, variant=variant)
    assert gpu.kvq_check_error(dev_err) == 0
    assert_close(out_to_f64(out), _oracle(ew))


@pytest.mark.parametrize("kv_dtype", ["int8", "int4", "bf16"])
def test_short_chunks_over_long_prefixes_split_the_context(gpu, kv_dtype):
    # few query tiles, long contexts: the planner cuts the context into parts
    ew = synthetic.extend("exs", kv_dtype, [3000, 2100, 1700], [5, 1, 12], 32, 8,
                          outliers=True)
    kvq = _kvq()
    wl = ew.wl
    ws = kvq.paged_extend_attn_workspace_size(wl.batch, ew.total_q, wl.q_heads, wl.kv_heads,
                                              wl.max_seq_len)
    assert ws > 4096  # records of the parts
    pool = _stored_pool(wl)
    out, dev_err = _gpu_extend(ew, pool)
    assert gpu.kvq_check_error(dev_err) == 0
    assert_close(out_to_f64(out), _oracle(ew))


def test_one_token_chunks_agree_with_decode(gpu):
    ew = synthetic.extend("ex1", "int4", [70, 5, 1029, 640], [1, 1, 1, 1], 32, 8)
    wl = ew.wl
    pool = _stored_pool(wl)
    q = to_dev(ew.q_ext(), wl.q_dtype)
    out, dev_err = _gpu_extend(ew, pool, q=q)
    assert gpu.kvq_check_error(dev_err) == 0
    kvq = _kvq()
    dec = torch.empty_like(q)
    ws = kvq.paged_decode_attn_workspace_size(wl.batch, wl.q_heads, wl.kv_heads, wl.max_seq_len)
    w = torch.empty(max(ws, 16), dtype=torch.uint8, device="cuda")
    kvq.paged_decode_attn(pool, q, dec, i32(wl.block_tables), i32(wl.seq_lens), wl.max_seq_len,
                          wl.sm_scale, 0, w, dev_err)
    assert_close(out_to_f64(out), out_to_f64(dec))


def test_bad_requests_are_reported_and_skipped(gpu):
    ew = synthetic.extend("exb", "int8", [64, 40], [10, 40], 16, 8)
    wl = ew.wl
    pool = _stored_pool(wl)
    kvq = _kvq()
    q = to_dev(ew.q_ext(), wl.q_dtype)
    out = torch.zeros_like(q)
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = kvq.paged_extend_attn_workspace_size(wl.batch, ew.total_q, wl.q_heads, wl.kv_heads, 64)
    w = torch.empty(max(ws, 16), dtype=torch.uint8, device="cuda")
    bad_lens = i32([64, 30])  # request 1: chunk of 40 over a context of 30
    ref = _oracle(synthetic.extend("exb", "int8", [64], [10], 16, 8))
    for variant in ("mma_sync", "tcgen05"):
        out.zero_()
        kvq.paged_extend_attn(pool, q, out, i32(ew.qo_indptr), bad_lens, i32(wl.block_tables),
                              64, wl.sm_scale, w, dev_err, variant=variant)
        assert gpu.kvq_check_error(dev_err) == kvq.DEV_ERR_BITS["length"]
        assert not out[10:].any()  # its rows are not written
        assert_close(out_to_f64(out[:10]), ref)


@pytest.mark.slow
@pytest.mark.parametrize("variant", ["mma_sync", "tcgen05"])
def test_full_size_prefill_chunk_sampled(gpu, variant):
    """The mixed step's 4096-token chunk (INT8, GQA 32q/8kv) prefilled on its own;
    sampled rows (first, last, middle, a block boundary) against the oracle."""
    ew = synthetic.cfg5_prefill()
    wl = ew.wl
    pool = _stored_pool(wl)
    out, dev_err = _gpu_extend(ew, pool, variant=variant)
    assert gpu.kvq_check_error(dev_err) == 0
    got = out_to_f64(out)
    assert np.isfinite(got).all()
    opool, _ = oracle.run_workload(wl)
    q = ew.q_ext()
    for i in (0, 15, 16, 1000, 2047, 4095):
        for h in (0, 5, 31):
            ref, _ = oracle.decode_one(opool, q[i, h], wl.q_dtype, wl.block_tables[0], i + 1,
                                       h // wl.group, wl.sm_scale)
            assert_close(got[i, h], ref)


@pytest.mark.parametrize("variant", ["mma_sync", "tcgen05"])
def test_block_ids_outside_the_pool_are_skipped_and_reported(gpu, variant):
    """A block id past the pool in one request: the bit is set, that block's
    tokens are left out (its rows stay finite), the other request is exact."""
    ew = synthetic.extend("exh", "int8", [300, 200], [300, 120], 32, 8)
    wl = ew.wl
    pool = _stored_pool(wl)
    kvq = _kvq()
    bt = wl.block_tables.copy()
    bt[1, 3] = wl.num_blocks + 7  # request 1, tokens 48 .. 63
    q = to_dev(ew.q_ext(), wl.q_dtype)
    out = torch.full_like(q, float("nan"))
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = kvq.paged_extend_attn_workspace_size(wl.batch, ew.total_q, wl.q_heads, wl.kv_heads,
                                              wl.max_seq_len)
    w = torch.empty(max(ws, 16), dtype=torch.uint8, device="cuda")
    kvq.paged_extend_attn(pool, q, out, i32(ew.qo_indptr), i32(ew.kv_lens), i32(bt),
                          wl.max_seq_len, wl.sm_scale, w, dev_err, variant=variant)
    assert gpu.kvq_check_error(dev_err) == kvq.DEV_ERR_BITS["block_id"]
    got = out_to_f64(out)
    assert np.isfinite(got).all()
    ref = _oracle(ew)
    assert_close(got[:300], ref[:300])


@pytest.mark.parametrize("variant", ["mma_sync", "tcgen05"])
@pytest.mark.parametrize("kv_dtype,q_dtype", [("int8", "f16"), ("int4", "f16"), ("int8", "bf16")])
@pytest.mark.parametrize("sm_scale", [0.0, -0.0625])
def test_zero_and_negative_softmax_scales(gpu, kv_dtype, q_dtype, sm_scale, variant):
    """A scale of 0 (uniform weights over the causal window) and a negative
    scale (the maximum of s is the minimum of q.k): the fp16-query tcgen05
    path applies such scales before the maximum instead of in the exponent."""
    ew = synthetic.extend("exsc", kv_dtype, [300, 100], [300, 37], 32, 8, q_dtype=q_dtype)
    wl = ew.wl
    pool = _stored_pool(wl)
    kvq = _kvq()
    q = to_dev(ew.q_ext(), wl.q_dtype)
    out = torch.full_like(q, float("nan"))
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = kvq.paged_extend_attn_workspace_size(wl.batch, ew.total_q, wl.q_heads, wl.kv_heads,
                                              wl.max_seq_len)
    w = torch.empty(max(ws, 16), dtype=torch.uint8, device="cuda")
    kvq.paged_extend_attn(pool, q, out, i32(ew.qo_indptr), i32(ew.kv_lens),
                          i32(wl.block_tables), wl.max_seq_len, sm_scale, w, dev_err,
                          variant=variant)
    assert gpu.kvq_check_error(dev_err) == 0
    opool, _ = oracle.run_workload(wl)
    ref = oracle.paged_extend(opool, ew.q_ext(), wl.q_dtype, ew.qo_indptr, wl.block_tables,
                              ew.kv_lens, sm_scale)
    assert_close(out_to_f64(out), ref)


def test_tcgen05_refuses_batches_above_4096(gpu):
    """The tcgen05 variant keeps its per-request unit table in shared memory
    and takes at most 4096 requests; a larger batch is refused before
    anything launches (AUTO takes the mma.sync kernel for it)."""
    kvq = _kvq()
    n = 4097
    ew = synthetic.extend("exr", "int8", [1] * n, [1] * n, 16, 8)
    wl = ew.wl
    pool = _stored_pool(wl)
    q = to_dev(ew.q_ext(), wl.q_dtype)
    out = torch.zeros_like(q)
    ws = kvq.paged_extend_attn_workspace_size(wl.batch, ew.total_q, wl.q_heads, wl.kv_heads,
                                              wl.max_seq_len)
    w = torch.empty(max(ws, 16), dtype=torch.uint8, device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        kvq.paged_extend_attn(pool, q, out, i32(ew.qo_indptr), i32(ew.kv_lens),
                              i32(wl.block_tables), wl.max_seq_len, wl.sm_scale, w,
                              variant="tcgen05")
    assert e.value.status == 2  # KVQ_ERR_UNSUPPORTED
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.paged_extend_attn(pool, q, out, i32(ew.qo_indptr), i32(ew.kv_lens),
                          i32(wl.block_tables), wl.max_seq_len, wl.sm_scale, w, dev_err)
    assert gpu.kvq_check_error(dev_err) == 0
    # one token attending itself: the output is that token's dequantized V
    opool, _ = oracle.run_workload(wl)
    ref = oracle.paged_extend(opool, ew.q_ext()[:64], wl.q_dtype, ew.qo_indptr[:65],
                              wl.block_tables[:64], ew.kv_lens[:64], wl.sm_scale)
    assert_close(out_to_f64(out[:64]), ref)
