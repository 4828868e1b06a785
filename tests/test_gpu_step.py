"""GPU parity of the fused decode step (kvq_decode_step: block tables, store
of the step's tokens and attention in one cooperative launch) against the
oracle and against the same step run as its three calls.

"pymllm Runtime Design", forward stage: a decode step stores each request's
new token and attends over its cache. The pool after the step must be
bit-exact with the oracle's, the block tables bit-exact, the outputs within
the decode tolerance of the oracle's fp64 result.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic

pytestmark = pytest.mark.gpu

from gpu_harness import (TORCH_DT, assert_close, fill_pool, gpu_request_rows,  # noqa: E402
                         i32, i64, oracle_request, oracle_request_rows, out_to_f64,
                         pool_to_host, run_step, to_dev)


def fused_step(gpu, wl, pool, num_splits=0, dev_err=None, req_to_token=None):
    """The whole step through kvq_decode_step; returns (out, block tables, error word)."""
    if dev_err is None:
        dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    r2t = wl.req_to_token if req_to_token is None else req_to_token
    bt = torch.full((wl.batch, wl.max_blocks_per_seq), 7, dtype=torch.int32, device="cuda")
    slots, k, v = wl.step_store()
    q = to_dev(wl.q(), wl.q_dtype)
    out = torch.empty_like(q)
    ws = gpu.kvq_decode_step_workspace_size(wl.batch, wl.q_heads, wl.kv_heads, wl.max_seq_len,
                                            num_splits)
    workspace = torch.empty(ws, dtype=torch.uint8, device="cuda")
    gpu.kvq_decode_step(pool, i32(r2t), i32(wl.req_pool_indices), i32(wl.seq_lens), bt,
                        to_dev(k, wl.in_dtype), to_dev(v, wl.in_dtype), i64(slots), q, out,
                        wl.max_seq_len, wl.sm_scale, num_splits, workspace, dev_err)
    return out, bt, dev_err


def _compare_pools(gpu_pool, opool):
    g = pool_to_host(gpu_pool)
    for key in ("k", "v", "k_sz", "v_sz"):
        ref = getattr(opool, key)
        if ref is not None:
            assert np.array_equal(g[key], ref), key


SMALL = {
    "cfg1": lambda: synthetic.cfg1(),
    "cfg2": lambda: synthetic.cfg2(batch=6),
    "cfg3": lambda: synthetic.cfg3(batch=3, length=1000, heads=32),
    "cfg4": lambda: synthetic.cfg4(batch=6, prefix_blocks=64),
    "cfg5": lambda: synthetic.cfg5(batch=10, chunk=512, slack_blocks=8),
}


def test_step_barrier_timeout_is_reported_and_context_survives(gpu):
    # the step's grid barrier waiting for one CTA more than the grid has: the
    # bounded wait runs out after 5 ms, sets the timeout bit and every CTA
    # returns (no fault, no hang)
    counter = torch.zeros(1, dtype=torch.int32, device="cuda")
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu.kvq_selftest_step_barrier(counter, dev_err, grid_ctas=0, limit_us=5000)
    bits = gpu.kvq_check_error(dev_err)
    assert bits == 64, bits  # KVQ_DEV_ERR_TIMEOUT alone
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    assert int(counter.item()) == n_sm  # every CTA arrived, none was waited for in vain
    # the context is still usable: a fused step right after matches the oracle
    wl = SMALL["cfg3"]()
    pool = fill_pool(wl)
    out, bt, err = fused_step(gpu, wl, pool)
    assert gpu.kvq_check_error(err) == 0
    opool, oout = oracle.run_workload(wl)
    _compare_pools(pool, opool)
    assert_close(out_to_f64(out), oout)


@pytest.mark.parametrize("name", list(SMALL))
def test_small_workloads_match_oracle_and_separate_calls(gpu, name):
    wl = SMALL[name]()
    pool = fill_pool(wl)
    out, bt, dev_err = fused_step(gpu, wl, pool)
    assert gpu.kvq_check_error(dev_err) == 0
    opool, oout = oracle.run_workload(wl)
    _compare_pools(pool, opool)
    obt, oerr = oracle.block_tables(wl.req_to_token, wl.req_pool_indices, wl.seq_lens,
                                    wl.max_blocks_per_seq)
    assert oerr == 0
    assert np.array_equal(bt.cpu().numpy(), obt)
    assert_close(out_to_f64(out), oout)
    # the same step as three calls on a second pool: same pool bytes and tables
    pool2 = fill_pool(wl)
    out2, bt2, _ = run_step(wl, pool2)
    for key in ("k", "v", "k_sz", "v_sz"):
        if getattr(pool, key) is not None:
            assert torch.equal(getattr(pool, key), getattr(pool2, key)), key
    assert torch.equal(bt, bt2)
    assert_close(out_to_f64(out), out_to_f64(out2))


@pytest.mark.parametrize("kv_dtype,dt", [("int8", "f16"), ("int8", "bf16"), ("int4", "f16"),
                                         ("int4", "bf16"), ("f16", "f16"), ("bf16", "bf16")])
@pytest.mark.parametrize("heads", [(8, 8), (16, 4), (16, 1), (32, 2)])
@pytest.mark.parametrize("splits", [0, 3])
def test_dtypes_groups_and_splits(gpu, kv_dtype, dt, heads, splits):
    Hq, Hkv = heads
    lens = [1, 15, 16, 17, 31, 33, 250, 513]
    wl = synthetic.custom(f"s_{kv_dtype}_{Hq}_{Hkv}", kv_dtype, lens, Hq, Hkv, seed=70 + Hq,
                          in_dtype=dt, q_dtype=dt)
    pool = fill_pool(wl)
    out, _, dev_err = fused_step(gpu, wl, pool, num_splits=splits)
    assert gpu.kvq_check_error(dev_err) == 0
    opool, oout = oracle.run_workload(wl)
    _compare_pools(pool, opool)
    assert out.dtype == {"f16": torch.float16, "bf16": torch.bfloat16}[dt]
    assert_close(out_to_f64(out), oout)


def test_empty_and_single_token_requests(gpu):
    wl = synthetic.custom("step_edge", "int4", [0, 1, 0, 2, 16, 17], 4, 2, seed=72)
    pool = fill_pool(wl)
    out, _, dev_err = fused_step(gpu, wl, pool)
    assert gpu.kvq_check_error(dev_err) == 0
    opool, oout = oracle.run_workload(wl)
    _compare_pools(pool, opool)
    got = out_to_f64(out)
    assert (got[0] == 0).all() and (got[2] == 0).all()
    assert_close(got, oout)


def test_repeated_calls_and_graph_replay_are_bitwise_equal(gpu):
    """The barrier counter is reset by every call, so the step replays (also
    from a CUDA graph) to the same bits."""
    wl = synthetic.cfg2(batch=12)
    pool = fill_pool(wl)
    step = gpu.DecodeStep(pool, wl.batch, wl.q_heads, wl.max_blocks_per_seq, wl.max_seq_len,
                          TORCH_DT[wl.q_dtype], fused=True)
    slots, k, v = wl.step_store()
    args = (i32(wl.req_to_token), i32(wl.req_pool_indices), i32(wl.seq_lens),
            to_dev(wl.q(), wl.q_dtype), to_dev(k, wl.in_dtype), to_dev(v, wl.in_dtype),
            i64(slots), wl.sm_scale)
    first = step(*args).clone()
    second = step(*args).clone()
    assert torch.equal(first.view(torch.int16), second.view(torch.int16))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(*args)
    for _ in range(3):
        step.out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(first.view(torch.int16), step.out.view(torch.int16))
    assert gpu.kvq_check_error(step.dev_err) == 0
    _, oout = oracle.run_workload(wl)
    assert_close(out_to_f64(first), oout)


def test_errors_match_the_separate_calls(gpu):
    """A ReqToTokenPool row that is not block-contiguous and one whose block
    lies past the pool: the step completes, flags what the three calls flag
    and leaves finite outputs."""
    wl = synthetic.custom("step_errs", "int8", [20, 40, 70], 4, 2, seed=73)
    r2t = wl.req_to_token.copy()
    row1, row2 = int(wl.req_pool_indices[1]), int(wl.req_pool_indices[2])
    r2t[row1, 17] = r2t[row1, 16] + 5                              # not block-contiguous
    r2t[row2, 32:48] = (wl.num_blocks + 2) * 16 + np.arange(16)   # a block past the pool
    pool = fill_pool(wl)
    out, _, dev_err = fused_step(gpu, wl, pool, req_to_token=r2t)
    bits = gpu.kvq_check_error(dev_err)
    _, oerr = oracle.block_tables(r2t, wl.req_pool_indices, wl.seq_lens, wl.max_blocks_per_seq)
    assert oerr != 0 and bits & oerr == oerr
    assert bits & gpu.DEV_ERR_BITS["block_id"]
    assert torch.isfinite(out.float()).all()
    # the three calls flag the same bits on a fresh error word
    pool2 = fill_pool(wl)
    dev_err2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    bt2 = torch.empty((wl.batch, wl.max_blocks_per_seq), dtype=torch.int32, device="cuda")
    gpu.kvq_block_tables_from_req_to_token(i32(r2t), i32(wl.req_pool_indices),
                                           i32(wl.seq_lens), bt2, dev_err2)
    slots, k, v = wl.step_store()
    gpu.kv_store_quant(pool2, to_dev(k, wl.in_dtype), to_dev(v, wl.in_dtype), i64(slots),
                       dev_err2)
    q = to_dev(wl.q(), wl.q_dtype)
    out2 = torch.empty_like(q)
    ws = gpu.paged_decode_attn_workspace_size(wl.batch, wl.q_heads, wl.kv_heads, wl.max_seq_len)
    gpu.paged_decode_attn(pool2, q, out2, bt2, i32(wl.seq_lens), wl.max_seq_len, wl.sm_scale,
                          0, torch.empty(ws, dtype=torch.uint8, device="cuda"), dev_err2)
    assert gpu.kvq_check_error(dev_err2) == bits
    # the request without a bad row attends as the oracle does
    _, oout = oracle.run_workload(wl)
    assert_close(out_to_f64(out)[0], oout[0])


def test_no_requests_stores_only(gpu):
    """A step with no requests still stores its tokens."""
    wl = synthetic.custom("step_store_only", "int4", [40], 4, 2, seed=74)
    pool = gpu.KVPool.allocate(wl.num_blocks, wl.kv_heads, wl.kv_dtype)
    slots, k, v = wl.step_store()
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    empty = torch.empty(0, dtype=torch.int32, device="cuda")
    q = torch.empty((0, wl.q_heads, 128), dtype=torch.float16, device="cuda")
    gpu.kvq_decode_step(pool, i32(wl.req_to_token), empty, empty,
                        torch.empty((0, wl.max_blocks_per_seq), dtype=torch.int32,
                                    device="cuda"),
                        to_dev(k, wl.in_dtype), to_dev(v, wl.in_dtype), i64(slots), q,
                        torch.empty_like(q), wl.max_seq_len, wl.sm_scale, 0, None, dev_err)
    assert gpu.kvq_check_error(dev_err) == 0
    opool = oracle.Pool(wl.num_blocks, wl.kv_heads, 128, wl.kv_dtype)
    oracle.kv_store(opool, k, v, wl.in_dtype, slots)
    _compare_pools(pool, opool)


def test_mixed_dtypes_are_refused(gpu):
    wl = synthetic.custom("step_mixed", "int8", [20], 4, 2, seed=75, in_dtype="f16",
                          q_dtype="bf16")
    pool = fill_pool(wl)
    with pytest.raises(ValueError):
        fused_step(gpu, wl, pool)


FULL = ["cfg1", "cfg2", "cfg3", "cfg4", "cfg5"]


@pytest.mark.slow
@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(gpu, name):
    wl = synthetic.by_name(name)
    pool = fill_pool(wl)
    out, bt, dev_err = fused_step(gpu, wl, pool)
    assert gpu.kvq_check_error(dev_err) == 0
    obt, oerr = oracle.block_tables(wl.req_to_token, wl.req_pool_indices, wl.seq_lens,
                                    wl.max_blocks_per_seq)
    assert oerr == 0 and np.array_equal(bt.cpu().numpy(), obt)
    got = out_to_f64(out)
    lens = wl.seq_lens
    picks = sorted({0, wl.batch - 1, int(lens.argmax()), int(lens.argmin()), wl.batch // 2})
    for b in picks:
        opool, oout = oracle_request(wl, b)
        g = gpu_request_rows(wl, pool, b)
        o = oracle_request_rows(opool, int(lens[b]))
        for key in o:
            assert np.array_equal(g[key], o[key]), (name, b, key)
        assert_close(got[b], oout)
