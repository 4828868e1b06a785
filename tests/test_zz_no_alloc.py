"""paged_decode_attn_noalloc: decode attention without a caller workspace.

Some callers cannot allocate device memory (an operator inside an engine that
only receives its tensors, a program that reserves all device memory at load
time, a loop where an allocation is not acceptable). For them libkvq keeps the
split-K scratch in a fixed array of its own. These tests call that entry point
through the C ABI and check that two calls in a row, with different sizes,
give the same outputs as paged_decode_attn with a caller-allocated workspace,
within the tolerance of the other parity tests. This file sorts last so that
a run stopping at its first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import synthetic

pytestmark = pytest.mark.gpu

from gpu_harness import assert_close, decode, fill_pool, i32, out_to_f64, run_step, to_dev  # noqa: E402

SCRATCH_BYTES = 16 * 1024 * 1024
PART_STRIDE = 132  # floats per partial record (128 outputs, max, sum, padding)
HDR_CUM = 5        # ints before the per-request prefix sums in the header


def _static_bytes(kvq, batch, q_heads, kv_heads, max_len, splits=0):
    """Scratch the static ranges alone need: counters, the length header and
    one record slot (2 rows per q head of a group slot) per warp of the plan."""
    plan = kvq.paged_decode_attn_plan(batch, q_heads, kv_heads, max_len, splits)
    records_off = 256 + ((batch + HDR_CUM + 1) * 4 + 255) // 256 * 256
    return records_off + plan["warps"] * 2 * plan["heads_per_group"] * PART_STRIDE * 4


def _noalloc(kvq, wl, pool, bt, num_splits=0):
    q = to_dev(wl.q(), wl.q_dtype)
    out = torch.full_like(q, float("nan"))
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.paged_decode_attn_noalloc(pool, q, out, bt, i32(wl.seq_lens), wl.max_seq_len,
                                  wl.sm_scale, num_splits, dev_err)
    assert kvq.kvq_check_error(dev_err) == 0
    return out


def test_two_calls_match_the_workspace_entry_point(gpu):
    # two different shapes back to back: the second call sees the first
    # call's leftovers in the shared scratch
    cases = [
        (synthetic.cfg4(batch=12), 0),
        (synthetic.custom("noalloc_int8", "int8", [700, 33, 1500, 5, 260], 16, 4, seed=90), 5),
    ]
    for wl, splits in cases:
        pool = fill_pool(wl)
        ref, bt, dev_err = run_step(wl, pool, num_splits=splits)
        assert gpu.kvq_check_error(dev_err) == 0
        assert gpu.paged_decode_attn_workspace_size(
            wl.batch, wl.q_heads, wl.kv_heads, wl.max_seq_len, splits) > 0  # scratch is used
        got = _noalloc(gpu, wl, pool, bt, splits)
        assert_close(out_to_f64(got), out_to_f64(ref))
        # a repeated call gives the same bits
        again = _noalloc(gpu, wl, pool, bt, splits)
        assert torch.equal(got.view(torch.int16), again.view(torch.int16))


def test_long_gqa_contexts_run_without_the_tail(gpu):
    # 4 q heads per kv head over long contexts: the array holds the static
    # ranges but not the balanced tail's records, so this entry point runs
    # the static cut while paged_decode_attn (full workspace) uses the tail
    lens = [8192 + 64 * i for i in range(64)]
    wl = synthetic.custom("noalloc_gqa_long", "int4", lens, 32, 8, seed=92)
    full = gpu.paged_decode_attn_workspace_size(wl.batch, wl.q_heads, wl.kv_heads,
                                                wl.max_seq_len, 0)
    static = _static_bytes(gpu, wl.batch, wl.q_heads, wl.kv_heads, wl.max_seq_len)
    assert static <= SCRATCH_BYTES < full
    pool = fill_pool(wl)
    ref, bt, dev_err = run_step(wl, pool)
    assert gpu.kvq_check_error(dev_err) == 0
    for _ in range(2):
        got = _noalloc(gpu, wl, pool, bt)
        assert_close(out_to_f64(got), out_to_f64(ref))


def test_sizes_beyond_the_scratch_are_rejected(gpu):
    # 8 q heads per kv head need 8 partial rows per warp slot: more than the array holds
    wl = synthetic.custom("noalloc_big", "int8", [16], 64, 8, seed=91)
    pool = gpu.KVPool.allocate(wl.num_blocks, wl.kv_heads, "int8")
    batch, q_heads, max_len = 8, 64, 4096
    # the entry point refuses a size when the static ranges alone do not fit
    assert _static_bytes(gpu, batch, q_heads, 8, max_len) > SCRATCH_BYTES
    q = torch.zeros((batch, q_heads, 128), dtype=torch.float16, device="cuda")
    out = torch.zeros_like(q)
    bt = torch.zeros((batch, max_len // 16), dtype=torch.int32, device="cuda")
    sl = torch.ones(batch, dtype=torch.int32, device="cuda")
    with pytest.raises(gpu.KvqError) as e:
        gpu.paged_decode_attn_noalloc(pool, q, out, bt, sl, max_len, 0.1)
    assert e.value.status == 5
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0  # nothing was launched
