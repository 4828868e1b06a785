"""Pins for the oracle's store (quantizing scatter) and block-table builder.

"pymllm Runtime Design", section "KV cache 与 prefix cache": ReqToTokenPool
maps (request slot, position) to a kv index, and KVPool rows are written by a
store kernel. LMDeploy article §2.2: blocks of 16 tokens, per-sequence tables
of physical block ids; the pool shape is [num_blocks, block_size, kv_heads,
head_dim].
"""
import json
import os

import numpy as np
import pytest

import oracle
import synthetic

GOLDEN_DIR = os.path.join(os.path.dirname(__file__), "golden")


@pytest.mark.parametrize("kv_dtype", ["int8", "int4", "f16", "bf16"])
def test_scatter_lands_rows_at_their_slots(kv_dtype):
    Hkv, D, nb = 3, 128, 7
    in_dtype = "bf16" if kv_dtype == "bf16" else "f16"
    slots = np.array([5, 111, 16, -1, 0, 47, 200, 15], dtype=np.int64)  # 200 is past the pool
    N = slots.size
    k = synthetic.normal(31, 1, 0, N * Hkv * D, dtype=in_dtype).reshape(N, Hkv, D)
    v = synthetic.normal(31, 2, 0, N * Hkv * D, dtype=in_dtype).reshape(N, Hkv, D)
    pool = oracle.Pool(nb, Hkv, D, kv_dtype)
    bad = oracle.kv_store(pool, k, v, in_dtype, slots)
    assert bad == 1
    touched = np.zeros((nb, 16), bool)
    for t, s in enumerate(slots):
        if s < 0 or s >= nb * 16:
            continue
        blk, off = divmod(int(s), 16)
        touched[blk, off] = True
        for which, src, arr, sz in (("k", k, pool.k, pool.k_sz), ("v", v, pool.v, pool.v_sz)):
            row = arr[blk, off]  # [Hkv, row_bytes], read by plain indexing
            if kv_dtype in ("f16", "bf16"):
                assert np.array_equal(row.view(np.uint16), src[t])
                continue
            x = oracle.to_f32(src[t], in_dtype)
            codes, sb, zb = oracle.quantize_rows(x, 8 if kv_dtype == "int8" else 4)
            if kv_dtype == "int8":
                assert np.array_equal(row, codes)
            else:
                assert np.array_equal(row & 0xF, codes[:, 0::2])
                assert np.array_equal(row >> 4, codes[:, 1::2])
            assert np.array_equal(sz[blk, :, off, 0], sb)
            assert np.array_equal(sz[blk, :, off, 1], zb)
    # untouched slots stay zero
    assert not pool.k[~touched].any() and not pool.v[~touched].any()


def test_int4_packing_matches_golden_bytes():
    with open(os.path.join(GOLDEN_DIR, "quant_rows.json")) as f:
        cases = [c for c in json.load(f)["cases"] if c["bits"] == 4]
    for c in cases:
        x = np.full(128, c["x_fill"], dtype=np.float32)
        x[: len(c["x_prefix"])] = c["x_prefix"]
        bits = x.astype(np.float16).view(np.uint16).reshape(1, 1, 128)
        pool = oracle.Pool(1, 1, 128, "int4")
        oracle.kv_store(pool, bits, bits, "f16", np.array([3], np.int64))
        row = pool.k[0, 3, 0]
        want = np.full(64, int(c["packed_fill"], 16), dtype=np.uint8)
        want[: len(c["packed_prefix"])] = [int(b, 16) for b in c["packed_prefix"]]
        assert np.array_equal(row, want), c["name"]


def test_block_tables_hand_example():
    with open(os.path.join(GOLDEN_DIR, "block_tables.json")) as f:
        g = json.load(f)
    for case in g["cases"]:
        r2t = np.array(case["req_to_token"], dtype=np.int32)
        bt, err = oracle.block_tables(r2t, np.array(case["req_pool_indices"], np.int32),
                                      np.array(case["seq_lens"], np.int32),
                                      case["max_blocks_per_seq"])
        assert err == case["error_mask"], case["name"]
        if "block_tables" in case:
            assert bt.tolist() == case["block_tables"], case["name"]


@pytest.mark.parametrize("name", ["cfg1", "cfg2", "cfg4", "cfg5"])
def test_block_tables_recover_workload_tables(name):
    wl = synthetic.by_name(name)
    bt, err = oracle.block_tables(wl.req_to_token, wl.req_pool_indices, wl.seq_lens,
                                  wl.max_blocks_per_seq)
    assert err == 0
    assert np.array_equal(bt, wl.block_tables)
