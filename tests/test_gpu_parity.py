"""GPU parity: libkvq (through its C ABI) against the CPU oracle.

Store path: codes, scales and zeros must be bit-exact. Block tables: bit-exact.
Decode attention: every output element within 2e-3 absolute or 1e-2 relative
of the oracle's fp64 result on the same stored values.

Sizes: reduced versions of the five workloads that the oracle finishes in
seconds (whole pools and every output compared), plus the full-size
workloads with the oracle run on sampled requests.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic

pytestmark = pytest.mark.gpu

from gpu_harness import (assert_close, decode, fill_pool, gpu_request_rows, i32, i64,  # noqa: E402
                         oracle_request, oracle_request_rows, out_to_f64, pool_to_host,
                         run_step, to_dev)

SMALL = {
    "cfg1": lambda: synthetic.cfg1(),
    "cfg2": lambda: synthetic.cfg2(batch=6),
    "cfg3": lambda: synthetic.cfg3(batch=3, length=1000, heads=32),
    "cfg4": lambda: synthetic.cfg4(batch=6, prefix_blocks=64),
    "cfg5": lambda: synthetic.cfg5(batch=10, chunk=512, slack_blocks=8),
}


def _compare_pools(gpu_pool, opool):
    g = pool_to_host(gpu_pool)
    assert np.array_equal(g["k"], opool.k), "K codes/elements differ"
    assert np.array_equal(g["v"], opool.v), "V codes/elements differ"
    if opool.k_sz is not None:
        assert np.array_equal(g["k_sz"], opool.k_sz), "K scale/zero differ"
        assert np.array_equal(g["v_sz"], opool.v_sz), "V scale/zero differ"


@pytest.mark.parametrize("name", list(SMALL))
def test_small_workload_store_tables_decode(gpu, name):
    wl = SMALL[name]()
    pool = fill_pool(wl)
    out, bt, dev_err = run_step(wl, pool)
    assert gpu.kvq_check_error(dev_err) == 0
    opool, oout = oracle.run_workload(wl)
    _compare_pools(pool, opool)
    obt, oerr = oracle.block_tables(wl.req_to_token, wl.req_pool_indices, wl.seq_lens,
                                    wl.max_blocks_per_seq)
    assert oerr == 0
    assert np.array_equal(bt.cpu().numpy(), obt)
    assert_close(out_to_f64(out), oout)


@pytest.mark.parametrize("name", ["cfg2", "cfg4"])
@pytest.mark.parametrize("splits", [1, 2, 3, 7, 0])
def test_split_counts_agree(gpu, name, splits):
    wl = SMALL[name]()
    pool = fill_pool(wl)
    out, _, dev_err = run_step(wl, pool, num_splits=splits)
    assert gpu.kvq_check_error(dev_err) == 0
    _, oout = oracle.run_workload(wl)
    assert_close(out_to_f64(out), oout)


@pytest.mark.parametrize("kv_dtype,in_dtype", [("int8", "f16"), ("int4", "f16"),
                                               ("int8", "bf16"), ("int4", "bf16"),
                                               ("f16", "f16"), ("bf16", "bf16")])
@pytest.mark.parametrize("heads", [(8, 8), (16, 4), (12, 4), (16, 1), (32, 2), (64, 16)])
def test_dtypes_and_groups(gpu, kv_dtype, in_dtype, heads):
    Hq, Hkv = heads
    lens = [1, 15, 16, 17, 31, 33, 250, 513]
    wl = synthetic.custom(f"g_{kv_dtype}_{Hq}_{Hkv}", kv_dtype, lens, Hq, Hkv, seed=40 + Hq,
                          in_dtype=in_dtype)
    pool = fill_pool(wl)
    out, _, dev_err = run_step(wl, pool, num_splits=2)
    assert gpu.kvq_check_error(dev_err) == 0
    opool, oout = oracle.run_workload(wl)
    _compare_pools(pool, opool)
    assert_close(out_to_f64(out), oout)


@pytest.mark.parametrize("kv_dtype,q_dtype", [("int8", "f16"), ("int4", "f16"),
                                               ("int4", "bf16")])
def test_long_context_with_outlier_channels(gpu, kv_dtype, q_dtype):
    """Long contexts and x8 outlier channels stress the accumulation of the
    code offsets and the 16-bit rounding of p * scale."""
    wl = synthetic.custom("long_outliers", kv_dtype, [4096, 3001, 17, 2048], 8, 2, seed=55,
                          q_dtype=q_dtype, outliers=True)
    pool = fill_pool(wl)
    out, _, dev_err = run_step(wl, pool)
    assert gpu.kvq_check_error(dev_err) == 0
    opool, oout = oracle.run_workload(wl)
    _compare_pools(pool, opool)
    assert_close(out_to_f64(out), oout)


@pytest.mark.parametrize("kv_dtype", ["int8", "int4"])
def test_bf16_queries_over_quantized_pool(gpu, kv_dtype):
    wl = synthetic.custom("bfq", kv_dtype, [40, 300, 77], 8, 2, seed=51, in_dtype="f16",
                          q_dtype="bf16")
    pool = fill_pool(wl)
    out, _, dev_err = run_step(wl, pool)
    assert gpu.kvq_check_error(dev_err) == 0
    _, oout = oracle.run_workload(wl)
    assert out.dtype == torch.bfloat16
    assert_close(out_to_f64(out), oout)


def test_empty_and_single_token_requests(gpu):
    wl = synthetic.custom("edge", "int8", [0, 1, 0, 2, 16], 4, 2, seed=52)
    pool = fill_pool(wl)
    out, _, dev_err = run_step(wl, pool, num_splits=0)
    assert gpu.kvq_check_error(dev_err) == 0
    _, oout = oracle.run_workload(wl)
    got = out_to_f64(out)
    assert (got[0] == 0).all() and (got[2] == 0).all()
    assert_close(got, oout)


@pytest.mark.parametrize("kv_dtype", ["int8", "int4", "f16"])
def test_block_permutation_is_bitwise_invariant(gpu, kv_dtype):
    wl = synthetic.custom("perm", kv_dtype, [3, 40, 97, 160, 700], 8, 4, seed=53)
    pool = fill_pool(wl)
    out, bt, _ = run_step(wl, pool, num_splits=3)
    perm = torch.from_numpy(synthetic.permutation(77, 1, wl.num_blocks)).cuda()
    pool2 = type(pool).allocate(wl.num_blocks, wl.kv_heads, wl.kv_dtype)
    pool2.k[perm] = pool.k
    pool2.v[perm] = pool.v
    if pool.k_sz is not None:
        pool2.k_sz[perm] = pool.k_sz
        pool2.v_sz[perm] = pool.v_sz
    bt2 = torch.where(bt >= 0, perm[bt.clamp(min=0).long()].int(), bt)
    out2 = decode(wl, pool2, bt2, num_splits=3)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


def test_shared_prefix_equals_duplicated_prefix(gpu):
    wl = synthetic.cfg4(batch=5)
    pool = fill_pool(wl)
    out, _, _ = run_step(wl, pool)
    # a second pool where each request owns a private copy of the prefix
    k = wl.shared_tokens // 16
    extra = int(k.sum())
    pool2 = type(pool).allocate(wl.num_blocks + extra, wl.kv_heads, wl.kv_dtype)
    pool2.k[:wl.num_blocks] = pool.k
    pool2.v[:wl.num_blocks] = pool.v
    pool2.k_sz[:wl.num_blocks] = pool.k_sz
    pool2.v_sz[:wl.num_blocks] = pool.v_sz
    bt2 = wl.block_tables.copy()
    nxt = wl.num_blocks
    for b in range(wl.batch):
        for j in range(int(k[b])):
            src = int(bt2[b, j])
            pool2.k[nxt] = pool.k[src]
            pool2.v[nxt] = pool.v[src]
            pool2.k_sz[nxt] = pool.k_sz[src]
            pool2.v_sz[nxt] = pool.v_sz[src]
            bt2[b, j] = nxt
            nxt += 1
    out2 = decode(wl, pool2, i32(bt2))
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


def test_uniform_k_gives_mean_of_v(gpu):
    L, D = 300, 128
    wl = synthetic.custom("uni", "int8", [L], 4, 1, seed=54)
    pool = gpu.KVPool.allocate(wl.num_blocks, 1, "int8")
    pos = np.arange(L)
    slots = wl.block_tables[0, pos // 16].astype(np.int64) * 16 + pos % 16
    k = np.full((L, 1, D), np.float16(0.7).view(np.uint16), dtype=np.uint16)
    v = synthetic.normal(54, 9, 0, L * D).reshape(L, 1, D)
    gpu.kv_store_quant(pool, to_dev(k, "f16"), to_dev(v, "f16"), i64(slots))
    out = decode(wl, pool, i32(wl.block_tables), num_splits=0)
    opool = oracle.Pool(wl.num_blocks, 1, D, "int8")
    oracle.kv_store(opool, k, v, "f16", slots)
    rows = opool.v.reshape(-1, 1, D)[slots].astype(np.float64)[:, 0]
    sz = opool.v_sz[slots // 16, 0, slots % 16]
    vhat = rows * oracle.f16_to_f32(sz[:, 0])[:, None] + oracle.f16_to_f32(sz[:, 1])[:, None]
    for h in range(4):
        assert_close(out_to_f64(out)[0, h], vhat.mean(axis=0))


def test_store_random_token_slots(gpu):
    """Token-granular random slots (not block-contiguous), both quantized kinds."""
    rng_slots = synthetic.permutation(60, 3, 100 * 16)[:1500].astype(np.int64)
    rng_slots[::97] = -1  # padding tokens are skipped
    N, Hkv, D = rng_slots.size, 4, 128
    for kv_dtype in ("int8", "int4"):
        k = synthetic.normal(60, 4, 0, N * Hkv * D, scale=3.0).reshape(N, Hkv, D)
        v = synthetic.normal(60, 5, 0, N * Hkv * D, scale=0.01).reshape(N, Hkv, D)
        pool = gpu.KVPool.allocate(100, Hkv, kv_dtype)
        gpu.kv_store_quant(pool, to_dev(k, "f16"), to_dev(v, "f16"), i64(rng_slots))
        opool = oracle.Pool(100, Hkv, D, kv_dtype)
        oracle.kv_store(opool, k, v, "f16", rng_slots)
        _compare_pools(pool, opool)


def test_device_errors_are_reported_not_trapped(gpu):
    wl = synthetic.custom("errs", "int8", [20, 40], 4, 2, seed=61)
    pool = fill_pool(wl)
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    # a slot past the pool is skipped and flagged
    k = to_dev(synthetic.normal(61, 1, 0, 2 * 2 * 128).reshape(2, 2, 128), "f16")
    before = pool.k.clone()
    gpu.kv_store_quant(pool, k, k, i64([wl.num_blocks * 16 + 5, -1]), dev_err)
    assert gpu.kvq_check_error(dev_err) == gpu.DEV_ERR_BITS["slot"]
    assert torch.equal(before, pool.k)
    # a block id outside the pool is skipped and flagged; the step completes
    bt = wl.block_tables.copy()
    bt[1, 1] = wl.num_blocks + 100
    out = decode(wl, pool, i32(bt), dev_err=dev_err)
    assert gpu.kvq_check_error(dev_err) == gpu.DEV_ERR_BITS["block_id"]
    assert torch.isfinite(out.float()).all()
    # a length past the table is clamped and flagged
    out = decode(wl, pool, i32(wl.block_tables), dev_err=dev_err,
                 seq_lens=i32([20, 40 + 16 * 8]), max_seq_len=40)
    assert gpu.kvq_check_error(dev_err) & gpu.DEV_ERR_BITS["length"]


def test_block_table_errors_match_oracle(gpu):
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", "block_tables.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        r2t = np.array(c["req_to_token"], np.int32)
        rpi = np.array(c["req_pool_indices"], np.int32)
        sl = np.array(c["seq_lens"], np.int32)
        bt = torch.full((len(sl), c["max_blocks_per_seq"]), 7, dtype=torch.int32, device="cuda")
        dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
        gpu.kvq_block_tables_from_req_to_token(i32(r2t), i32(rpi), i32(sl), bt, dev_err)
        bits = gpu.kvq_check_error(dev_err)
        obt, oerr = oracle.block_tables(r2t, rpi, sl, c["max_blocks_per_seq"])
        assert bits == oerr == c["error_mask"], c["name"]
        assert np.array_equal(bt.cpu().numpy(), obt), c["name"]


# ---- full-size workloads, oracle on sampled requests ---------------------------

FULL = ["cfg1", "cfg2", "cfg3", "cfg4", "cfg5"]


@pytest.mark.slow
@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(gpu, name):
    wl = synthetic.by_name(name)
    pool = fill_pool(wl)
    out, bt, dev_err = run_step(wl, pool)  # the launch configuration the bench times
    assert gpu.kvq_check_error(dev_err) == 0
    obt, oerr = oracle.block_tables(wl.req_to_token, wl.req_pool_indices, wl.seq_lens,
                                    wl.max_blocks_per_seq)
    assert oerr == 0 and np.array_equal(bt.cpu().numpy(), obt)
    got = out_to_f64(out)
    # sampled requests: the first, the last, the longest, the shortest and two more
    lens = wl.seq_lens
    picks = sorted({0, wl.batch - 1, int(lens.argmax()), int(lens.argmin()),
                    wl.batch // 3, (2 * wl.batch) // 3})
    for b in picks:
        opool, oout = oracle_request(wl, b)
        L = int(lens[b])
        g = gpu_request_rows(wl, pool, b)
        o = oracle_request_rows(opool, L)
        for key in o:
            assert np.array_equal(g[key], o[key]), (name, b, key)
        assert_close(got[b], oout)
    if wl.chunk_slots is not None:  # the prefill chunk of the mixed step
        slots, k, v = wl.step_store()
        n = len(wl.chunk_slots)
        opool = oracle.Pool(wl.num_blocks, wl.kv_heads, wl.head_dim, wl.kv_dtype)
        oracle.kv_store(opool, k[:n], v[:n], wl.in_dtype, slots[:n])
        blk = np.unique(slots[:n] // 16)
        bidx = torch.from_numpy(blk).cuda()
        for key in ("k", "v", "k_sz", "v_sz"):
            g = getattr(pool, key)[bidx].cpu().numpy()
            if key.endswith("_sz"):
                g = g.view(np.uint16).reshape(g.shape + (2,))
            assert np.array_equal(g, getattr(opool, key)[blk]), key


def _near_tie_rows(kv_dtype, in_dtype, n_rows, seed):
    """Rows whose codes (x - Z) / S sit on or next to rounding ties k + 1/2:
    each row's min and max set the scale, the other 126 elements are the
    representable inputs in between whose quotients are nearest a tie."""
    qmax = 255 if kv_dtype == "int8" else 15
    bits = np.arange(65536, dtype=np.uint32)
    if in_dtype == "f16":
        with np.errstate(invalid="ignore"):
            vals = bits.astype(np.uint16).view(np.float16).astype(np.float32)
    else:
        vals = (bits << 16).view(np.float32)
    ok = np.isfinite(vals)
    rng = np.random.default_rng(seed)
    rows = np.empty((n_rows, 128), np.uint16)
    for r in range(n_rows):
        if r == 0:
            mn, mx = 0.0, float(qmax)  # S = 1: exact ties
        else:
            mn = float(rng.uniform(-4, 1))
            mx = mn + float(rng.uniform(0.01, 8))
        sel = ok & (vals >= mn) & (vals <= mx)
        cand, cbits = vals[sel], bits[sel].astype(np.uint16)
        lo, hi = cand.min(), cand.max()
        S = np.float32(np.float16(np.float32(np.float32(hi) - np.float32(lo)) / np.float32(qmax)))
        Z = np.float32(np.float16(lo))
        q = (cand.astype(np.float64) - float(Z)) / float(S)
        dist = np.abs(q - np.floor(q) - 0.5)
        pick = np.resize(cbits[np.argsort(dist, kind="stable")], 126)  # repeats in a narrow range
        rows[r] = np.concatenate([[cbits[cand.argmin()], cbits[cand.argmax()]], pick])
    return rows


@pytest.mark.parametrize("kv_dtype", ["int8", "int4"])
@pytest.mark.parametrize("in_dtype", ["f16", "bf16"])
def test_store_rounding_ties(gpu, kv_dtype, in_dtype):
    """Inputs on and next to rounding ties: the stored codes must equal the
    oracle's (a correctly rounded fp32 division, round half to even)."""
    N, Hkv = 48, 2
    rows = _near_tie_rows(kv_dtype, in_dtype, 2 * N * Hkv, seed=81)
    k = rows[:N * Hkv].reshape(N, Hkv, 128)
    v = rows[N * Hkv:].reshape(N, Hkv, 128)
    slots = np.arange(N, dtype=np.int64) * 3 % (4 * 16)
    pool = gpu.KVPool.allocate(4, Hkv, kv_dtype)
    gpu.kv_store_quant(pool, to_dev(k, in_dtype), to_dev(v, in_dtype), i64(slots))
    opool = oracle.Pool(4, Hkv, 128, kv_dtype)
    oracle.kv_store(opool, k, v, in_dtype, slots)
    _compare_pools(pool, opool)


@pytest.mark.slow
@pytest.mark.parametrize("kv_dtype", ["int8", "int4", "bf16", "f16"])
def test_balanced_tail_on_long_contexts(gpu, kv_dtype):
    """Per-warp shares above 128 blocks: the decode hands the last tenth of
    the stream out in chunks (tail). Same outputs as the oracle, and as the
    static split (a workspace that holds one range per warp) and an explicit
    split count, both of which run without the tail."""
    wl = synthetic.custom(f"tail_{kv_dtype}", kv_dtype, [49152, 20000, 49152, 33333], 48, 48,
                          seed=58)
    pool = fill_pool(wl)
    out, bt, dev_err = run_step(wl, pool)
    assert gpu.kvq_check_error(dev_err) == 0
    got = out_to_f64(out)
    for b in range(wl.batch):
        _, oout = oracle_request(wl, b)
        assert_close(got[b], oout)
    plan = gpu.paged_decode_attn_plan(wl.batch, wl.q_heads, wl.kv_heads, wl.max_seq_len)
    static = (256 + -(-(wl.batch + 6) * 4 // 256) * 256
              + plan["warps"] * 2 * plan["heads_per_group"] * 132 * 4)
    assert static < plan["workspace_bytes"]
    q = to_dev(wl.q(), wl.q_dtype)
    for ws_bytes, splits in ((static, 0), (plan["workspace_bytes"], 3)):
        out2 = torch.empty_like(q)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        gpu.paged_decode_attn(pool, q, out2, bt, i32(wl.seq_lens), wl.max_seq_len, wl.sm_scale,
                              splits, ws, dev_err)
        assert gpu.kvq_check_error(dev_err) == 0
        assert_close(out_to_f64(out2), got)
    small = torch.empty(static - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(gpu.KvqError):
        gpu.paged_decode_attn(pool, q, torch.empty_like(q), bt, i32(wl.seq_lens),
                              wl.max_seq_len, wl.sm_scale, 0, small, dev_err)
    # a chunk's result does not depend on the warp that takes it, and every
    # call resets the chunk counter: repeated calls and CUDA-graph replays
    # give the same bits
    ws = torch.empty(plan["workspace_bytes"], dtype=torch.uint8, device="cuda")
    sl = i32(wl.seq_lens)
    first = torch.empty_like(q)
    gpu.paged_decode_attn(pool, q, first, bt, sl, wl.max_seq_len, wl.sm_scale, 0, ws, dev_err)
    assert torch.equal(first.view(torch.int16), out.view(torch.int16))
    again = torch.empty_like(q)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        gpu.paged_decode_attn(pool, q, again, bt, sl, wl.max_seq_len, wl.sm_scale, 0, ws,
                              dev_err)
    for _ in range(3):
        again.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(again.view(torch.int16), first.view(torch.int16))
    assert gpu.kvq_check_error(dev_err) == 0
