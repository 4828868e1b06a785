"""Whole-pool bit-exactness of the quantizing store at full size.

"pymllm Runtime Design", section "KV cache 与 prefix cache": the store
kernel writes every new token's K/V rows into its pool slot; LMDeploy article
§2.4: INT8/INT4 KV quantized per token and head, min/max online. For each
workload at its full size the whole context is stored through the C ABI
(setup chunks, then the step's own tokens, as the benchmark does), and then
every stored row -- each request's positions read back through its block
table, the shared prefix through every member, and the mixed step's prefill
chunk -- is compared bit for bit (codes, fp16 scale and zero, or the 16-bit
elements of unquantized pools) with the oracle's store of the same
regenerated inputs, request by request.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

from gpu_harness import fill_pool, gpu_request_rows, oracle_request_rows, run_step  # noqa: E402


def _oracle_store_request(wl, b):
    """Compact oracle pool holding request b's rows at positions 0..L-1."""
    L = int(wl.seq_lens[b])
    pool = oracle.Pool(max(1, (L + 15) // 16), wl.kv_heads, wl.head_dim, wl.kv_dtype)
    if L > 0:
        bad = oracle.kv_store(pool, wl.ctx_rows("k", b, 0, L), wl.ctx_rows("v", b, 0, L),
                              wl.in_dtype, np.arange(L, dtype=np.int64))
        assert bad == 0
    return pool


@pytest.mark.parametrize("name", ["cfg1", "cfg2", "cfg3", "cfg4", "cfg5"])
def test_every_stored_row_matches_the_oracle(gpu, name):
    wl = synthetic.by_name(name)
    pool = fill_pool(wl, max_tokens=1 << 17)
    _, _, dev_err = run_step(wl, pool)  # the step's own stores
    assert gpu.kvq_check_error(dev_err) == 0
    rows = 0
    for b in range(wl.batch):
        L = int(wl.seq_lens[b])
        if L == 0:
            continue
        g = gpu_request_rows(wl, pool, b)
        o = oracle_request_rows(_oracle_store_request(wl, b), L)
        for key in o:
            assert np.array_equal(g[key], o[key]), (name, b, key)
        rows += L
    assert rows == int(np.sum(wl.seq_lens))
    if wl.chunk_slots is not None:  # the mixed step's prefill chunk, block by block
        slots, k, v = wl.step_store()
        n = len(wl.chunk_slots)
        opool = oracle.Pool(wl.num_blocks, wl.kv_heads, wl.head_dim, wl.kv_dtype)
        assert oracle.kv_store(opool, k[:n], v[:n], wl.in_dtype, slots[:n]) == 0
        blk = np.unique(slots[:n] // 16)
        bidx = torch.from_numpy(blk).cuda()
        for key in ("k", "v", "k_sz", "v_sz"):
            if getattr(opool, key) is None:
                continue
            got = getattr(pool, key)[bidx].cpu().numpy()
            if key.endswith("_sz"):
                got = got.view(np.uint16).reshape(got.shape + (2,))
            assert np.array_equal(got, getattr(opool, key)[blk]), key
