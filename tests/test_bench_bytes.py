"""The roofline's numerator: bench.py's algorithmic and logical byte counts
per decode call, pinned to closed forms of the pool layout (a 16-token block
of one kv head holds 16 rows of codes or elements for K and for V, plus a
4-byte scale/zero pair per row for the quantized kinds) and to the sharing
structure of the shared-prefix workload. No GPU involved."""
import numpy as np

import bench
import synthetic


def _closed_form(batch, tokens_per_request, q_heads, kv_heads, row_bytes, quantized):
    per_token = 2 * kv_heads * (row_bytes + (4 if quantized else 0))
    kv = batch * tokens_per_request * per_token
    q_and_out = 2 * batch * q_heads * 128 * 2
    tables = 4 * batch * (-(-tokens_per_request // 16))
    lengths = 4 * batch
    return kv + q_and_out + tables + lengths


def test_int8_mha_headline_bytes():
    wl = synthetic.cfg3()
    want = _closed_form(128, 4096, 32, 32, 128, True)
    assert want == 4431413760  # the figure the roofline divides by
    assert bench.decode_algorithmic_bytes(wl) == want
    assert bench.decode_logical_bytes(wl) == want


def test_per_token_bytes_by_kind():
    for kind, row in (("int8", 128), ("int4", 64), ("f16", 256), ("bf16", 256)):
        wl = synthetic.custom("bytes_" + kind, kind, [33, 100], 8, 2, seed=3)
        quant = kind in ("int8", "int4")
        assert wl.kv_token_bytes() == 2 * 2 * (row + (4 if quant else 0))
        want = (133 * wl.kv_token_bytes() + 2 * 2 * 8 * 128 * 2 + 4 * (3 + 7) + 4 * 2)
        assert bench.decode_algorithmic_bytes(wl) == want


def test_shared_prefix_is_counted_once():
    """Logical bytes count a shared block for every request that reads it,
    algorithmic bytes once: the difference is (readers - 1) x the prefix's
    tokens for each shared block."""
    prefix_blocks = 12
    lens = [12 * 16 + 1, 17, 300, 193, 500, 12 * 16 + 16, 260]
    wl = synthetic.shared_prefix("bytes_sp", "int8", lens, 8, 2, prefix_blocks, seed=5)
    shared = np.asarray(wl.shared_tokens) // 16  # shared blocks per request
    extra = 0
    for j in range(prefix_blocks):
        readers = int(np.sum(shared > j))
        if readers > 1:
            extra += (readers - 1) * 16 * wl.kv_token_bytes()
    assert extra > 0
    assert (bench.decode_logical_bytes(wl) - bench.decode_algorithmic_bytes(wl)) == extra


def test_long_prefix_is_read_once_by_the_cascade_workload():
    """The cascade comparison's workload: 64 INT4 requests that all hold the
    same 512-block (8192-token) prefix. Algorithmic bytes count the prefix
    once, logical bytes 64 times, so they differ by 63 prefixes; the prefix
    is the one group prefix_groups returns."""
    wl = synthetic.cfg4_long_prefix()
    assert wl.batch == 64 and wl.kv_dtype == "int4"
    assert np.all(np.asarray(wl.shared_tokens) == 8192)
    assert np.all((wl.seq_lens >= 8208) & (wl.seq_lens <= 9216))
    token = wl.kv_token_bytes()
    assert token == 2 * 8 * (64 + 4)
    gap = bench.decode_logical_bytes(wl) - bench.decode_algorithmic_bytes(wl)
    assert gap == 63 * 8192 * token
    members, shared = bench.prefix_groups(wl)
    assert shared == 512 and sorted(members) == list(range(64))
