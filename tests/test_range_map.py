"""The decode's split of its block stream into ranges (kvq_ranges.h), checked
on the host: static ranges per warp (one cut of the whole stream, or the same
cut in every q-head group), then tail chunks from a counter. The ranges must
partition the stream, the block -> range-id map the combine uses must invert
them, range ids must fit the workspace's records, and an explicit split count
must bound the pieces of every request. The header is compiled here with the
host C++ compiler; no GPU is involved."""
import ctypes
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "paged_quantized_kv_store_gb300", "csrc")
SRC = os.path.join(ROOT, "tests", "range_map_check.cpp")


@pytest.fixture(scope="module")
def lib():
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    d = tempfile.mkdtemp(prefix="kvq_ranges_")
    so = os.path.join(d, "range_map_check.so")
    subprocess.run([cxx, "-O1", "-std=c++17", "-shared", "-fPIC", "-I", CSRC, SRC, "-o", so],
                   check=True)
    lib = ctypes.CDLL(so)
    I32, I64 = ctypes.c_int32, ctypes.c_int64
    lib.kvq_check_range_map.argtypes = [I32, I64, I32, I32, I32, I64, I32,
                                        ctypes.POINTER(I64)]
    lib.kvq_check_range_map.restype = I32
    lib.kvq_max_pieces.argtypes = [I32, I64, I32, ctypes.c_void_p, I32, I32, I64, I32]
    lib.kvq_max_pieces.restype = I64
    yield lib
    shutil.rmtree(d, ignore_errors=True)


def check(lib, tail_ok, max_ranges, min_blocks, tb, groups, nwarps, lockstep):
    out = (ctypes.c_int64 * 6)()
    rc = lib.kvq_check_range_map(tail_ok, max_ranges, min_blocks, tb, groups, nwarps,
                                 lockstep, out)
    assert rc == 0, (rc, tail_ok, max_ranges, min_blocks, tb, groups, nwarps, lockstep)
    return dict(zip(("Pst", "C", "ntail", "k", "ranges", "ids"), list(out)))


def test_headline_shape_takes_the_tail_on_aligned_ranges(lib):
    # INT8 MHA 32/32, 128 x 4096: 256 blocks per request, 3 CTAs of 4 warps on 152 SMs
    m = check(lib, 1, 5 * 2432, 4, 128 * 256, 32, 1824, 1)
    assert m["C"] >= 8 and m["Pst"] == 512 and m["k"] == 0
    assert m["ntail"] <= 4 * 1824
    # nine tenths static, the rest in chunks
    static = 1824 * m["Pst"]
    assert 0.85 <= static / (128 * 256 * 32) <= 0.95


def test_short_shares_have_no_tail_and_cut_per_group(lib):
    # INT8 GQA-4, 256 requests x ~71 blocks, 8 kv heads: 80 blocks per warp
    m = check(lib, 1, 5 * 2432, 4, 256 * 71, 8, 1824, 1)
    assert m["C"] == 0 and m["k"] == 1824 // 8
    # the INT4 kind keeps one cut of the whole stream
    m = check(lib, 1, 5 * 2432, 4, 256 * 71, 8, 2432, 0)
    assert m["C"] == 0 and m["k"] == 0


def test_a_small_workspace_drops_the_tail(lib):
    m = check(lib, 1, 1824, 4, 128 * 256, 32, 1824, 1)  # one range per warp only
    assert m["C"] == 0 and m["ids"] <= 1824


@pytest.mark.parametrize("seed", range(6))
def test_random_shapes_partition_the_stream(lib, seed):
    rng = np.random.default_rng(seed)
    for _ in range(300):
        nwarps = int(rng.choice([8, 40, 456, 608, 1824, 2432]))
        groups = int(rng.choice([1, 2, 8, 32, 64, 128]))
        tb = int(rng.choice([0, 1, 7, 250, 4096, 33333, 300000]) // max(1, groups // 8))
        min_blocks = int(rng.choice([4, 4, 4, 13, 100]))
        check(lib, int(rng.integers(0, 2)), int(rng.choice([nwarps, 5 * nwarps])), min_blocks,
              tb, groups, nwarps, int(rng.integers(0, 2)))


@pytest.mark.parametrize("splits", [1, 2, 3, 7])
def test_explicit_split_count_bounds_the_pieces(lib, splits):
    """An explicit split count turns the tail off and keeps every request
    to at most num_splits + 1 pieces, under either static cut."""
    rng = np.random.default_rng(splits)
    for _ in range(50):
        batch = int(rng.integers(1, 40))
        nblk = rng.integers(0, 400, batch).astype(np.int32)
        min_blocks = max(1, -(-int(nblk.max()) // splits))
        for lockstep in (0, 1):
            most = lib.kvq_max_pieces(0, 5 * 608, min_blocks, nblk.ctypes.data, batch,
                                      int(rng.choice([1, 8, 32])), 608, lockstep)
            assert most <= splits + 1
