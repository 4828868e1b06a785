"""The C ABI library: it loads, exports what kvq.h declares, validates on the host.

No compute call is made here (these tests run without a GPU): only argument
checks that return before any launch, and the host-only launch planner.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import paged_quantized_kv_store_gb300 as kvq
from paged_quantized_kv_store_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvq.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return kvq.load()


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^[a-z_][\w ]*?\**\s*\b(\w+)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while")))


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert set(kvq.EXPORTED) <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    out = os.popen(f"nm -D --defined-only {_build.LIB_PATH}").read()
    for n in names:
        assert re.search(rf"\bT {n}$", out, flags=re.M), n


def test_version_and_status_strings(lib):
    assert kvq.kvq_version() >= 100
    for s in range(6):
        assert kvq.kvq_status_string(s)


def _pool(**kw):
    d = dict(k=16, v=32, k_sz=48, v_sz=64, num_blocks=4, block_size=16, kv_heads=2,
             head_dim=128, kv_dtype=kvq.KVQ_INT8)
    d.update(kw)
    return kvq._Pool(d["k"], d["v"], d["k_sz"], d["v_sz"], d["num_blocks"], d["block_size"],
                     d["kv_heads"], d["head_dim"], d["kv_dtype"])


def test_store_validation(lib):
    f = lib.kv_store_quant
    ok_ptr = 256
    assert f(None, ok_ptr, ok_ptr, 0, ok_ptr, 1, None, None) == 1
    assert f(ctypes.byref(_pool(head_dim=64)), ok_ptr, ok_ptr, 0, ok_ptr, 1, None, None) == 2
    assert f(ctypes.byref(_pool(block_size=32)), ok_ptr, ok_ptr, 0, ok_ptr, 1, None, None) == 2
    assert f(ctypes.byref(_pool(k_sz=None)), ok_ptr, ok_ptr, 0, ok_ptr, 1, None, None) == 1
    assert f(ctypes.byref(_pool(k=17)), ok_ptr, ok_ptr, 0, ok_ptr, 1, None, None) == 1  # misaligned
    assert f(ctypes.byref(_pool()), ok_ptr, ok_ptr, 4, ok_ptr, 1, None, None) == 2  # int4 input
    assert f(ctypes.byref(_pool(kv_dtype=kvq.KVQ_F16)), ok_ptr, ok_ptr, kvq.KVQ_BF16, ok_ptr, 1,
             None, None) == 2  # copy pools need matching dtypes
    assert f(ctypes.byref(_pool()), None, ok_ptr, 0, ok_ptr, 1, None, None) == 1
    assert f(ctypes.byref(_pool()), ok_ptr, ok_ptr, 0, ok_ptr, -1, None, None) == 1
    assert f(ctypes.byref(_pool()), None, None, 0, None, 0, None, None) == 0  # nothing to do


def test_decode_validation(lib):
    f = lib.paged_decode_attn
    p = 256
    args = dict(q=p, q_dtype=0, out=p, bt=p, mb=4, sl=p, batch=2, hq=4, msl=64, scale=0.1,
                splits=0, ws=None, wsb=0, err=None, s=None)

    def call(pool, **kw):
        a = dict(args)
        a.update(kw)
        return f(ctypes.byref(pool) if pool is not None else None, a["q"], a["q_dtype"],
                 a["out"], a["bt"], a["mb"], a["sl"], a["batch"], a["hq"], a["msl"],
                 a["scale"], a["splits"], a["ws"], a["wsb"], a["err"], a["s"])

    assert call(None) == 1
    assert call(_pool(), q_dtype=4) == 2
    assert call(_pool(kv_dtype=kvq.KVQ_BF16), q_dtype=0) == 2
    assert call(_pool(), hq=3) == 1          # q heads not a multiple of kv heads
    assert call(_pool(), mb=0) == 1
    assert call(_pool(), scale=float("nan")) == 1
    assert call(_pool(head_dim=256)) == 2


def test_tables_validation(lib):
    f = lib.kvq_block_tables_from_req_to_token
    assert f(256, 4, 64, 256, 256, -1, 4, 256, None, None) == 1
    assert f(256, 4, 64, 256, 256, 2, 0, 256, None, None) == 1
    assert f(None, 4, 64, 256, 256, 2, 4, 256, None, None) == 1
    assert f(None, 4, 64, None, None, 0, 4, None, None, None) == 0


def test_planner(lib):
    plan = kvq.paged_decode_attn_plan
    p = plan(128, 32, 32, 4096, num_sms=152)
    assert p["warps"] == 152 * 4 * 4 and p["max_ctas_per_sm"] == 4
    assert p["min_blocks_per_warp"] == 4
    assert p["head_groups"] == 1 and p["heads_per_group"] == 1
    # two partial records (132 floats) per warp and head, plus the length header
    assert p["workspace_bytes"] >= p["warps"] * 2 * 132 * 4 + 4 * 131
    p4 = plan(64, 32, 8, 8192, num_sms=152)
    assert p4["heads_per_group"] == 4
    assert p4["workspace_bytes"] >= p4["warps"] * 2 * 4 * 132 * 4
    # layout: 256 bytes of counters, the header ((batch + 6) int32, rounded
    # up to 256 bytes), then 2 records of 132 floats per q head of the group
    # slot for 5 ranges per warp
    for b, hq, hkv in ((128, 32, 32), (64, 32, 8), (1, 64, 2)):
        q = plan(b, hq, hkv, 4096, num_sms=152)
        header = -(-(b + 6) * 4 // 256) * 256
        assert q["workspace_bytes"] == (256 + header +
                                        5 * q["warps"] * 2 * q["heads_per_group"] * 132 * 4)
    # the workspace does not grow with the context
    assert plan(64, 32, 8, 100, num_sms=152)["workspace_bytes"] == p4["workspace_bytes"]
    # explicit split counts bound the pieces of a request
    for s in (1, 2, 3, 7):
        p = plan(6, 16, 8, 4000, num_splits=s, num_sms=152)
        assert p["min_blocks_per_warp"] == -(-250 // s)
    # q heads of a kv head are taken 8 at a time
    p = plan(2, 64, 2, 64, num_sms=10)
    assert p["head_groups"] == 4 and p["heads_per_group"] == 8
    p = plan(2, 12, 4, 64, num_sms=10)
    assert p["head_groups"] == 1 and p["heads_per_group"] == 3
    with pytest.raises(kvq.KvqError):
        plan(2, 6, 4, 64, num_sms=10)
    with pytest.raises(kvq.KvqError):
        plan(2, 8, 4, 64, num_sms=10, head_dim=64)


def test_product_path_has_no_oracle_dependency():
    """The product package neither imports nor links the oracle or the generator."""
    pkg = os.path.join(ROOT, "paged_quantized_kv_store_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, fn)).read()
                for banned in ("import oracle", "from oracle", "kvq_oracle", "synthetic",
                               "kvqgen"):
                    assert banned not in text, (fn, banned)


def test_shared_prefix_validation(lib):
    """Argument checks of paged_decode_attn_shared_prefix that run before any
    device access."""
    f = lib.paged_decode_attn_shared_prefix
    p = 256
    args = dict(q=p, q_dtype=0, out=p, bt=p, mb=4, sl=p, batch=2, hq=4, msl=64, scale=0.1,
                off=p, mem=p, sh=p, ng=1, nm=2, maxs=2, splits=0, ws=None, wsb=0, err=None,
                s=None)

    def call(**kw):
        a = dict(args)
        a.update(kw)
        return f(ctypes.byref(_pool()), a["q"], a["q_dtype"], a["out"], a["bt"], a["mb"],
                 a["sl"], a["batch"], a["hq"], a["msl"], a["scale"], a["off"], a["mem"],
                 a["sh"], a["ng"], a["nm"], a["maxs"], a["splits"], a["ws"], a["wsb"],
                 a["err"], a["s"])

    assert call(ng=-1) == 1
    assert call(nm=-1) == 1
    assert call(maxs=-1) == 1
    assert call(maxs=5) == 1          # more shared blocks than table columns
    assert call(off=None) == 1
    assert call(sh=None) == 1
    assert call(mem=None) == 1
    assert call(ng=9000) == 2


def test_shared_prefix_group_detection():
    """Host-side grouping by common leading blocks."""
    bt = np.array([[7, 8, 9, 1], [7, 8, 9, 2], [7, 8, 3, -1], [5, 6, -1, -1], [7, 8, 9, 4]],
                  dtype=np.int32)
    lens = np.array([60, 64, 40, 30, 50], dtype=np.int32)
    g = kvq.SharedPrefixGroups.detect(bt, lens, device="cpu")
    # requests 0, 1, 4 share 3 blocks (3 x 3 = 9 > 4 x 2 = 8); 2 stays out
    assert g.num_groups == 1
    assert g.members.tolist() == [0, 1, 4]
    assert g.shared_blocks.tolist() == [3] and g.offsets.tolist() == [0, 3]
    assert g.max_shared_blocks == 3
    # only full blocks are shared: a 47-token request has 2 full blocks
    lens2 = np.array([47, 64, 40, 30, 47], dtype=np.int32)
    g2 = kvq.SharedPrefixGroups.detect(bt, lens2, device="cpu")
    assert g2.members.tolist() == [0, 1, 2, 4] and g2.shared_blocks.tolist() == [2]
    e = kvq.SharedPrefixGroups.from_lists([], device="cpu")
    assert e.num_groups == 0 and e.num_members == 0 and e.max_shared_blocks == 0


def test_copy_blocks_validation(lib):
    f = lib.kvq_copy_blocks
    p = 256
    a, b = _pool(), _pool(num_blocks=9)
    assert f(ctypes.byref(a), ctypes.byref(b), p, p, 0, None, None) == 0   # nothing to do
    assert f(ctypes.byref(a), ctypes.byref(b), p, p, -1, None, None) == 1
    assert f(ctypes.byref(a), ctypes.byref(b), None, p, 3, None, None) == 1
    assert f(ctypes.byref(a), ctypes.byref(_pool(kv_dtype=kvq.KVQ_INT4)), p, p, 3, None,
             None) == 1  # different kinds
    assert f(ctypes.byref(a), ctypes.byref(_pool(kv_heads=4)), p, p, 3, None, None) == 1
    assert f(None, ctypes.byref(b), p, p, 3, None, None) == 1


def test_extend_validation(lib):
    f = lib.paged_extend_attn
    p = 256
    args = dict(q=p, q_dtype=0, out=p, qo=p, kl=p, bt=p, mb=4, batch=2, tq=8, hq=4, mkl=64,
                scale=0.1, var=0, ws=p, wsb=1 << 20, err=None, s=None)

    def call(pool=None, **kw):
        a = dict(args)
        a.update(kw)
        return f(ctypes.byref(pool or _pool()), a["q"], a["q_dtype"], a["out"], a["qo"],
                 a["kl"], a["bt"], a["mb"], a["batch"], a["tq"], a["hq"], a["mkl"], a["scale"],
                 a["var"], a["ws"], a["wsb"], a["err"], a["s"])

    assert call(batch=-1) == 1
    assert call(tq=-1) == 1
    assert call(hq=3) == 1                 # not a multiple of kv heads
    assert call(q_dtype=kvq.KVQ_INT8) == 2
    assert call(pool=_pool(kv_dtype=kvq.KVQ_F16), q_dtype=kvq.KVQ_BF16) == 2
    assert call(scale=float("nan")) == 1
    assert call(batch=0) == 0 and call(tq=0) == 0
    assert call(qo=None) == 1
    assert call(q=p + 8) == 1              # misaligned
    assert call(var=3) == 1 and call(var=-1) == 1
    assert call(var=2, pool=_pool(kv_dtype=kvq.KVQ_BF16), q_dtype=kvq.KVQ_BF16) == 2
    # the tcgen05 kernel: at most 4096 requests (its unit table lives in shared
    # memory), and a pool with at least one block (a missing block is read
    # from block 0 and masked); both refused before anything launches
    assert call(var=2, batch=4097) == 2
    assert call(var=2, pool=_pool(num_blocks=0)) == 2


def test_decode_step_validation(lib):
    f = lib.kvq_decode_step
    p = 256
    args = dict(r2t=p, nslots=4, mctx=64, rpi=p, sl=p, batch=2, bt=p, mb=4, k=p, v=p, sm=p,
                ntok=2, q=p, q_dtype=0, out=p, hq=4, msl=64, scale=0.1, splits=0, ws=None,
                wsb=0, err=None, s=None)

    def call(pool=None, **kw):
        a = dict(args)
        a.update(kw)
        return f(ctypes.byref(pool or _pool()), a["r2t"], a["nslots"], a["mctx"], a["rpi"],
                 a["sl"], a["batch"], a["bt"], a["mb"], a["k"], a["v"], a["sm"], a["ntok"],
                 a["q"], a["q_dtype"], a["out"], a["hq"], a["msl"], a["scale"], a["splits"],
                 a["ws"], a["wsb"], a["err"], a["s"])

    assert f(None, *args.values()) == 1        # args are in the C order
    assert call(q_dtype=kvq.KVQ_INT8) == 2
    assert call(k=None) == 1 and call(sm=None) == 1
    assert call(v=p + 4) == 1                     # misaligned new rows
    assert call(batch=-1) == 1 and call(ntok=-1) == 1 and call(nslots=-1) == 1
    assert call(rpi=None) == 1
    assert call(batch=0, ntok=0) == 0             # nothing to do
    # no requests: the step is the store, which refuses a 16-bit pool of another dtype
    assert call(pool=_pool(kv_dtype=kvq.KVQ_F16), q_dtype=kvq.KVQ_BF16, batch=0) == 2
    n = ctypes.c_size_t(7)
    g = lib.kvq_decode_step_workspace_size
    assert g(2, 4, 2, 128, 64, 0, None) == 1
    assert g(-1, 4, 2, 128, 64, 0, ctypes.byref(n)) == 1 and n.value == 0
    assert g(2, 3, 2, 128, 64, 0, ctypes.byref(n)) == 1
    assert g(2, 4, 2, 256, 64, 0, ctypes.byref(n)) == 2


def test_decode_step_form(lib):
    """One launch for a decode batch's tokens, four kernels with a prefill chunk."""
    assert lib.kvq_decode_step_fused(4, 4) == 1
    assert lib.kvq_decode_step_fused(4, 8) == 1
    assert lib.kvq_decode_step_fused(4, 9) == 0
    assert lib.kvq_decode_step_fused(256, 4352) == 0
    assert lib.kvq_decode_step_fused(0, 0) == 0
    assert kvq.kvq_decode_step_fused(128, 128) is True
