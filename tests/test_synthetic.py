"""The seeded input generator and the workload recipes."""
import numpy as np
import pytest

import synthetic


def test_bits_do_not_depend_on_threads_or_offsets():
    a = synthetic.normal(3, 2, 1000, 300_000, nthreads=1)
    b = synthetic.normal(3, 2, 1000, 300_000, nthreads=7)
    c = synthetic.normal(3, 2, 0, 301_000, nthreads=3)[1000:]
    assert np.array_equal(a, b) and np.array_equal(a, c)


def test_moments_and_range():
    x = synthetic.normal(0, 1, 0, 2_000_000, dtype="f32").astype(np.float64)
    assert abs(x.mean()) < 3e-3
    assert abs(x.std() - 1) < 3e-3
    assert np.abs(x).max() <= 6


def test_f16_and_bf16_are_rne_of_f32():
    torch = pytest.importorskip("torch")
    f = synthetic.normal(4, 9, 0, 500_000, scale=8.0, dtype="f32")
    h = synthetic.normal(4, 9, 0, 500_000, scale=8.0, dtype="f16")
    b = synthetic.normal(4, 9, 0, 500_000, scale=8.0, dtype="bf16")
    assert np.array_equal(h, f.astype(np.float16).view(np.uint16))
    tb = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(b, tb)


def test_splitmix64_reference_value():
    # splitmix64(0) = 0xE220A8397B1DCDAF, the generator's published first output
    assert int(synthetic._splitmix64(np.array([0], np.uint64))[0]) == 0xE220A8397B1DCDAF


def test_permutation_is_a_permutation():
    p = synthetic.permutation(1, 2, 1000)
    assert sorted(p.tolist()) == list(range(1000))


def test_cfg_shapes():
    w1 = synthetic.cfg1()
    assert w1.seq_lens.tolist() == [17, 33, 64, 100]
    assert (w1.block_tables >= 0).sum() == 16 and w1.num_blocks == 64
    w2 = synthetic.cfg2()
    assert w2.batch == 32 and w2.seq_lens.min() >= 512 and w2.seq_lens.max() <= 4096
    assert w2.num_blocks == int(((w2.seq_lens + 15) // 16).sum())
    used = w2.block_tables[w2.block_tables >= 0]
    assert len(np.unique(used)) == used.size == w2.num_blocks
    w3 = synthetic.cfg3(batch=4)
    assert (w3.k_chan_scale == 8).sum() == 41 and (w3.v_chan_scale == 8).sum() == 41
    w4 = synthetic.cfg4()
    assert w4.seq_lens.min() >= 128 and w4.seq_lens.max() <= 8192
    k = w4.shared_tokens // 16
    for b in range(w4.batch):
        assert np.array_equal(w4.block_tables[b, :k[b]], w4.prefix_blocks[:k[b]])
        # the block holding the newest token is private
        last = (int(w4.seq_lens[b]) - 1) // 16
        assert w4.block_tables[b, last] not in set(w4.prefix_blocks.tolist())
    w5 = synthetic.cfg5()
    assert w5.batch == 256 and len(w5.chunk_slots) == 4096
    used = set(w5.block_tables[w5.block_tables >= 0].tolist())
    assert not used & set((w5.chunk_slots // 16).tolist())


def test_setup_plus_step_cover_every_position_once():
    wl = synthetic.cfg4(batch=6)
    seen = {}
    for slots, k, v in wl.setup_chunks(max_tokens=500):
        for s in slots.tolist():
            seen[s] = seen.get(s, 0) + 1
    slots, _, _ = wl.step_store()
    for s in slots.tolist():
        seen[s] = seen.get(s, 0) + 1
    assert max(seen.values()) == 1
    want = set()
    for b in range(wl.batch):
        for p in range(int(wl.seq_lens[b])):
            want.add(wl.slot(b, p))
    assert want <= set(seen)
