"""The seeded workloads have the structure the configurations describe."""
import numpy as np
import pytest

import workloads as W


def _owned(wl):
    return [wl.block_tables[s][wl.block_tables[s] >= 0] for s in range(wl.batch)]


@pytest.mark.parametrize("name", ["tiny-prefill", "tiny-decode", "decode-b64", "prefill-prefix",
                                  "long-decode", "full-step"])
def test_tables_are_valid(name):
    wl = W.ALL[name]()
    bs = wl.block_size
    assert wl.block_tables.dtype == np.int32
    for s, ids in enumerate(_owned(wl)):
        assert len(ids) * bs >= wl.kv_lens[s]
        assert np.all((ids >= 0) & (ids < wl.num_blocks))
        assert len(set(ids.tolist())) == len(ids)
        assert np.all(wl.block_tables[s][len(ids):] == -1)
    assert np.all(wl.q_lens >= 1) and np.all(wl.q_lens <= wl.kv_lens)


def test_private_blocks_are_not_shared_and_pool_is_permuted():
    wl = W.decode_b64()
    ids = np.concatenate(_owned(wl))
    assert len(np.unique(ids)) == len(ids)
    assert wl.num_blocks == int(np.ceil(1.25 * len(ids)))
    assert not np.all(np.diff(wl.block_tables[0][: 4]) == 1)
    assert wl.kv_lens.min() >= 512 and wl.kv_lens.max() <= 4096 and wl.batch == 64


def test_tiny_shapes():
    pre, dec = W.tiny_prefill(), W.tiny_decode()
    assert pre.kv_lens.tolist() == [37, 256, 300, 511] and pre.num_blocks == 16
    assert dec.kv_lens.tolist() == [38, 257, 301, 512] and dec.q_lens.tolist() == [1, 1, 1, 1]
    assert np.array_equal(pre.block_tables, dec.block_tables)
    assert [len(x) for x in _owned(pre)] == [1, 2, 2, 2]


def test_prefix_sharing_structure():
    wl = W.prefill_prefix()
    assert wl.batch == 32 and wl.kv_lens.min() >= 100 and wl.kv_lens.max() <= 1024
    shared_any = False
    for members, ids in wl.shared_groups:
        c = len(ids)
        assert 0 <= c <= 2
        for s in members:
            assert wl.block_tables[s][:c].tolist() == ids
            assert wl.kv_lens[s] - wl.q_lens[s] == c * wl.block_size
            assert wl.q_lens[s] >= 1
        shared_any |= c > 0
    assert shared_any
    counts = np.bincount(np.concatenate(_owned(wl)), minlength=wl.num_blocks)
    assert counts.max() == 4           # refcount of a block shared by a group of 4


def test_long_and_full_step_shapes():
    ld = W.long_decode()
    assert ld.num_blocks == 1400 and ld.batch == 8
    assert ld.kv_lens.min() >= 16384 and ld.kv_lens.max() <= 40960
    fs = W.full_step()
    assert fs.batch == 256 and fs.num_layers == 28
    assert fs.kv_lens.min() >= 128 and fs.kv_lens.max() <= 2048


def test_values_are_seeded_and_poisonable():
    wl = W.tiny_decode()
    a = W.paged_values(wl)
    b = W.paged_values(wl)
    assert a.q.dtype.is_floating_point and tuple(a.q.shape) == (4, 16, 128)
    assert bool((a.k_cache.view(-1).float() == b.k_cache.view(-1).float()).all())
    p = W.paged_values(wl, poison_unreferenced=True)
    unused = wl.unreferenced_blocks()
    assert p.k_cache[unused].float().isnan().all()
    used = wl.referenced_blocks()
    assert not p.k_cache[used].float().isnan().any()


def test_sampler_inputs():
    s = W.sampler_inputs(batch=8, vocab=1000)
    assert tuple(s.logits.shape) == (8, 1000)
    assert float(s.temperatures.min()) >= 0.5 and float(s.temperatures.max()) <= 1.0
    assert 2.5 < float(s.logits.std()) < 3.5
