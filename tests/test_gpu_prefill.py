"""a3 varlen prefill attention (tcgen05) on the GPU against the fp64 oracle."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import paged_attention as pa
from pkv_testutil import GpuBatch, assert_attention_close, bits, expect_no_device_error, f32

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny-prefill", "prefill-prefix"])
def test_prefill_configs(pkv, name):
    """Slot mapping + scatter of the new tokens, then prefill over the paged cache."""
    wl = W.ALL[name]()
    b = GpuBatch(wl, W.paged_values(wl, poison_unreferenced=True))
    shared = sorted({i for _, ids in (wl.shared_groups or []) for i in ids})
    before = bits(b.k_cache[shared]) if shared else None
    b.run_slots_and_store(pkv, decode=False)
    out = b.run_prefill(pkv)
    ref = b.oracle_prefill()
    assert_attention_close(out, ref, name)
    if shared:   # blocks shared through the prefix cache are read, never written
        assert np.array_equal(bits(b.k_cache[shared]), before)
    expect_no_device_error(pkv)


def _prefill_only(pkv, q_lens, kv_lens, seed, poison=False):
    wl = W.build_workload("edge", q_lens, kv_lens, seed)
    vals = W.paged_values(wl, poison_unreferenced=poison)
    if poison:
        for s, L in enumerate(wl.kv_lens):
            nblk = -(-int(L) // wl.block_size)
            for pos in range(int(L), nblk * wl.block_size):
                blk, off = divmod(pa.slot_of(wl.block_tables[s], pos, wl.block_size), wl.block_size)
                vals.k_cache[blk, off] = float("nan")
                vals.v_cache[blk, off] = float("nan")
    b = GpuBatch(wl, vals)
    out = b.run_prefill(pkv)
    ref = pa.prefill_varlen(f32(vals.q), f32(vals.k_cache), f32(vals.v_cache), wl.cu_seqlens_q, wl.cu_seqlens_k,
                            wl.block_tables, wl.block_size, wl.softmax_scale)
    return wl, b, out, ref


PAIRS = [(1, 1), (1, 300), (5, 5), (63, 63), (64, 64), (65, 65), (127, 200), (128, 128), (129, 129),
         (200, 456), (256, 256), (300, 557), (17, 1000), (511, 511), (700, 1024)]


def test_prefill_edge_lengths_and_mid_block_offsets(pkv):
    q, k = zip(*PAIRS)
    wl, b, out, ref = _prefill_only(pkv, q, k, seed=21)
    assert_attention_close(out, ref, "edge pairs")
    expect_no_device_error(pkv)


def test_prefill_nan_in_unused_slots_does_not_leak(pkv):
    wl, b, out, ref = _prefill_only(pkv, [37, 100, 3], [37, 300, 259], seed=22, poison=True)
    assert_attention_close(out, ref, "poisoned")
    expect_no_device_error(pkv)


def test_prefill_single_sequence_many_tiles(pkv):
    wl, b, out, ref = _prefill_only(pkv, [2048], [2048], seed=23)
    assert_attention_close(out, ref, "2048 tokens")
    expect_no_device_error(pkv)


def test_prefill_deterministic_and_matches_decode_of_last_token(pkv):
    wl, b, out, ref = _prefill_only(pkv, [300, 40], [300, 812], seed=24)
    out2 = b.run_prefill(pkv)
    assert np.array_equal(bits(out), bits(out2))
    last = torch.as_tensor(wl.cu_seqlens_q[1:] - 1, dtype=torch.long, device="cuda")
    dec = pkv.pkv_decode(b.q[last].contiguous(), b.k_cache, b.v_cache, b.block_tables, b.kv_lens,
                         int(wl.kv_lens.max()), wl.softmax_scale)
    assert_attention_close(dec, ref[wl.cu_seqlens_q[1:] - 1], "decode of the last token")
    expect_no_device_error(pkv)
