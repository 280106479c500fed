"""a4 decode attention on the GPU against the fp64 oracle."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import paged_attention as pa
from pkv_testutil import GpuBatch, assert_attention_close, bits, expect_no_device_error, f32

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny-decode", "decode-b64", "long-decode", "full-step"])
def test_decode_configs_all_rows(pkv, name):
    """Write the new token's K/V through the slot mapping, then decode; every row vs the oracle."""
    wl = W.ALL[name]()
    b = GpuBatch(wl, W.paged_values(wl))
    b.run_slots_and_store(pkv, decode=True)
    out = b.run_decode(pkv)
    ref = b.oracle_decode()
    assert_attention_close(out, ref, name)
    expect_no_device_error(pkv)


def _decode_only(pkv, kv_lens, seed, poison=False, pool_factor=1.25):
    """Decode over a seeded pool without a store step (lengths may be 0)."""
    kv_lens = np.asarray(kv_lens, dtype=np.int32)
    wl = W.build_workload("edge", np.ones_like(kv_lens), kv_lens, seed, pool_factor=pool_factor)
    vals = W.paged_values(wl, poison_unreferenced=poison)
    if poison:   # every slot a sequence has not reached holds NaN as well
        for s, L in enumerate(kv_lens):
            nblk = -(-int(L) // wl.block_size)
            for pos in range(int(L), nblk * wl.block_size):
                blk, off = divmod(pa.slot_of(wl.block_tables[s], pos, wl.block_size), wl.block_size)
                vals.k_cache[blk, off] = float("nan")
                vals.v_cache[blk, off] = float("nan")
    b = GpuBatch(wl, vals)
    out = b.run_decode(pkv)
    ref = pa.decode(f32(vals.q), f32(vals.k_cache), f32(vals.v_cache), wl.block_tables, kv_lens,
                    wl.block_size, wl.softmax_scale)
    return b, out, ref


def test_decode_edge_lengths(pkv):
    lens = [1, 2, 31, 32, 33, 255, 256, 257, 511, 512, 513, 1000, 4096, 0, 7, 0]
    b, out, ref = _decode_only(pkv, lens, seed=11)
    assert_attention_close(out, ref, "edge lengths")
    assert torch.count_nonzero(out[13]).item() == 0 and torch.count_nonzero(out[15]).item() == 0
    expect_no_device_error(pkv)


def test_decode_nan_in_unused_slots_does_not_leak(pkv):
    lens = [5, 300, 257, 1023, 64]
    b, out, ref = _decode_only(pkv, lens, seed=12, poison=True)
    assert_attention_close(out, ref, "poisoned pool")
    expect_no_device_error(pkv)


def test_decode_single_long_sequence_split_over_all_warps(pkv):
    b, out, ref = _decode_only(pkv, [40960], seed=13)
    assert_attention_close(out, ref, "one long sequence")
    expect_no_device_error(pkv)


def test_decode_many_short_sequences(pkv):
    rng = np.random.default_rng(14)
    lens = rng.integers(1, 70, size=600)
    b, out, ref = _decode_only(pkv, lens, seed=14)
    assert_attention_close(out, ref, "600 short sequences")
    expect_no_device_error(pkv)


def test_decode_deterministic_and_block_relabel_invariant(pkv):
    wl = W.decode_b64(batch=16)
    vals = W.paged_values(wl)
    b = GpuBatch(wl, vals)
    o1 = b.run_decode(pkv).clone()
    o2 = b.run_decode(pkv).clone()
    assert np.array_equal(bits(o1), bits(o2))
    # move physical block i to pi[i]: the same logical data, other addresses
    pi = np.random.default_rng(15).permutation(wl.num_blocks)
    inv = torch.from_numpy(np.argsort(pi)).cuda()
    k2 = b.k_cache[inv].contiguous()
    v2 = b.v_cache[inv].contiguous()
    bt2 = torch.from_numpy(np.where(wl.block_tables >= 0, pi[np.maximum(wl.block_tables, 0)], -1).astype(np.int32)).cuda()
    o3 = pkv.pkv_decode(b.q, k2, v2, bt2, b.kv_lens, int(wl.kv_lens.max()), wl.softmax_scale)
    assert np.array_equal(bits(o1), bits(o3))
    expect_no_device_error(pkv)


@pytest.mark.parametrize("name", ["decode-b8", "tiny-decode"])
def test_decode_reuses_caller_workspace_and_out(pkv, name):
    """Stale workspace contents must not matter, also when the grid has more warps than KV chunks."""
    wl = W.decode_b64(batch=8) if name == "decode-b8" else W.tiny_decode()
    b = GpuBatch(wl, W.paged_values(wl))
    ws = pkv.decode_workspace(wl.batch, wl.num_heads, wl.num_kv_heads, wl.head_dim)
    ws.fill_(0xAB)                       # contents need no initialisation
    out = torch.full_like(b.q, float("nan"))
    b.run_decode(pkv, out=out, workspace=ws)
    assert_attention_close(out, b.oracle_decode(pools=(f32(b.cpu.k_cache), f32(b.cpu.v_cache))), "workspace reuse")
    small = ws[: ws.numel() // 2]
    with pytest.raises(pkv.PkvError) as e:
        b.run_decode(pkv, workspace=small)
    assert e.value.status == 3


def test_decode_flags_block_id_outside_pool(pkv):
    wl = W.decode_b64(batch=4)
    b = GpuBatch(wl, W.paged_values(wl))
    bt = b.block_tables.clone()
    bt[1, 0] = wl.num_blocks + 5
    pkv.pkv_decode(b.q, b.k_cache, b.v_cache, bt, b.kv_lens, int(wl.kv_lens.max()), wl.softmax_scale)
    code, info = pkv.pkv_get_device_error(clear=True)
    assert code == 1 and info == 1


@pytest.mark.parametrize("name", ["tiny-decode", "decode-b64", "long-decode", "full-step"])
def test_decode_append_matches_oracle(pkv, name):
    """KV write fused into decode: pool bit-exact, slots bit-exact, output vs the fp64 oracle."""
    wl = W.ALL[name]()
    b = GpuBatch(wl, W.paged_values(wl, poison_unreferenced=True))
    slots = torch.full((wl.batch,), -7, dtype=torch.int32, device="cuda")
    out = pkv.pkv_decode_append(b.q, b.k_new, b.v_new, b.k_cache, b.v_cache, b.block_tables, b.kv_lens,
                                int(wl.kv_lens.max()), wl.softmax_scale, slot_mapping=slots)
    kc, vc = b.oracle_pools()
    assert np.array_equal(slots.cpu().numpy().astype(np.int64), b.oracle_slots())
    assert np.array_equal(bits(b.k_cache), bits(torch.from_numpy(kc).to(torch.bfloat16)))
    assert np.array_equal(bits(b.v_cache), bits(torch.from_numpy(vc).to(torch.bfloat16)))
    assert_attention_close(out, b.oracle_decode(pools=(kc, vc)), name)
    expect_no_device_error(pkv)


def test_decode_append_bit_identical_to_unfused_path(pkv):
    wl = W.decode_b64(batch=32)
    vals = W.paged_values(wl)
    fused = GpuBatch(wl, vals)
    plain = GpuBatch(wl, vals)
    o1 = pkv.pkv_decode_append(fused.q, fused.k_new, fused.v_new, fused.k_cache, fused.v_cache, fused.block_tables,
                               fused.kv_lens, int(wl.kv_lens.max()), wl.softmax_scale)
    plain.run_slots_and_store(pkv, decode=True)
    o2 = plain.run_decode(pkv)
    assert np.array_equal(bits(o1), bits(o2))
    assert np.array_equal(bits(fused.k_cache), bits(plain.k_cache))
    expect_no_device_error(pkv)


def test_decode_append_zero_context_writes_nothing(pkv):
    kv_lens = np.array([5, 0, 300, 0], dtype=np.int32)
    wl = W.build_workload("zeros", np.ones(4, np.int32), kv_lens, seed=16)
    vals = W.paged_values(wl)
    b = GpuBatch(wl, vals)
    before = bits(b.k_cache).copy()
    slots = torch.full((4,), 99, dtype=torch.int32, device="cuda")
    out = pkv.pkv_decode_append(b.q, b.k_new, b.v_new, b.k_cache, b.v_cache, b.block_tables, b.kv_lens, 300,
                                wl.softmax_scale, slot_mapping=slots)
    s = slots.cpu().tolist()
    assert s[1] == -1 and s[3] == -1 and s[0] >= 0 and s[2] >= 0
    after = bits(b.k_cache)
    changed = np.argwhere((before != after).reshape(wl.num_blocks, wl.block_size, -1).any(axis=2))
    assert len(changed) == 2                                   # one row for each non-empty sequence
    assert torch.count_nonzero(out[1]).item() == 0 and torch.count_nonzero(out[3]).item() == 0
    expect_no_device_error(pkv)


def test_prepared_decode_append_call(pkv):
    """DecodeAppendCall: checked and marshalled once, then each call sees the buffers' current contents."""
    wl = W.decode_b64(batch=16)
    vals = W.paged_values(wl)
    b = GpuBatch(wl, vals)
    out = torch.empty_like(b.q)
    call = pkv.DecodeAppendCall(b.q, b.k_new, b.v_new, b.k_cache, b.v_cache, b.block_tables, b.kv_lens,
                                int(wl.kv_lens.max()), wl.softmax_scale, out=out)
    ref = GpuBatch(wl, vals)
    o_ref = pkv.pkv_decode_append(ref.q, ref.k_new, ref.v_new, ref.k_cache, ref.v_cache, ref.block_tables,
                                  ref.kv_lens, int(wl.kv_lens.max()), wl.softmax_scale)
    assert np.array_equal(bits(out), bits(o_ref))
    # new inputs copied into the same buffers are picked up by the next call
    g = torch.Generator().manual_seed(5)
    q2 = torch.randn(tuple(b.q.shape), generator=g).to(torch.bfloat16).cuda()
    b.q.copy_(q2)
    ref.q.copy_(q2)
    assert call() is out
    o_ref2 = pkv.pkv_decode_append(ref.q, ref.k_new, ref.v_new, ref.k_cache, ref.v_cache, ref.block_tables,
                                   ref.kv_lens, int(wl.kv_lens.max()), wl.softmax_scale)
    torch.cuda.synchronize()
    assert np.array_equal(bits(out), bits(o_ref2))
    assert not np.array_equal(bits(o_ref2), bits(o_ref))
    expect_no_device_error(pkv)


def test_decode_at_the_batch_limit(pkv):
    """4096 sequences, the largest batch (the chunk-prefix scan then sums 32 sequences per
    thread), over a small pool that the sequences share read-only through random block tables;
    zero-length rows come out zero; sampled rows against the oracle.  4097 is refused."""
    B, nb, bs, hq, hkv, d = 4096, 64, 256, 16, 8, 128
    g = torch.Generator().manual_seed(61)
    kc = torch.randn(nb, bs, hkv, d, generator=g).to(torch.bfloat16)
    vc = torch.randn(nb, bs, hkv, d, generator=g).to(torch.bfloat16)
    q = torch.randn(B, hq, d, generator=g).to(torch.bfloat16)
    lens = torch.randint(0, 2 * bs + 1, (B,), generator=g).to(torch.int32)
    lens[::97] = 0
    bt = torch.randint(0, nb, (B, 2), generator=g).to(torch.int32)
    scale = d ** -0.5
    out = pkv.pkv_decode(q.cuda(), kc.cuda(), vc.cuda(), bt.cuda(), lens.cuda(), 2 * bs, scale)
    rows = list(range(0, B, 41)) + [B - 1]
    ref = pa.decode_rows(f32(q), f32(kc), f32(vc), bt.numpy(), lens.numpy(), bs, scale, rows)
    assert_attention_close(out[rows], ref, "batch 4096")
    zero = torch.nonzero(lens == 0).flatten().tolist()
    assert torch.count_nonzero(out[zero]).item() == 0
    expect_no_device_error(pkv)
    q2 = torch.zeros(B + 1, hq, d, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_decode(q2, kc.cuda(), vc.cuda(), torch.zeros(B + 1, 2, dtype=torch.int32, device="cuda"),
                       torch.ones(B + 1, dtype=torch.int32, device="cuda"), 2 * bs, scale)
    assert e.value.status == 2                        # PKV_ERR_UNSUPPORTED
