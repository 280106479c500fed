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


def test_prefill_many_units_per_cta(pkv):
    """~2400 work units over the persistent grid: exercises the cross-unit pipeline."""
    rng = np.random.default_rng(25)
    kl = rng.integers(1, 400, size=200)
    ql = np.maximum(1, (kl * rng.uniform(0.2, 1.0, size=200)).astype(int))
    ql = np.minimum(ql, kl)
    wl, b, out, ref = _prefill_only(pkv, ql, kl, seed=25)
    assert_attention_close(out, ref, "200 sequences, mid-block offsets")
    expect_no_device_error(pkv)


def test_prefill_long_sequence_with_prefix(pkv):
    """Long rescale chains: 3000 new tokens after a 5192-token cached prefix."""
    wl, b, out, ref = _prefill_only(pkv, [3000, 129], [8192, 129], seed=26)
    assert_attention_close(out, ref, "3000 new tokens after a 5192-token prefix")
    expect_no_device_error(pkv)


def test_prefill_zero_length_queries(pkv):
    wl, b, out, ref = _prefill_only(pkv, [0, 5, 0, 70], [10, 5, 300, 300], seed=27)
    assert_attention_close(out, ref, "sequences with no new tokens")
    expect_no_device_error(pkv)


def test_prefill_large_score_range_forces_rescale(pkv):
    """Scores growing along the keys make the row max climb by more than 2^8 several times."""
    wl = W.build_workload("ramp", [200], [1000], seed=28)
    vals = W.paged_values(wl)
    ramp = torch.linspace(0.0, 6.0, wl.block_size * vals.k_cache.shape[0]).view(vals.k_cache.shape[0], wl.block_size, 1, 1)
    vals.k_cache = (vals.k_cache.float() * ramp).to(torch.bfloat16)
    vals.q = (vals.q.float() * 3.0).to(torch.bfloat16)
    # a peaked softmax returns nearly single V rows; keep |o| moderate so bf16 output
    # rounding stays inside the stated absolute tolerance
    vals.v_cache = (vals.v_cache.float() * 0.25).to(torch.bfloat16)
    b = GpuBatch(wl, vals)
    out = b.run_prefill(pkv)
    ref = pa.prefill_varlen(f32(vals.q), f32(vals.k_cache), f32(vals.v_cache), wl.cu_seqlens_q, wl.cu_seqlens_k,
                            wl.block_tables, wl.block_size, wl.softmax_scale)
    assert_attention_close(out, ref, "large score range")
    expect_no_device_error(pkv)


# ---- planned once per batch, run per layer -----------------------------------------------------

def _plan(pkv, b, wl, hq, hkv, max_seqlen_k=None):
    return pkv.pkv_prefill_plan(b.cu_q, b.cu_k, wl.total_q, int(wl.q_lens.max()),
                                int(wl.kv_lens.max()) if max_seqlen_k is None else max_seqlen_k,
                                hq, hkv, 128, wl.block_size, b.block_tables.shape[1])


def test_prefill_plan_serves_every_layer(pkv):
    """One plan, then three planned calls (three layers: their own q and pools, written in between
    by the scatter) in order on one stream: each equals pkv_prefill_varlen on the same inputs bit for
    bit and the oracle within tolerance; every call leaves the work queue reset for the next."""
    wl = W.prefill_prefix()
    layers = [GpuBatch(wl, W.paged_values(wl, layer=i)) for i in range(3)]
    hq, hkv = layers[0].q.shape[1], layers[0].k_cache.shape[2]
    ws = _plan(pkv, layers[0], wl, hq, hkv)
    outs = []
    for b in layers:
        b.run_slots_and_store(pkv, decode=False)
        outs.append(pkv.pkv_prefill_varlen_planned(b.q, b.k_cache, b.v_cache, b.cu_q, b.cu_k, b.block_tables,
                                                   int(wl.q_lens.max()), int(wl.kv_lens.max()),
                                                   wl.softmax_scale, ws))
    for i, b in enumerate(layers):
        ref = b.run_prefill(pkv)
        assert torch.equal(outs[i].view(torch.int16), ref.view(torch.int16)), f"layer {i}"
    assert_attention_close(outs[2], layers[2].oracle_prefill(), "third planned layer")
    expect_no_device_error(pkv)


def test_prefill_planned_call_on_a_plan_for_other_arguments(pkv):
    """A plan made for another max_seqlen_k (so other cost buckets) is not used: the planned call
    computes nothing, leaves out as it was and records the plan error."""
    wl = W.prefill_prefix()
    b = GpuBatch(wl, W.paged_values(wl))
    b.run_slots_and_store(pkv, decode=False)
    hq, hkv = b.q.shape[1], b.k_cache.shape[2]
    ws = _plan(pkv, b, wl, hq, hkv, max_seqlen_k=int(wl.kv_lens.max()) + 1024)
    out = torch.full_like(b.q, 7.0)
    pkv.pkv_prefill_varlen_planned(b.q, b.k_cache, b.v_cache, b.cu_q, b.cu_k, b.block_tables,
                                   int(wl.q_lens.max()), int(wl.kv_lens.max()), wl.softmax_scale, ws, out=out)
    code, _ = pkv.pkv_get_device_error(clear=True)
    assert code == 7
    assert bool((out == 7.0).all())
    # the same workspace, planned again for the right arguments, works
    pkv.pkv_prefill_plan(b.cu_q, b.cu_k, wl.total_q, int(wl.q_lens.max()), int(wl.kv_lens.max()), hq, hkv, 128,
                         wl.block_size, b.block_tables.shape[1], workspace=ws)
    pkv.pkv_prefill_varlen_planned(b.q, b.k_cache, b.v_cache, b.cu_q, b.cu_k, b.block_tables,
                                   int(wl.q_lens.max()), int(wl.kv_lens.max()), wl.softmax_scale, ws, out=out)
    assert_attention_close(out, b.oracle_prefill(), "after planning again")
    expect_no_device_error(pkv)


def test_prefill_plan_and_planned_calls_in_a_cuda_graph(pkv):
    """plan + two planned layers captured once; replays with new q in the captured buffer match
    eager pkv_prefill_varlen bit for bit."""
    wl = W.prefill_prefix()
    b = GpuBatch(wl, W.paged_values(wl))
    b.run_slots_and_store(pkv, decode=False)
    hq, hkv = b.q.shape[1], b.k_cache.shape[2]
    ws = torch.empty(pkv.pkv_prefill_workspace_size(len(wl.q_lens), hq, hkv, 128, int(wl.q_lens.max())),
                     dtype=torch.uint8, device="cuda")
    o1, o2 = torch.empty_like(b.q), torch.empty_like(b.q)
    q2 = b.q.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    args = (int(wl.q_lens.max()), int(wl.kv_lens.max()), wl.softmax_scale, ws)
    with torch.cuda.stream(s):
        def step():
            pkv.pkv_prefill_plan(b.cu_q, b.cu_k, wl.total_q, int(wl.q_lens.max()), int(wl.kv_lens.max()), hq, hkv,
                                 128, wl.block_size, b.block_tables.shape[1], workspace=ws)
            pkv.pkv_prefill_varlen_planned(b.q, b.k_cache, b.v_cache, b.cu_q, b.cu_k, b.block_tables, *args, out=o1)
            pkv.pkv_prefill_varlen_planned(q2, b.k_cache, b.v_cache, b.cu_q, b.cu_k, b.block_tables, *args, out=o2)
        step()                      # warm-up outside the capture
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    gen = torch.Generator().manual_seed(5)
    for _ in range(2):
        b.q.copy_(torch.randn(b.q.shape, generator=gen).to(torch.bfloat16))
        q2.copy_(torch.randn(q2.shape, generator=gen).to(torch.bfloat16))
        g.replay()
        torch.cuda.synchronize()
        r1 = b.run_prefill(pkv)
        r2 = pkv.pkv_prefill_varlen(q2, b.k_cache, b.v_cache, b.cu_q, b.cu_k, b.block_tables,
                                    int(wl.q_lens.max()), int(wl.kv_lens.max()), wl.softmax_scale)
        assert torch.equal(o1.view(torch.int16), r1.view(torch.int16))
        assert torch.equal(o2.view(torch.int16), r2.view(torch.int16))
    expect_no_device_error(pkv)


def test_prefill_plan_lists_every_unit_costliest_first(pkv):
    """The plan's records, read back from the workspace: exactly one record per (sequence, pair of
    128/G-token tiles) with its query start and lengths, the header's count equal to their number,
    and the list ordered by non-increasing cost (twice the longer tile's KV tiles, plus one when
    the second tile has tokens).  Ties may come in any order."""
    wl = W.prefill_prefix()
    b = GpuBatch(wl, W.paged_values(wl))
    hq, hkv = b.q.shape[1], b.k_cache.shape[2]
    ws = _plan(pkv, b, wl, hq, hkv)
    torch.cuda.synchronize()
    words = ws.view(torch.int32).cpu().numpy()
    qtok = 128 // (hq // hkv)
    expect = []
    for s, (ql, kl) in enumerate(zip(wl.q_lens.astype(int), wl.kv_lens.astype(int))):
        for pr in range(-(-ql // (2 * qtok))):
            expect.append((s, pr, int(wl.cu_seqlens_q[s]), ql, kl))
    n = int(words[0])
    assert n == len(expect)
    recs = words[4:4 + 4 * n].reshape(n, 4)
    got = sorted((int(r[0]) >> 16, int(r[0]) & 0xFFFF, int(r[1]), int(r[2]), int(r[3])) for r in recs)
    assert got == sorted(expect)

    def tiles(first, ql, off):
        return 0 if first >= ql else (min(first + qtok, ql) - 1 + off + 128) // 128

    costs = []
    for r in recs:
        pr, ql, kl = int(r[0]) & 0xFFFF, int(r[2]), int(r[3])
        na, nb = tiles(pr * 2 * qtok, ql, kl - ql), tiles(pr * 2 * qtok + qtok, ql, kl - ql)
        costs.append(2 * max(na, nb) + (1 if nb > 0 else 0))
    assert all(costs[i] >= costs[i + 1] for i in range(n - 1))
