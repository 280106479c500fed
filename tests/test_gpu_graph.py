"""Steps captured in a CUDA graph and replayed (atlas fig. 26: a replay reads
new inputs from pre-allocated buffers; shapes and addresses are fixed, values
may change).  The captured decode step -- layers of pkv_decode_append and
pkv_sample_dev, whose noise offset lives in device memory and advances inside
the graph -- is checked against the oracle at the full decode step's shape
(batch 256, context U[128, 2048], full vocabulary), replay after replay with
new inputs; smaller captures, and the captured prefill step (slot mapping, KV
scatter, prefill), must give exactly what the eager calls give."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import paged_attention as pa
from pkv_testutil import (GpuBatch, assert_attention_close, bits, check_sampler_ids, expect_no_device_error,
                          f32)

pytestmark = pytest.mark.gpu


def test_decode_step_graph_replay_matches_eager(pkv):
    wl = W.decode_b64(batch=16, lo=100, hi=900)
    layers = [W.paged_values(wl, device="cuda", layer=i) for i in range(2)]
    eager_pools = [(v.k_cache.clone(), v.v_cache.clone()) for v in layers]
    bt = torch.from_numpy(wl.block_tables).cuda()
    ctx = torch.from_numpy(wl.kv_lens).cuda()
    ws = pkv.decode_workspace(wl.batch, wl.num_heads, wl.num_kv_heads, wl.head_dim)
    s_in = W.sampler_inputs(batch=wl.batch, vocab=5000, device="cuda")
    outs = [torch.empty_like(v.q) for v in layers]
    ids = torch.empty(wl.batch, dtype=torch.int64, device="cuda")
    seed_offset = torch.tensor([s_in.seed, 0], dtype=torch.int64, device="cuda")
    max_ctx = int(wl.kv_lens.max())

    def step(pools):
        for i, v in enumerate(layers):
            pkv.pkv_decode_append(v.q, v.k_new, v.v_new, pools[i][0], pools[i][1], bt, ctx, max_ctx,
                                  wl.softmax_scale, out=outs[i], workspace=ws)
        pkv.pkv_sample_dev(s_in.logits, s_in.temperatures, seed_offset, out_ids=ids)
        seed_offset[1:].add_(wl.batch)              # next replay draws fresh noise

    graph_pools = [(v.k_cache, v.v_cache) for v in layers]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(graph_pools)                            # first call on the device: set-up before capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(graph_pools)
    seed_offset[1] = 0
    for replay in range(2):
        g.replay()
        torch.cuda.synchronize()
        got_out = [bits(o).copy() for o in outs]
        got_ids = ids.cpu().clone()
        # eager: the same calls with the offset this replay used
        for i, v in enumerate(layers):
            ref = pkv.pkv_decode_append(v.q, v.k_new, v.v_new, eager_pools[i][0], eager_pools[i][1], bt, ctx,
                                        max_ctx, wl.softmax_scale, workspace=ws)
            assert np.array_equal(bits(ref), got_out[i])
        ref_ids = pkv.pkv_sample(s_in.logits, s_in.temperatures, s_in.seed, offset=replay * wl.batch)
        assert torch.equal(ref_ids.cpu(), got_ids)
    for i in range(2):
        assert np.array_equal(bits(eager_pools[i][0]), bits(graph_pools[i][0]))
    first = pkv.pkv_sample(s_in.logits, s_in.temperatures, s_in.seed, offset=0).cpu()
    second = pkv.pkv_sample(s_in.logits, s_in.temperatures, s_in.seed, offset=wl.batch).cpu()
    assert not torch.equal(first, second)            # the offset really changes the draw
    expect_no_device_error(pkv)


def test_sample_dev_equals_sample(pkv):
    s_in = W.sampler_inputs(batch=32, vocab=20000, seed=41, device="cuda")
    so = torch.tensor([12345, 77], dtype=torch.int64, device="cuda")
    a = pkv.pkv_sample_dev(s_in.logits, s_in.temperatures, so)
    b = pkv.pkv_sample(s_in.logits, s_in.temperatures, 12345, offset=77)
    assert torch.equal(a, b)
    expect_no_device_error(pkv)


def test_prepared_call_made_before_capture_is_captured(pkv):
    """A DecodeAppendCall built on the default stream and then called inside a capture must land in the
    graph: after new q values are copied into its buffer, a replay must give the eager result for them."""
    wl = W.decode_b64(batch=8, lo=100, hi=600)
    v = W.paged_values(wl, device="cuda")
    bt = torch.from_numpy(wl.block_tables).cuda()
    ctx = torch.from_numpy(wl.kv_lens).cuda()
    out = torch.empty_like(v.q)
    call = pkv.DecodeAppendCall(v.q, v.k_new, v.v_new, v.k_cache, v.v_cache, bt, ctx, int(wl.kv_lens.max()),
                                wl.softmax_scale, out=out)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    out.zero_()
    gen = torch.Generator().manual_seed(77)
    v.q.copy_(torch.randn(tuple(v.q.shape), generator=gen).to(torch.bfloat16).cuda())
    g.replay()
    torch.cuda.synchronize()
    ref = pkv.pkv_decode_append(v.q, v.k_new, v.v_new, v.k_cache, v.v_cache, bt, ctx, int(wl.kv_lens.max()),
                                wl.softmax_scale)
    assert np.array_equal(bits(out), bits(ref))
    expect_no_device_error(pkv)


def test_prefill_step_graph_replay_matches_eager(pkv):
    """Slot mapping, KV scatter and prefill of a chunked batch with prefix hits, captured once
    and replayed: bit-identical to the eager calls, also after new Q/K/V values are written into
    the captured buffers."""
    wl = W.prefill_prefix(batch=8)
    b = GpuBatch(wl, W.paged_values(wl))
    out = torch.empty_like(b.q)
    ws = torch.empty(max(pkv.pkv_prefill_workspace_size(wl.batch, wl.num_heads, wl.num_kv_heads, wl.head_dim,
                                                        int(wl.q_lens.max())), 256),
                     dtype=torch.uint8, device="cuda")
    mq, mk = int(wl.q_lens.max()), int(wl.kv_lens.max())

    def step():
        b.run_slots_and_store(pkv, decode=False)
        pkv.pkv_prefill_varlen(b.q, b.k_cache, b.v_cache, b.cu_q, b.cu_k, b.block_tables, mq, mk,
                               wl.softmax_scale, out=out, workspace=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()                                        # first call on the device: set-up before capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    gen = torch.Generator(device="cuda").manual_seed(71)
    for replay in range(2):
        if replay:                                    # new values, same buffers
            b.q.copy_(torch.randn(b.q.shape, generator=gen, device="cuda").to(torch.bfloat16))
            b.k_new.copy_(torch.randn(b.k_new.shape, generator=gen, device="cuda").to(torch.bfloat16))
            b.v_new.copy_(torch.randn(b.v_new.shape, generator=gen, device="cuda").to(torch.bfloat16))
        g.replay()
        torch.cuda.synchronize()
        got = bits(out).copy()
        b.run_slots_and_store(pkv, decode=False)
        ref = pkv.pkv_prefill_varlen(b.q, b.k_cache, b.v_cache, b.cu_q, b.cu_k, b.block_tables, mq, mk,
                                     wl.softmax_scale, workspace=ws)
        assert np.array_equal(bits(ref), got)
    expect_no_device_error(pkv)


def test_full_step_graph_replays_match_the_oracle(pkv):
    """Two layers of the full decode step (batch 256, context U[128, 2048], each layer its own
    pool) plus the sampler on [256, 151936] logits, captured once and replayed twice.  Before
    each replay new Q and new K/V rows are copied into the captured buffers; the noise offset
    advances inside the graph.  After each replay: every layer's output element by element
    against the oracle's decode on that replay's inputs, every layer's pool bit for bit
    against the oracle's scatter into the initial pool, and the ids against the oracle's race
    with that replay's offset."""
    wl = W.full_step(num_layers=2)
    n_layers, B = 2, wl.batch
    init = [W.paged_values(wl, device="cpu", layer=i) for i in range(n_layers)]
    pools = [(v.k_cache.cuda(), v.v_cache.cuda()) for v in init]
    qs = [v.q.cuda() for v in init]                          # the captured input buffers
    kns = [v.k_new.cuda() for v in init]
    vns = [v.v_new.cuda() for v in init]
    outs = [torch.empty_like(q) for q in qs]
    bt = torch.from_numpy(wl.block_tables).cuda()
    ctx = torch.from_numpy(wl.kv_lens).cuda()
    max_ctx = int(wl.kv_lens.max())
    ws = pkv.decode_workspace(B, wl.num_heads, wl.num_kv_heads, wl.head_dim)
    s_in = W.sampler_inputs(batch=B, device="cpu")
    logits, temps = s_in.logits.cuda(), s_in.temperatures.cuda()
    ids = torch.empty(B, dtype=torch.int64, device="cuda")
    seed_offset = torch.tensor([s_in.seed, 0], dtype=torch.int64, device="cuda")

    def step():
        for i in range(n_layers):
            pkv.pkv_decode_append(qs[i], kns[i], vns[i], pools[i][0], pools[i][1], bt, ctx, max_ctx,
                                  wl.softmax_scale, out=outs[i], workspace=ws)
        pkv.pkv_sample_dev(logits, temps, seed_offset, out_ids=ids)
        seed_offset[1:].add_(B)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()                                               # first call on the device: set-up before capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    torch.cuda.synchronize()
    for i in range(n_layers):                                # the captured step has not changed the pools yet;
        pools[i][0].copy_(init[i].k_cache)                   # the warm-up call's KV write is undone
        pools[i][1].copy_(init[i].v_cache)
    seed_offset[1] = 0

    # the oracle reads each layer's pool through a compact copy of the blocks the batch uses
    used = wl.referenced_blocks()
    remap = np.full(wl.num_blocks, -1, dtype=np.int64)
    remap[used] = np.arange(len(used))
    tables = np.where(wl.block_tables >= 0, remap[np.maximum(wl.block_tables, 0)], -1)
    slots = pa.slot_mapping(wl.q_lens, wl.kv_lens, tables, wl.block_size)
    unused = torch.from_numpy(wl.unreferenced_blocks()).long()
    used_t = torch.from_numpy(used).long()

    for replay in range(2):
        new = []
        for i in range(n_layers):                            # new values in the same buffers
            base = 77000 + 100 * replay + 10 * i
            q = W.normal_bf16(tuple(qs[i].shape), base + 1)
            kn = W.normal_bf16(tuple(kns[i].shape), base + 2)
            vn = W.normal_bf16(tuple(vns[i].shape), base + 3)
            qs[i].copy_(q)
            kns[i].copy_(kn)
            vns[i].copy_(vn)
            new.append((q, kn, vn))
        g.replay()
        torch.cuda.synchronize()
        expect_no_device_error(pkv)
        check_sampler_ids(ids, s_in.logits, s_in.temperatures, s_in.seed, offset=replay * B)
        for i in range(n_layers):
            q, kn, vn = new[i]
            kc, vc = pa.store_kvcache(f32(init[i].k_cache[used_t]), f32(init[i].v_cache[used_t]), f32(kn), f32(vn),
                                      slots, wl.block_size)
            ref = pa.decode(f32(q), kc, vc, tables, wl.kv_lens, wl.block_size, wl.softmax_scale)
            assert_attention_close(outs[i], ref, f"replay {replay}, layer {i}")
            got_k, got_v = pools[i][0].cpu(), pools[i][1].cpu()
            assert np.array_equal(bits(got_k[used_t]), bits(torch.from_numpy(kc).to(torch.bfloat16)))
            assert np.array_equal(bits(got_v[used_t]), bits(torch.from_numpy(vc).to(torch.bfloat16)))
            assert torch.equal(got_k[unused].view(torch.int16), init[i].k_cache[unused].view(torch.int16))
            del kc, vc, got_k, got_v
