"""Steps captured in a CUDA graph and replayed (atlas fig. 26: a replay reads
new inputs from pre-allocated buffers; shapes and addresses are fixed, values
may change).  The captured decode step -- two layers of pkv_decode_append and
pkv_sample_dev, whose noise offset lives in device memory and advances inside
the graph -- and the captured prefill step (slot mapping, KV scatter, prefill)
must give, replay after replay, exactly what the eager calls give."""
import numpy as np
import pytest
import torch

import workloads as W
from pkv_testutil import GpuBatch, bits, expect_no_device_error

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
