"""Supported shapes beyond the benchmark's: block sizes that are other multiples of
256 tokens, other KV-head counts, and every supported group size (query heads per
KV head: MHA 1, GQA 2, 4 and 8; atlas fig. 18 draws MHA, GQA and MQA), through the
slot mapping, the scatter, prefill, decode and the fused decode, against the
fp64 oracle.  Lengths are chosen to sit on and next to block edges."""
import numpy as np
import pytest
import torch

import workloads as W
from pkv_testutil import GpuBatch, assert_attention_close, bits, expect_no_device_error

pytestmark = pytest.mark.gpu

SHAPES = {
    "block512": dict(block_size=512),
    "block1024": dict(block_size=1024),
    "heads4-2": dict(num_heads=4, num_kv_heads=2),
    "heads8-4": dict(num_heads=8, num_kv_heads=4),
    "heads32-16": dict(num_heads=32, num_kv_heads=16),
    "mha16-16": dict(num_heads=16, num_kv_heads=16),
    "gqa16-4": dict(num_heads=16, num_kv_heads=4),
    "gqa16-2": dict(num_heads=16, num_kv_heads=2),
    "gqa32-4": dict(num_heads=32, num_kv_heads=4),
    "mqa8-1": dict(num_heads=8, num_kv_heads=1),
}

# prefill: whole prompts, chunks after a prefix that ends mid-block, single-token chunks
PREFILL_Q = [37, 300, 129, 1, 64, 700, 513]
PREFILL_K = [37, 812, 429, 1025, 64, 700, 1537]
# decode: context lengths around block edges of every supported size
DECODE_L = [1, 255, 256, 257, 511, 512, 513, 1024, 1025, 1500, 3000, 4096]


@pytest.mark.parametrize("shape", list(SHAPES), ids=list(SHAPES))
def test_prefill_other_shapes(pkv, shape):
    wl = W.build_workload("shape-prefill", PREFILL_Q, PREFILL_K, seed=41, **SHAPES[shape])
    b = GpuBatch(wl, W.paged_values(wl, poison_unreferenced=True))
    b.run_slots_and_store(pkv, decode=False)
    assert np.array_equal(b.slots.cpu().numpy().astype(np.int64), b.oracle_slots())
    out = b.run_prefill(pkv)
    assert_attention_close(out, b.oracle_prefill(), f"prefill {shape}")
    # the same attention on a plan made once (its tag covers the group size and block size)
    hq, hkv, d = b.q.shape[1], b.k_cache.shape[2], b.q.shape[2]
    mq, mk = int(wl.q_lens.max()), int(wl.kv_lens.max())
    ws = pkv.pkv_prefill_plan(b.cu_q, b.cu_k, wl.total_q, mq, mk, hq, hkv, d, wl.block_size, b.block_tables.shape[1])
    planned = pkv.pkv_prefill_varlen_planned(b.q, b.k_cache, b.v_cache, b.cu_q, b.cu_k, b.block_tables, mq, mk,
                                             wl.softmax_scale, ws)
    assert torch.equal(planned.view(torch.int16), out.view(torch.int16)), f"planned prefill {shape}"
    expect_no_device_error(pkv)


@pytest.mark.parametrize("shape", list(SHAPES), ids=list(SHAPES))
def test_decode_other_shapes(pkv, shape):
    wl = W.build_workload("shape-decode", np.ones(len(DECODE_L), np.int32), DECODE_L, seed=42, **SHAPES[shape])
    b = GpuBatch(wl, W.paged_values(wl, poison_unreferenced=True))
    b.run_slots_and_store(pkv, decode=True)
    out = b.run_decode(pkv)
    assert_attention_close(out, b.oracle_decode(), f"decode {shape}")
    expect_no_device_error(pkv)


@pytest.mark.parametrize("shape", list(SHAPES), ids=list(SHAPES))
def test_decode_append_other_shapes(pkv, shape):
    """The fused write: pools and slots bit-exact, output against the oracle."""
    wl = W.build_workload("shape-append", np.ones(len(DECODE_L), np.int32), DECODE_L, seed=43, **SHAPES[shape])
    b = GpuBatch(wl, W.paged_values(wl, poison_unreferenced=True))
    slots = torch.full((wl.batch,), -7, dtype=torch.int32, device="cuda")
    out = pkv.pkv_decode_append(b.q, b.k_new, b.v_new, b.k_cache, b.v_cache, b.block_tables, b.kv_lens,
                                int(wl.kv_lens.max()), wl.softmax_scale, slot_mapping=slots)
    kc, vc = b.oracle_pools()
    assert np.array_equal(slots.cpu().numpy().astype(np.int64), b.oracle_slots())
    assert np.array_equal(bits(b.k_cache), bits(torch.from_numpy(kc).to(torch.bfloat16)))
    assert np.array_equal(bits(b.v_cache), bits(torch.from_numpy(vc).to(torch.bfloat16)))
    assert_attention_close(out, b.oracle_decode(pools=(kc, vc)), f"decode_append {shape}")
    expect_no_device_error(pkv)
