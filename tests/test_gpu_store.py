"""a1 slot mapping and a2 KV scatter on the GPU: bit-exact against the oracle."""
import json
import os

import numpy as np
import pytest
import torch

import workloads as W
from oracle import paged_attention as pa
from conftest import GOLDEN
from pkv_testutil import GpuBatch, bits, expect_no_device_error, f32

pytestmark = pytest.mark.gpu


def test_slot_mapping_worked_example(pkv):
    g = json.load(open(os.path.join(GOLDEN, "slot_worked_example.json")))
    bt = torch.tensor([g["block_table"]], dtype=torch.int32, device="cuda")
    cu = torch.tensor([0, g["T"]], dtype=torch.int32, device="cuda")
    slots = torch.empty(g["T"], dtype=torch.int32, device="cuda")
    pkv.pkv_slot_mapping(bt, 5, g["block_size"], slots, cu_seqlens_q=cu, cu_seqlens_k=cu)
    assert slots.cpu().tolist() == g["slot"]
    expect_no_device_error(pkv)


@pytest.mark.parametrize("name", ["tiny-prefill", "tiny-decode", "prefill-prefix", "decode-b64", "long-decode"])
def test_slot_mapping_matches_oracle(pkv, name):
    wl = W.ALL[name]()
    bt = torch.from_numpy(wl.block_tables).cuda()
    slots = torch.full((wl.total_q,), -7, dtype=torch.int32, device="cuda")
    if name.endswith("decode"):
        pkv.pkv_slot_mapping(bt, wl.num_blocks, wl.block_size, slots,
                             context_lens=torch.from_numpy(wl.kv_lens).cuda())
    else:
        pkv.pkv_slot_mapping(bt, wl.num_blocks, wl.block_size, slots,
                             cu_seqlens_q=torch.from_numpy(wl.cu_seqlens_q).cuda(),
                             cu_seqlens_k=torch.from_numpy(wl.cu_seqlens_k).cuda())
    ref = pa.slot_mapping(wl.q_lens, wl.kv_lens, wl.block_tables, wl.block_size)
    assert np.array_equal(slots.cpu().numpy().astype(np.int64), ref)
    expect_no_device_error(pkv)


def test_slot_mapping_flags_bad_tables(pkv):
    # seq 0: position 600 needs logical block 2 of a 2-wide table; seq 1: block id outside the pool
    bt = torch.tensor([[0, 1], [9, 2]], dtype=torch.int32, device="cuda")
    ctx = torch.tensor([601, 3], dtype=torch.int32, device="cuda")
    slots = torch.zeros(2, dtype=torch.int32, device="cuda")
    pkv.pkv_slot_mapping(bt, 4, 256, slots, context_lens=ctx)
    assert slots.cpu().tolist() == [-1, -1]
    code, _ = pkv.pkv_get_device_error(clear=True)
    assert code in (1, 6)


@pytest.mark.parametrize("name", ["tiny-prefill", "prefill-prefix", "decode-b64"])
def test_store_kvcache_bit_exact(pkv, name):
    wl = W.ALL[name]()
    b = GpuBatch(wl, W.paged_values(wl, poison_unreferenced=True))
    b.run_slots_and_store(pkv, decode=name.startswith("decode"))
    kc, vc = b.oracle_pools()
    assert np.array_equal(bits(b.k_cache), bits(torch.from_numpy(kc).to(torch.bfloat16)))
    assert np.array_equal(bits(b.v_cache), bits(torch.from_numpy(vc).to(torch.bfloat16)))
    expect_no_device_error(pkv)


@pytest.mark.parametrize("n", [3, 2048])
def test_store_skips_padding_and_flags_out_of_pool(pkv, n):
    """Slot -1 (padding) is skipped and a slot past the pool is flagged, for a handful of
    tokens and for a prefill-sized batch of 2048."""
    nb, bs = 16, 256
    g = torch.Generator().manual_seed(51)
    k = torch.randn(n, 8, 128, generator=g).to(torch.bfloat16).cuda()
    v = torch.randn(n, 8, 128, generator=g).to(torch.bfloat16).cuda()
    kc = torch.zeros(nb, bs, 8, 128, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    slots = torch.randperm(nb * bs, generator=g)[:n].to(torch.int32)
    pad = torch.arange(n) % 7 == 1                 # every seventh token is padding
    slots[pad] = -1
    bad = n - 1 if n > 3 else 2                    # exactly one slot past the pool
    slots[bad] = nb * bs + 3
    pkv.pkv_store_kvcache(k, v, slots.cuda(), kc, vc)
    torch.cuda.synchronize()
    ok = (slots >= 0) & (slots < nb * bs)
    flat_k, flat_v = kc.view(nb * bs, 8, 128).cpu(), vc.view(nb * bs, 8, 128).cpu()
    assert torch.equal(flat_k[slots[ok].long()], k.cpu()[ok]) and torch.equal(flat_v[slots[ok].long()], v.cpu()[ok])
    untouched = torch.ones(nb * bs, dtype=torch.bool)
    untouched[slots[ok].long()] = False
    assert int(flat_k[untouched].count_nonzero()) == 0 and int(flat_v[untouched].count_nonzero()) == 0
    code, info = pkv.pkv_get_device_error(clear=True)
    assert code == 2 and info == bad


@pytest.mark.parametrize("n", [37, 3000])
def test_store_from_fused_qkv_rows(pkv, n):
    """k and v may be strided views into one [n, (16+8+8)*128] projection output."""
    nb, bs = 16, 256
    qkv = torch.randn(n, (16 + 8 + 8) * 128, device="cuda").to(torch.bfloat16)
    k = qkv[:, 16 * 128:24 * 128].view(n, 8, 128)
    v = qkv[:, 24 * 128:].view(n, 8, 128)
    kc = torch.zeros(nb, bs, 8, 128, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    perm = torch.randperm(nb * bs)[:n].to(torch.int32).cuda()
    pkv.pkv_store_kvcache(k, v, perm, kc, vc)
    ref_k, ref_v = pa.store_kvcache(f32(kc), f32(vc), f32(k), f32(v), perm.cpu().numpy(), bs)
    assert np.array_equal(f32(kc), ref_k) and np.array_equal(f32(vc), ref_v)
    expect_no_device_error(pkv)
