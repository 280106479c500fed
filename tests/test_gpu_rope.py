"""f2 rotary embedding fused into the KV write, on the GPU, against the oracle.

Tolerance (rotated Q and K): the kernel reduces the angle exactly in
fixed-point turns, rotates in fp32 and rounds once to bf16, so each element is
within one bf16 rounding of the fp64 value, 2^-8 |ref|, plus the fp32 error of
the rotation, of the reduced angle (below 4e-7 rad, also at |position| near
2^31, where the oracle's own double angle is off by 2.4e-7 rad) and of the
hardware sine and cosine (4e-7 absolute each), together below 2e-6 of the
pair's norm.  V must be bit-exact."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import paged_attention as pa
from oracle import rope as rp
from pkv_testutil import bits, expect_no_device_error, f32

pytestmark = pytest.mark.gpu

BASE = 1e6     # Qwen3-0.6B's rotary base


def _assert_rotated_close(got, x, positions, base):
    ref = rp.rope(f32(x), positions, base)
    xd = f32(x)
    half = xd.shape[-1] // 2
    hyp = np.hypot(xd[..., :half], xd[..., half:])
    hyp = np.concatenate([hyp, hyp], axis=-1)
    err = np.abs(f32(got) - ref)
    tol = 2.0 ** -8 * np.abs(ref) + 2e-6 * hyp
    bad = err > tol
    assert not bad.any(), (int(bad.sum()), float((err - tol).max()))


def _rand(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g).to(torch.bfloat16)


@pytest.mark.parametrize("name", ["tiny-prefill", "prefill-prefix", "decode-b64"])
def test_rope_store_vs_oracle(pkv, name):
    wl = W.ALL[name]()
    n, hq, hkv, d = wl.total_q, 16, 8, 128
    slots = pa.slot_mapping(wl.q_lens, wl.kv_lens, wl.block_tables, wl.block_size).astype(np.int32)
    pos = np.concatenate([np.arange(kl - ql, kl) for ql, kl in zip(wl.q_lens, wl.kv_lens)]).astype(np.int32)
    q, k, v = _rand((n, hq, d), 1), _rand((n, hkv, d), 2), _rand((n, hkv, d), 3)
    pool = (wl.num_blocks, wl.block_size, hkv, d)
    kc0, vc0 = _rand(pool, 4), _rand(pool, 5)
    kc, vc = kc0.cuda(), vc0.cuda()
    q_out = pkv.pkv_rope_store_kvcache(q.cuda(), k.cuda(), v.cuda(), torch.from_numpy(pos).cuda(),
                                       torch.from_numpy(slots).cuda(), kc, vc, BASE)
    torch.cuda.synchronize()
    expect_no_device_error(pkv)
    _assert_rotated_close(q_out.cpu(), q, pos, BASE)
    # every slot that was not written keeps its old bits; written V rows are exact copies
    kcc, vcc = kc.cpu().view(-1, hkv, d), vc.cpu().view(-1, hkv, d)
    untouched = np.ones(kcc.shape[0], bool)
    untouched[slots] = False
    untouched = torch.from_numpy(untouched)
    slots = torch.from_numpy(slots).long()
    assert np.array_equal(bits(kcc[untouched]), bits(kc0.view(-1, hkv, d)[untouched]))
    assert np.array_equal(bits(vcc[untouched]), bits(vc0.view(-1, hkv, d)[untouched]))
    assert np.array_equal(bits(vcc[slots]), bits(v))
    _assert_rotated_close(kcc[slots], k, pos, BASE)


def test_rope_store_positions_zero_is_plain_store(pkv):
    """cos 0 = 1 and sin 0 = 0 exactly: at position 0 the call is the a2 scatter, bit for bit."""
    n, hkv, d, nb, bs = 40, 8, 128, 4, 256
    q, k, v = _rand((n, 16, d), 6).cuda(), _rand((n, hkv, d), 7).cuda(), _rand((n, hkv, d), 8).cuda()
    slots = torch.randperm(nb * bs, generator=torch.Generator().manual_seed(9))[:n].to(torch.int32).cuda()
    kc = torch.zeros(nb, bs, hkv, d, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    kc2, vc2 = torch.zeros_like(kc), torch.zeros_like(kc)
    q_out = pkv.pkv_rope_store_kvcache(q, k, v, torch.zeros(n, dtype=torch.int32, device="cuda"), slots, kc, vc,
                                       BASE)
    pkv.pkv_store_kvcache(k, v, slots, kc2, vc2)
    torch.cuda.synchronize()
    assert np.array_equal(bits(q_out), bits(q))
    assert np.array_equal(bits(kc), bits(kc2)) and np.array_equal(bits(vc), bits(vc2))


def test_rope_store_large_positions_and_bases(pkv):
    """Positions far beyond the context lengths (up to 2^31 - 1, and negative) and other bases:
    the angle is reduced in double, so accuracy does not decay with the position."""
    pos = np.array([0, 1, 40959, 40960, 1 << 20, (1 << 31) - 1, -5, 123457], np.int32)
    n, d = len(pos), 128
    for base in (1e4, 1e6, 5e5):
        q, k, v = _rand((n, 16, d), 10), _rand((n, 8, d), 11), _rand((n, 8, d), 12)
        kc = torch.zeros(1, 256, 8, d, dtype=torch.bfloat16, device="cuda")
        vc = torch.zeros_like(kc)
        slots = torch.arange(n, dtype=torch.int32, device="cuda")
        q_out = pkv.pkv_rope_store_kvcache(q.cuda(), k.cuda(), v.cuda(), torch.from_numpy(pos).cuda(), slots, kc, vc,
                                           base)
        torch.cuda.synchronize()
        _assert_rotated_close(q_out.cpu(), q, pos, base)
        _assert_rotated_close(kc.cpu()[0, :n], k, pos, base)


@pytest.mark.parametrize("head_dim", [64, 256])
def test_rope_store_other_head_dims(pkv, head_dim):
    n, hkv = 33, 4
    pos = np.arange(1000, 1000 + n, dtype=np.int32)
    q, k, v = _rand((n, 8, head_dim), 13), _rand((n, hkv, head_dim), 14), _rand((n, hkv, head_dim), 15)
    kc = torch.zeros(2, 256, hkv, head_dim, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    slots = torch.arange(n, dtype=torch.int32, device="cuda") * 3
    q_out = pkv.pkv_rope_store_kvcache(q.cuda(), k.cuda(), v.cuda(), torch.from_numpy(pos).cuda(), slots, kc, vc,
                                       BASE)
    torch.cuda.synchronize()
    _assert_rotated_close(q_out.cpu(), q, pos, BASE)
    written = kc.cpu().view(-1, hkv, head_dim)[slots.cpu().long()]
    _assert_rotated_close(written, k, pos, BASE)
    assert np.array_equal(bits(vc.cpu().view(-1, hkv, head_dim)[slots.cpu().long()]), bits(v))


def test_rope_store_in_place_strided_and_k_only(pkv):
    """q rotated in place inside one fused [n, (16+8+8)*128] projection row; k, v strided views;
    then a K-only call (q = None) on the same rows."""
    n, d, nb, bs = 29, 128, 2, 256
    qkv = _rand((n, (16 + 8 + 8) * d), 16).cuda()
    orig = qkv.clone()
    q = qkv[:, :16 * d].view(n, 16, d)
    k = qkv[:, 16 * d:24 * d].view(n, 8, d)
    v = qkv[:, 24 * d:].view(n, 8, d)
    pos = torch.arange(n, dtype=torch.int32).mul_(37).cuda()
    slots = torch.arange(n, dtype=torch.int32, device="cuda") + 100
    kc = torch.zeros(nb, bs, 8, d, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    r = pkv.pkv_rope_store_kvcache(q, k, v, pos, slots, kc, vc, BASE, q_out=q)
    torch.cuda.synchronize()
    assert r.data_ptr() == q.data_ptr()
    _assert_rotated_close(q.cpu(), orig[:, :16 * d].view(n, 16, d).cpu(), pos.cpu().numpy(), BASE)
    assert torch.equal(qkv[:, 16 * d:], orig[:, 16 * d:])        # k and v inputs untouched
    kc_q = kc.clone()
    kc.zero_()
    assert pkv.pkv_rope_store_kvcache(None, k, v, pos, slots, kc, vc, BASE) is None
    torch.cuda.synchronize()
    assert np.array_equal(bits(kc), bits(kc_q))
    expect_no_device_error(pkv)


def test_rope_store_skips_padding_and_flags_out_of_pool(pkv):
    n, d, nb, bs = 3, 128, 2, 256
    q, k, v = _rand((n, 16, d), 17).cuda(), _rand((n, 8, d), 18).cuda(), _rand((n, 8, d), 19).cuda()
    kc = torch.zeros(nb, bs, 8, d, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    pos = torch.tensor([3, 4, 5], dtype=torch.int32, device="cuda")
    slots = torch.tensor([7, -1, nb * bs], dtype=torch.int32, device="cuda")
    q_out = pkv.pkv_rope_store_kvcache(q, k, v, pos, slots, kc, vc, BASE)
    torch.cuda.synchronize()
    code, info = pkv.pkv_get_device_error(clear=True)
    assert code == 2 and info == 2
    _assert_rotated_close(q_out.cpu(), q.cpu(), [3, 4, 5], BASE)     # q rotated for every token
    assert torch.equal(vc[0, 7], v[0])
    kc[0, 7] = 0
    vc[0, 7] = 0
    assert int(kc.count_nonzero()) == 0 and int(vc.count_nonzero()) == 0
