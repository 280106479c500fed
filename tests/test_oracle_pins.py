"""Pins for the CPU oracle: values the pages print, closed forms, invariants,
library routines and brute force -- never the oracle's own formula retyped.

Each test names the plausible oracle mistake it would catch."""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import paged_attention as pa
from oracle import sampler as sm

from conftest import GOLDEN


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# Slot mapping and scatter
# ---------------------------------------------------------------------------

def test_slot_worked_example():
    """Atlas slot figure T=5, bs=2, table=[3,0,4] (catches swapped // and %, wrong table index)."""
    g = _golden("slot_worked_example.json")
    slots = [pa.slot_of(g["block_table"], p, g["block_size"]) for p in range(g["T"])]
    assert slots == g["slot"]
    mapped = pa.slot_mapping([g["T"]], [g["T"]], np.array([g["block_table"]]), g["block_size"])
    assert mapped.tolist() == g["slot"]


def _allocator_walk(table, n_tokens, block_size):
    """Independent construction: append tokens one at a time, moving to the next
    table entry whenever the current block fills (no division or modulo)."""
    out = []
    logical, offset = 0, 0
    for _ in range(n_tokens):
        out.append((int(table[logical]), offset))
        offset += 1
        if offset == block_size:
            logical, offset = logical + 1, 0
    return out


@pytest.mark.parametrize("block_size", [2, 4, 256])
def test_slot_matches_allocator_walk(block_size):
    rng = np.random.default_rng(block_size)
    n = 3 * block_size + 5
    table = rng.permutation(16)[: -(-n // block_size)]
    for pos, (blk, off) in enumerate(_allocator_walk(table, n, block_size)):
        assert pa.slot_of(table, pos, block_size) == blk * block_size + off


def test_slot_mapping_new_tokens_are_the_tail():
    """Decode token sits at position L-1 ([A,B,C]->D counter example); a prefix hit
    of c tokens leaves positions c..kl-1 new (catches off-by-one in the offset)."""
    table = np.array([[5, 2, 7]])
    assert pa.slot_mapping([1], [4], table, 2).tolist() == [2 * 2 + 1]      # pos 3 -> block 2, off 1
    assert pa.slot_mapping([2], [5], table, 2).tolist() == [2 * 2 + 1, 7 * 2 + 0]


def test_store_kvcache_scatter_and_skip():
    rng = np.random.default_rng(0)
    kc = rng.standard_normal((6, 4, 2, 3))
    vc = rng.standard_normal((6, 4, 2, 3))
    k = rng.standard_normal((3, 2, 3))
    v = rng.standard_normal((3, 2, 3))
    slots = [9, -1, 22]
    nk, nv = pa.store_kvcache(kc, vc, k, v, slots, 4)
    assert np.array_equal(nk[2, 1], k[0]) and np.array_equal(nv[2, 1], v[0])
    assert np.array_equal(nk[5, 2], k[2]) and np.array_equal(nv[5, 2], v[2])
    changed = np.zeros(kc.shape[:2], bool)
    changed[2, 1] = changed[5, 2] = True
    assert np.array_equal(nk[~changed], kc[~changed])
    assert np.array_equal(nv[~changed], vc[~changed])
    assert np.array_equal(kc, kc)  # inputs untouched (copies returned)


# ---------------------------------------------------------------------------
# Varlen packing and the offset causal mask
# ---------------------------------------------------------------------------

def test_cu_seqlens_example():
    g = _golden("varlen_cu_seqlens.json")
    assert pa.boundaries(g["cu_seqlens"]) == [(0, 3), (3, 5)]
    padded = np.arange(np.prod(g["padded_shape"])).reshape(g["padded_shape"])
    packed = pa.pack(padded, g["lengths"])
    assert list(packed.shape) == g["packed_shape"]
    for row, (r, t) in zip(packed, g["packed_source_rows"]):
        assert np.array_equal(row, padded[r, t])


def test_offset_mask_2x5():
    g = _golden("offset_mask_2x5.json")
    m = pa.offset_causal_mask(g["q_len"], g["k_len"])
    assert m.astype(int).tolist() == g["visible"]
    assert m.astype(int).tolist() != g["top_left_tril_for_contrast"]


@pytest.mark.parametrize("n", [1, 2, 7])
def test_square_mask_is_tril(n):
    assert np.array_equal(pa.offset_causal_mask(n, n), np.tril(np.ones((n, n), bool)))


# ---------------------------------------------------------------------------
# Attention
# ---------------------------------------------------------------------------

def _sdpa_causal(q, K, V, scale):
    """torch's scaled_dot_product_attention (CPU, fp64), square causal, GQA."""
    qt = torch.from_numpy(np.ascontiguousarray(q.transpose(1, 0, 2)))[None]
    kt = torch.from_numpy(np.ascontiguousarray(K.transpose(1, 0, 2)))[None]
    vt = torch.from_numpy(np.ascontiguousarray(V.transpose(1, 0, 2)))[None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=scale,
                                                         enable_gqa=True)
    return o[0].numpy().transpose(1, 0, 2)


def test_attention_square_equals_library_sdpa():
    """Catches a dropped scale, transposed operand, wrong head map or mask sign."""
    rng = np.random.default_rng(1)
    q = rng.standard_normal((7, 4, 8))
    K = rng.standard_normal((7, 2, 8))
    V = rng.standard_normal((7, 2, 8))
    np.testing.assert_allclose(pa.attention_dense(q, K, V, 0.37), _sdpa_causal(q, K, V, 0.37),
                               rtol=0, atol=1e-12)


@pytest.mark.parametrize("q_len,k_len", [(1, 9), (3, 9), (2, 5), (9, 9)])
def test_chunk_equals_tail_of_full_causal(q_len, k_len):
    """A chunk of the last q_len queries over k_len keys is the last q_len rows of
    square causal attention over all k_len positions (bottom-right alignment)."""
    rng = np.random.default_rng(q_len * 100 + k_len)
    q_full = rng.standard_normal((k_len, 4, 8))
    K = rng.standard_normal((k_len, 2, 8))
    V = rng.standard_normal((k_len, 2, 8))
    ref = _sdpa_causal(q_full, K, V, 0.5)[k_len - q_len:]
    np.testing.assert_allclose(pa.attention_dense(q_full[k_len - q_len:], K, V, 0.5), ref,
                               rtol=0, atol=1e-12)


def test_gqa_equals_mha_on_repeated_kv():
    """K/V shared by consecutive query heads equals MHA on K/V repeated per head."""
    rng = np.random.default_rng(2)
    q = rng.standard_normal((5, 6, 4))
    K = rng.standard_normal((8, 3, 4))
    V = rng.standard_normal((8, 3, 4))
    mha = pa.attention_dense(q, np.repeat(K, 2, axis=1), np.repeat(V, 2, axis=1), 0.4)
    np.testing.assert_allclose(pa.attention_dense(q, K, V, 0.4), mha, rtol=0, atol=1e-13)


def test_single_key_returns_its_value():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 4, 8))
    K = rng.standard_normal((1, 2, 8))
    V = rng.standard_normal((1, 2, 8))
    o = pa.attention_dense(q, K, V, 1.0)
    for h in range(4):
        np.testing.assert_array_equal(o[0, h], V[0, h // 2])


def test_identical_keys_give_prefix_means():
    rng = np.random.default_rng(4)
    q_len, k_len = 3, 7
    q = rng.standard_normal((q_len, 2, 8))
    K = np.broadcast_to(rng.standard_normal((1, 1, 8)), (k_len, 1, 8)).copy()
    V = rng.standard_normal((k_len, 1, 8))
    o = pa.attention_dense(q, K, V, 0.9)
    for i in range(q_len):
        n_vis = i + (k_len - q_len) + 1
        for h in range(2):
            np.testing.assert_allclose(o[i, h], V[:n_vis, 0].mean(axis=0), rtol=0, atol=1e-13)


def test_dominant_key_selects_its_value_without_overflow():
    rng = np.random.default_rng(5)
    K = rng.standard_normal((6, 1, 4))
    V = rng.standard_normal((6, 1, 4))
    q = (K[4, 0] * 1e4)[None, None, :]
    o = pa.attention_dense(q, K, V, 1.0)
    assert np.all(np.isfinite(o))
    np.testing.assert_allclose(o[0, 0], V[4, 0], atol=1e-12)


def _random_paged(rng, kv_lens, bs, n_blocks, Hkv=2, d=8):
    need = [-(-int(L) // bs) for L in kv_lens]
    perm = rng.permutation(n_blocks)
    tables = np.full((len(kv_lens), max(need)), -1)
    cur = 0
    for s, n in enumerate(need):
        tables[s, :n] = perm[cur:cur + n]
        cur += n
    kc = rng.standard_normal((n_blocks, bs, Hkv, d))
    vc = rng.standard_normal((n_blocks, bs, Hkv, d))
    return tables, kc, vc


def _contiguous(cache, table, n, bs):
    """Brute force via the allocator walk, independent of the oracle's gather."""
    return np.stack([cache[b, o] for b, o in _allocator_walk(table, n, bs)])


def test_paged_prefill_equals_contiguous_and_permutation_invariant():
    rng = np.random.default_rng(6)
    bs = 4
    kv_lens = np.array([9, 4, 13])
    q_lens = np.array([9, 2, 5])                   # seq 1, 2: prefix hits
    tables, kc, vc = _random_paged(rng, kv_lens, bs, 12)
    q = rng.standard_normal((q_lens.sum(), 4, 8))
    cu_q = np.concatenate([[0], np.cumsum(q_lens)])
    cu_k = np.concatenate([[0], np.cumsum(kv_lens)])
    out = pa.prefill_varlen(q, kc, vc, cu_q, cu_k, tables, bs, 0.3)
    for s in range(3):
        K = _contiguous(kc, tables[s], kv_lens[s], bs)
        V = _contiguous(vc, tables[s], kv_lens[s], bs)
        ref = _sdpa_causal(np.concatenate([np.zeros((kv_lens[s] - q_lens[s], 4, 8)), q[cu_q[s]:cu_q[s + 1]]]),
                           K, V, 0.3)[kv_lens[s] - q_lens[s]:]
        np.testing.assert_allclose(out[cu_q[s]:cu_q[s + 1]], ref, rtol=0, atol=1e-12)
    # relabel the physical blocks: physical i moves to pi[i]
    pi = rng.permutation(12)
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[pi] = kc
    vc2[pi] = vc
    tables2 = np.where(tables >= 0, pi[np.maximum(tables, 0)], -1)
    out2 = pa.prefill_varlen(q, kc2, vc2, cu_q, cu_k, tables2, bs, 0.3)
    np.testing.assert_array_equal(out, out2)


def test_unused_slots_do_not_matter():
    """Freed blocks are not zeroed: NaN anywhere a sequence has not reached must not leak."""
    rng = np.random.default_rng(7)
    bs = 4
    kv_lens = np.array([6, 3])
    tables, kc, vc = _random_paged(rng, kv_lens, bs, 8)
    q = rng.standard_normal((2, 4, 8))
    ref = pa.decode(q, kc, vc, tables, kv_lens, bs, 0.5)
    kp, vp = kc.copy(), vc.copy()
    used = set()
    for s, L in enumerate(kv_lens):
        for b, o in _allocator_walk(tables[s], L, bs):
            used.add((b, o))
    for b in range(8):
        for o in range(bs):
            if (b, o) not in used:
                kp[b, o] = np.nan
                vp[b, o] = np.nan
    out = pa.decode(q, kp, vp, tables, kv_lens, bs, 0.5)
    assert np.all(np.isfinite(out))
    np.testing.assert_array_equal(out, ref)


def test_decode_equals_last_prefill_row():
    rng = np.random.default_rng(8)
    bs = 4
    kv_lens = np.array([7, 1, 12])
    tables, kc, vc = _random_paged(rng, kv_lens, bs, 10)
    q = rng.standard_normal((kv_lens.sum(), 4, 8))
    cu = np.concatenate([[0], np.cumsum(kv_lens)])
    pre = pa.prefill_varlen(q, kc, vc, cu, cu, tables, bs, 0.25)
    last = q[cu[1:] - 1]
    dec = pa.decode(last, kc, vc, tables, kv_lens, bs, 0.25)
    np.testing.assert_allclose(dec, pre[cu[1:] - 1], rtol=0, atol=1e-13)


def test_decode_zero_context_is_zero_row():
    rng = np.random.default_rng(9)
    tables, kc, vc = _random_paged(rng, [3], 4, 2)
    out = pa.decode(rng.standard_normal((2, 4, 8)), kc, vc, np.vstack([tables, tables]),
                    np.array([3, 0]), 4, 0.5)
    assert np.all(out[1] == 0) and np.any(out[0] != 0)


def test_decode_rows_selects_rows_in_the_listed_order():
    """decode_rows(rows)[i] is sequence rows[i] attending its paged context: checked against
    torch's SDPA on the allocator-walk copy of each listed sequence (a library reference that
    shares nothing with the oracle's gather), with the rows listed out of order, one of them
    twice and one with no context (its row is zero).  Catches indexing q or the tables by the
    output position instead of the sequence."""
    rng = np.random.default_rng(41)
    bs = 4
    kv_lens = np.array([5, 0, 11, 2, 8])
    tables, kc, vc = _random_paged(rng, np.maximum(kv_lens, 1), bs, 12)
    q = rng.standard_normal((5, 4, 8))
    rows = [4, 1, 2, 0, 4]
    out = pa.decode_rows(q, kc, vc, tables, kv_lens, bs, 0.35, rows)
    assert out.shape == (len(rows), 4, 8)
    for i, b in enumerate(rows):
        L = int(kv_lens[b])
        if L == 0:
            assert np.all(out[i] == 0)
            continue
        K = _contiguous(kc, tables[b], L, bs)
        V = _contiguous(vc, tables[b], L, bs)
        ref = _sdpa_causal(np.concatenate([np.zeros((L - 1, 4, 8)), q[b:b + 1]]), K, V, 0.35)[-1]
        np.testing.assert_allclose(out[i], ref, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(out, pa.decode(q, kc, vc, tables, kv_lens, bs, 0.35)[rows])


# ---------------------------------------------------------------------------
# Philox noise and the exponential race
# ---------------------------------------------------------------------------

def test_philox_known_answers():
    g = _golden("philox4x32_10_kat.json")
    for vec in g["vectors"]:
        ctr = np.array([[int(x, 16) for x in vec["counter"]]], dtype=np.uint64)
        key = np.array([int(x, 16) for x in vec["key"]], dtype=np.uint64)
        out = sm.philox4x32(ctr, key)[0]
        assert [int(x) for x in out] == [int(x, 16) for x in vec["output"]]


def test_uniforms_are_exact_odd_multiples_inside_unit_interval():
    u = sm.uniforms(seed=123, offset=5, rows=range(3), vocab=1001)
    k = u * 2.0 ** 24
    assert np.all(k == np.round(k)) and np.all(k.astype(np.int64) % 2 == 1)
    assert np.all((u > 0) & (u < 1))
    assert np.array_equal(u.astype(np.float32).astype(np.float64), u)


def test_exponential_noise_moments():
    e = sm.exponential_noise(seed=7, offset=0, rows=range(50), vocab=2000)
    n = e.size
    assert abs(e.mean() - 1.0) < 4 / math.sqrt(n)
    assert abs(e.var() - 1.0) < 4 * math.sqrt(8 / n)


def test_noise_depends_on_row_offset_and_seed():
    a = sm.noise_bits(1, 0, [3], 64)
    assert np.array_equal(a, sm.noise_bits(1, 3, [0], 64))
    assert not np.array_equal(a, sm.noise_bits(2, 0, [3], 64))
    assert not np.array_equal(a, sm.noise_bits(1, 0, [4], 64))


def test_race_with_unit_noise_is_argmax_and_real_noise_is_not():
    rng = np.random.default_rng(10)
    logits = rng.standard_normal((64, 50)) * 3
    T = rng.uniform(0.5, 1.0, 64)
    ids, _ = sm.exponential_race(logits, T, np.ones_like(logits))
    assert np.array_equal(ids, logits.argmax(axis=1))
    ids_noise, _ = sm.sample(logits, T, seed=11)
    assert np.any(ids_noise != ids)


def test_race_invariances():
    """Shift of all logits: same ids.  (logits*c, T*c): same ids (catches a dropped T)."""
    rng = np.random.default_rng(12)
    logits = rng.standard_normal((32, 40)) * 3
    T = rng.uniform(0.5, 1.0, 32)
    e = sm.exponential_noise(5, 0, range(32), 40)
    ids, _ = sm.exponential_race(logits, T, e)
    assert np.array_equal(sm.exponential_race(logits + 17.0, T, e)[0], ids)
    assert np.array_equal(sm.exponential_race(logits * 4.0, T * 4.0, e)[0], ids)
    ids_hot, _ = sm.exponential_race(logits, T * 50, e)
    assert np.any(ids_hot != ids)


def test_race_margin_closed_form():
    """Hand-picked 3-token rows where the race's two best ratios are known exactly.

    Row 0: logits ln(1), ln(2), ln(3) at T = 1, so p = (1, 2, 3) / 6; noise (1, 1, 2)
    gives p/e = (1, 2, 1.5) / 6: winner 1, margin ln(2 / 1.5) = ln(4/3).
    Row 1: logits (0, ln 3, ln 2) * 0.5 at T = 0.5 (p = (1, 3, 2) / 6); noise (0.25, 2, 1)
    gives p/e = (4, 1.5, 2) / 6: winner 0, margin ln(4 / 2) = ln 2, the second best not
    adjacent to the winner.  A margin taken against the wrong entry, from p*e, or without
    the temperature fails one of them."""
    logits = np.array([[0.0, math.log(2.0), math.log(3.0)],
                       [0.0, 0.5 * math.log(3.0), 0.5 * math.log(2.0)]])
    T = np.array([1.0, 0.5])
    e = np.array([[1.0, 1.0, 2.0], [0.25, 2.0, 1.0]])
    ids, margin = sm.exponential_race(logits, T, e)
    assert ids.tolist() == [1, 0]
    np.testing.assert_allclose(margin, [math.log(4.0 / 3.0), math.log(2.0)], rtol=0, atol=1e-14)


def test_race_frequencies_match_softmax():
    """The exponential race draws v with probability p_v (catches p*e, argmax p, e vs 1/e)."""
    p = np.array([0.1, 0.2, 0.3, 0.4])
    T = 0.7
    logits = np.log(p) * T
    n = 40000
    e = sm.exponential_noise(99, 0, range(n), 4)
    ids, _ = sm.exponential_race(np.broadcast_to(logits, (n, 4)), np.full(n, T), e)
    freq = np.bincount(ids, minlength=4) / n
    sigma = np.sqrt(p * (1 - p) / n)
    assert np.all(np.abs(freq - p) < 4 * sigma), (freq, p)


# ---------------------------------------------------------------------------
# Rotary position embedding (atlas fig. 19)
# ---------------------------------------------------------------------------

from oracle import rope as rp


def test_rope_single_pair_is_the_2d_rotation():
    """d = 2: one pair, frequency base^0 = 1, so the angle is the position itself."""
    x = np.array([[[0.6, -1.3]]])
    for pos in (0.0, 1.0, 2.5, 7.0):
        out = rp.rope(x, [pos], base=1e6)[0, 0]
        c, s = math.cos(pos), math.sin(pos)
        np.testing.assert_allclose(out, [0.6 * c + 1.3 * s, -1.3 * c + 0.6 * s], rtol=0, atol=1e-15)
    # quarter turn: (1, 0) -> (0, 1), counter-clockwise
    np.testing.assert_allclose(rp.rope(np.array([[[1.0, 0.0]]]), [math.pi / 2], 1e6)[0, 0], [0.0, 1.0], atol=1e-15)


def test_rope_identity_at_zero_and_norm_per_pair():
    rng = np.random.default_rng(30)
    x = rng.standard_normal((3, 2, 8))
    np.testing.assert_array_equal(rp.rope(x, [0, 0, 0], 1e4), x)
    y = rp.rope(x, [1, 17, 300], 1e4)
    for i in range(4):
        np.testing.assert_allclose(np.hypot(y[..., i], y[..., i + 4]), np.hypot(x[..., i], x[..., i + 4]),
                                   rtol=1e-13)


def test_rope_composes_and_inverts():
    rng = np.random.default_rng(31)
    x = rng.standard_normal((1, 3, 16))
    a = rp.rope(rp.rope(x, [5], 1e4), [11], 1e4)
    np.testing.assert_allclose(a, rp.rope(x, [16], 1e4), rtol=0, atol=1e-12)
    np.testing.assert_allclose(rp.rope(rp.rope(x, [9], 1e4), [-9], 1e4), x, rtol=0, atol=1e-12)


def test_rope_scores_depend_only_on_relative_position():
    """<R(m) q, R(n) k> = <R(m-n) q, k>: what makes RoPE a position encoding for attention."""
    rng = np.random.default_rng(32)
    q = rng.standard_normal((1, 1, 32))
    k = rng.standard_normal((1, 1, 32))
    for m, n in [(10, 3), (100, 64), (7, 7)]:
        lhs = float(np.sum(rp.rope(q, [m], 1e6) * rp.rope(k, [n], 1e6)))
        rhs = float(np.sum(rp.rope(q, [m - n], 1e6) * k))
        assert lhs == pytest.approx(rhs, abs=1e-10)


def test_rope_store_rotates_q_and_k_not_v():
    rng = np.random.default_rng(33)
    q = rng.standard_normal((2, 4, 8))
    k = rng.standard_normal((2, 2, 8))
    v = rng.standard_normal((2, 2, 8))
    kc = np.zeros((2, 4, 2, 8))
    vc = np.zeros((2, 4, 2, 8))
    qr, kc2, vc2 = rp.rope_store_kvcache(q, kc, vc, k, v, [3, 5], [1, 6], 4, 1e4)
    np.testing.assert_array_equal(vc2[0, 1], v[0])
    np.testing.assert_array_equal(vc2[1, 2], v[1])
    np.testing.assert_allclose(kc2[1, 2], rp.rope(k, [3, 5], 1e4)[1], atol=1e-15)
    np.testing.assert_allclose(qr, rp.rope(q, [3, 5], 1e4), atol=1e-15)


def test_rope_pairing_and_frequencies_closed_form():
    """d = 4, base = 100: pair 0 = elements (0, 2) at frequency 1, pair 1 = elements (1, 3) at
    frequency 100^(-2/4) = 0.1.  Catches an interleaved pairing or a wrong exponent."""
    for p in (0.0, 1.0, 3.0, 250.0):
        out = rp.rope(np.array([[[1.0, 1.0, 0.0, 0.0]]]), [p], base=100.0)[0, 0]
        np.testing.assert_allclose(out, [math.cos(p), math.cos(0.1 * p), math.sin(p), math.sin(0.1 * p)],
                                   rtol=0, atol=1e-13)


def test_rotate_pair_is_the_counter_clockwise_rotation():
    """rotate_pair, the figure's single pair: a quarter turn takes (1, 0) to (0, 1) and (0, 1) to
    (-1, 0); a half turn negates; any turn keeps the length; arrays of pairs turn elementwise."""
    np.testing.assert_allclose(rp.rotate_pair(1.0, 0.0, math.pi / 2), (0.0, 1.0), atol=1e-15)
    np.testing.assert_allclose(rp.rotate_pair(0.0, 1.0, math.pi / 2), (-1.0, 0.0), atol=1e-15)
    np.testing.assert_allclose(rp.rotate_pair(0.3, -0.8, math.pi), (-0.3, 0.8), atol=1e-15)
    a, b = rp.rotate_pair(np.array([3.0, 0.5]), np.array([4.0, -2.0]), np.array([0.7, 2.9]))
    np.testing.assert_allclose(np.hypot(a, b), [5.0, math.hypot(0.5, 2.0)], rtol=1e-15)
    np.testing.assert_allclose(a[0], 3.0 * math.cos(0.7) - 4.0 * math.sin(0.7), rtol=1e-15)
