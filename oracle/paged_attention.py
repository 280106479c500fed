"""Oracle: slot mapping, KV scatter and paged GQA attention, in float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Sources (page title and figure/section):

* Visual atlas (diomchen.github.io/reference/visual-atlas.html), the
  dimension walk-through figure "T=5, block_size=2, block_table=[3,0,4]":
  each token's logical block is ``pos // block_size``, its offset
  ``pos % block_size``, its physical block ``block_table[logical]`` and its
  slot in the flat pool ``physical * block_size + offset``.
* Same atlas, figure "two requests of length 3 and 2 ... cu_seqlens=[0,3,5]":
  variable-length requests are packed row after row; ``cu_seqlens`` holds the
  running start offsets and recovers each request's rows.
* Same atlas, figs. 16-17: attention = softmax(scale * Q K^T + mask) V, the
  causal mask keeps the diagonal, and a cached chunk keeps its position
  offset, so a non-square [q_len, k_len] mask is aligned to the bottom right,
  not the top-left tril.
* Same atlas, fig. 18 and the figure "two [3,2] Q heads point to the same K/V
  head": several query heads read one K/V head; K/V are shared, not copied.
* Same atlas, fig. 21 ("a decode step's real work"): the last sampled token
  has no KV yet; the step writes it and then attends over the whole history.
* Same atlas, fig. 22: naive attention materialises the full score and
  probability matrices; that is exactly what this oracle does.
* Nano-vLLM overview (wsj040303.github.io/notes/inference/nano-vllm/
  01-overview.html), the Sequence counters: after prompt [A,B,C] samples D the
  sequence has 4 tokens but only 3 with KV; the next decode feeds D.  Hence a
  decode step's context length counts the new token whose KV it writes.
* nano-vLLM offline explainer (3479845.xyz/nano-vllm/nano-vllm-offline),
  detail 02: the pool is reserved up front; blocks carry a contiguous logical
  sequence without being contiguous themselves; a block's unused tail slots
  stay unused.  Atlas fig. 25: a freed block is not zeroed, so nothing may
  depend on slots past a sequence's length.

Readings where the pages are silent:

* query head ``h`` uses KV head ``h // (Hq // Hkv)`` (consecutive grouping);
* ``slot < 0`` marks a padding row the scatter skips;
* block tables are padded with -1 past a sequence's last block.
"""
from __future__ import annotations

import numpy as np


# ---------------------------------------------------------------------------
# Slot mapping and scatter
# ---------------------------------------------------------------------------

def slot_of(block_table_row, pos: int, block_size: int) -> int:
    """Slot of logical position ``pos`` (atlas, slot worked-example figure)."""
    logical_block = pos // block_size
    offset = pos % block_size
    physical_block = int(block_table_row[logical_block])
    return physical_block * block_size + offset


def new_token_positions(q_len: int, kv_len: int) -> range:
    """Positions of a sequence's new tokens: the last ``q_len`` of its ``kv_len``.

    A prefix-cache hit leaves ``kv_len - q_len`` positions already cached
    (atlas fig. 26); a decode step has ``q_len = 1`` at position
    ``kv_len - 1`` (overview, Sequence counters)."""
    return range(kv_len - q_len, kv_len)


def slot_mapping(q_lens, kv_lens, block_tables, block_size: int) -> np.ndarray:
    """Slot of every new token, in packed (varlen) order."""
    out = []
    for s in range(len(q_lens)):
        for pos in new_token_positions(int(q_lens[s]), int(kv_lens[s])):
            out.append(slot_of(block_tables[s], pos, block_size))
    return np.asarray(out, dtype=np.int64)


def store_kvcache(k_cache, v_cache, k, v, slots, block_size: int):
    """Scatter row ``i`` of k/v to slot ``slots[i]`` of the pools; returns new pools.

    ``k_cache``/``v_cache`` are [num_blocks, block_size, Hkv, d]; ``k``/``v``
    are [N, Hkv, d].  A negative slot is a padding row and is skipped."""
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    for i, slot in enumerate(slots):
        slot = int(slot)
        if slot < 0:
            continue
        block, offset = divmod(slot, block_size)
        kc[block, offset] = k[i]
        vc[block, offset] = v[i]
    return kc, vc


# ---------------------------------------------------------------------------
# Varlen packing
# ---------------------------------------------------------------------------

def boundaries(cu_seqlens):
    """[(start, end)] of each packed request (atlas, cu_seqlens figure)."""
    cu = [int(x) for x in cu_seqlens]
    return [(cu[i], cu[i + 1]) for i in range(len(cu) - 1)]


def pack(padded, lengths):
    """Gather the first ``lengths[i]`` rows of each padded request into one array."""
    rows = []
    for i, n in enumerate(lengths):
        for t in range(int(n)):
            rows.append(padded[i][t])
    return np.asarray(rows)


# ---------------------------------------------------------------------------
# Attention
# ---------------------------------------------------------------------------

def gather_sequence(cache, block_table_row, n_tokens: int, block_size: int) -> np.ndarray:
    """Contiguous float64 copy of a sequence's first ``n_tokens`` cached rows."""
    out = np.empty((n_tokens,) + tuple(cache.shape[2:]), dtype=np.float64)
    for pos in range(n_tokens):
        block = int(block_table_row[pos // block_size])
        out[pos] = cache[block, pos % block_size]
    return out


def offset_causal_mask(q_len: int, k_len: int) -> np.ndarray:
    """Visible[i, j] for query i of a chunk whose first position is ``k_len - q_len``.

    Query ``i`` sits at absolute position ``i + (k_len - q_len)`` and sees every
    key at or before it (diagonal kept, atlas fig. 17)."""
    visible = np.zeros((q_len, k_len), dtype=bool)
    offset = k_len - q_len
    for i in range(q_len):
        visible[i, : i + offset + 1] = True
    return visible


def attention_dense(q, K, V, scale: float) -> np.ndarray:
    """Materialised causal GQA attention of one request (atlas figs. 16-18, 22).

    q: [q_len, Hq, d]; K, V: [k_len, Hkv, d] (the request's whole context in
    position order).  Returns [q_len, Hq, d] float64."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    q_len, Hq, d = q.shape
    k_len, Hkv, _ = K.shape
    group = Hq // Hkv
    visible = offset_causal_mask(q_len, k_len)
    out = np.empty((q_len, Hq, d), dtype=np.float64)
    for h in range(Hq):
        kv = h // group
        scores = scale * (q[:, h, :] @ K[:, kv, :].T)          # [q_len, k_len]
        scores = np.where(visible, scores, -np.inf)
        scores = scores - scores.max(axis=1, keepdims=True)
        probs = np.exp(scores)
        probs = probs / probs.sum(axis=1, keepdims=True)
        out[:, h, :] = probs @ V[:, kv, :]
    return out


def prefill_varlen(q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_tables,
                   block_size: int, scale: float) -> np.ndarray:
    """Varlen prefill: every request attends to its paged context.

    q is packed [total_q, Hq, d]; request s owns rows cu_seqlens_q[s]..[s+1]
    and has cu_seqlens_k[s+1]-cu_seqlens_k[s] keys in the pool (its new
    tokens' KV already written).  Returns packed [total_q, Hq, d] float64."""
    q = np.asarray(q)
    out = np.zeros(q.shape, dtype=np.float64)
    qb = boundaries(cu_seqlens_q)
    kb = boundaries(cu_seqlens_k)
    for s, ((q0, q1), (k0, k1)) in enumerate(zip(qb, kb)):
        q_len, k_len = q1 - q0, k1 - k0
        if q_len == 0:
            continue
        K = gather_sequence(k_cache, block_tables[s], k_len, block_size)
        V = gather_sequence(v_cache, block_tables[s], k_len, block_size)
        out[q0:q1] = attention_dense(q[q0:q1], K, V, scale)
    return out


def decode(q, k_cache, v_cache, block_tables, context_lens, block_size: int,
           scale: float) -> np.ndarray:
    """One decode token per sequence over ``context_lens[b]`` cached keys.

    q: [B, Hq, d].  A sequence with no context gives a zero row.  Every
    sequence is :func:`decode_rows` of its own row."""
    return decode_rows(q, k_cache, v_cache, block_tables, context_lens, block_size, scale,
                       range(np.asarray(q).shape[0]))


def decode_rows(q, k_cache, v_cache, block_tables, context_lens, block_size: int,
                scale: float, rows) -> np.ndarray:
    """Decode attention for the listed sequences, in the listed order.

    Row ``i`` of the result is sequence ``rows[i]``: its query token
    ``q[rows[i]]`` attends over the first ``context_lens[rows[i]]`` positions
    of its paged context (atlas fig. 21, with the KV of the newest token
    already written).  A sequence with no context gives a zero row."""
    rows = list(rows)
    q = np.asarray(q)
    out = np.zeros((len(rows),) + tuple(q.shape[1:]), dtype=np.float64)
    for i, b in enumerate(rows):
        L = int(context_lens[b])
        if L == 0:
            continue
        K = gather_sequence(k_cache, block_tables[b], L, block_size)
        V = gather_sequence(v_cache, block_tables[b], L, block_size)
        out[i] = attention_dense(q[b:b + 1], K, V, scale)[0]
    return out
