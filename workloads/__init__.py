"""Seeded synthetic inputs for the paged GQA attention path.

This module is shared by the tests, the benchmark and the CPU oracle's callers.
It only draws random numbers and lays out metadata (sequence lengths, which
physical block ids each sequence owns, random values).  It holds none of the
path's arithmetic: no slot formula, no attention, no sampling.  Both the CUDA
path and the oracle receive the arrays built here and nothing else.

Shapes follow Qwen3-0.6B's attention (16 query heads, 8 KV heads, head_dim
128, bf16) with the engine's default KV block of 256 tokens.  The nano-vLLM
offline explainer (3479845.xyz/nano-vllm/nano-vllm-offline, "accuracy & scope"
box) gives 256 as the default block size and requires a multiple of 256.

Every workload is a :class:`PagedWorkload`: per sequence, the number of new
(query) tokens this step, the number of keys it attends to after this step's
KV write, and a block table (logical block -> physical block id, padded with
-1).  Physical ids come from a seeded random permutation of the pool, so
consecutive logical blocks are scattered over the pool as a paging allocator
would leave them.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np
import torch

QWEN3_0_6B = dict(num_heads=16, num_kv_heads=8, head_dim=128, block_size=256)
VOCAB_QWEN3 = 151936


@dataclasses.dataclass
class PagedWorkload:
    name: str
    q_lens: np.ndarray            # int32 [B]: new tokens of each sequence this step
    kv_lens: np.ndarray           # int32 [B]: keys attended, including this step's tokens
    block_tables: np.ndarray      # int32 [B, max_blocks], -1 padded
    num_blocks: int               # physical blocks in the pool (per layer)
    seed: int
    num_heads: int = 16
    num_kv_heads: int = 8
    head_dim: int = 128
    block_size: int = 256
    num_layers: int = 1
    shared_groups: Optional[list] = None   # [(seq ids, shared block ids)] for prefix sharing

    @property
    def batch(self) -> int:
        return int(self.q_lens.shape[0])

    @property
    def total_q(self) -> int:
        return int(self.q_lens.sum())

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def cu_seqlens_q(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.q_lens)]).astype(np.int32)

    @property
    def cu_seqlens_k(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.kv_lens)]).astype(np.int32)

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def kv_bytes_read(self) -> int:
        """Bytes of K and V one attention pass reads per layer (bf16)."""
        return int(self.kv_lens.astype(np.int64).sum()) * 2 * self.num_kv_heads * self.head_dim * 2

    def referenced_blocks(self) -> np.ndarray:
        ids = self.block_tables[self.block_tables >= 0]
        return np.unique(ids)

    def unreferenced_blocks(self) -> np.ndarray:
        return np.setdiff1d(np.arange(self.num_blocks), self.referenced_blocks())


def _blocks_for(n_tokens: int, block_size: int) -> int:
    return -(-int(n_tokens) // block_size)


def _tables_from_perm(owned: Sequence[Sequence[int]], width: int) -> np.ndarray:
    bt = np.full((len(owned), max(width, 1)), -1, dtype=np.int32)
    for s, ids in enumerate(owned):
        bt[s, : len(ids)] = np.asarray(ids, dtype=np.int32)
    return bt


def build_workload(name: str, q_lens, kv_lens, seed: int, *, pool_factor: float = 1.25,
                   num_blocks: Optional[int] = None, capacity_tokens=None,
                   shared_prefix_blocks=None, group_size: int = 4, num_layers: int = 1,
                   **shape) -> PagedWorkload:
    """Lay out a paged batch.

    ``capacity_tokens[s]`` (default ``kv_lens[s]``) is the number of token
    positions sequence ``s`` owns blocks for.  ``shared_prefix_blocks[g]`` is
    the number of whole leading blocks that all sequences of group ``g``
    (``group_size`` consecutive sequences) share by using the same physical
    ids, as a prefix cache hit leaves them.
    """
    shp = dict(QWEN3_0_6B)
    shp.update(shape)
    bs = shp["block_size"]
    rng = np.random.default_rng(seed)
    q_lens = np.asarray(q_lens, dtype=np.int32)
    kv_lens = np.asarray(kv_lens, dtype=np.int32)
    cap = kv_lens if capacity_tokens is None else np.asarray(capacity_tokens, dtype=np.int64)
    B = len(q_lens)
    need = [_blocks_for(c, bs) for c in cap]
    groups = []
    shared_total = 0
    if shared_prefix_blocks is not None:
        for g, c in enumerate(shared_prefix_blocks):
            members = list(range(g * group_size, min(B, (g + 1) * group_size)))
            groups.append((members, int(c)))
            shared_total += int(c)
    private = sum(need) - sum(c * len(m) for m, c in groups)
    used = private + shared_total
    if num_blocks is None:
        num_blocks = int(math.ceil(pool_factor * used))
    if used > num_blocks:
        raise ValueError(f"pool of {num_blocks} blocks cannot hold {used}")
    perm = rng.permutation(num_blocks).astype(np.int32)
    cursor = 0
    owned = [[] for _ in range(B)]
    shared_groups = []
    for members, c in groups:
        ids = perm[cursor: cursor + c].tolist()
        cursor += c
        for s in members:
            owned[s].extend(ids)
        shared_groups.append((members, ids))
    for s in range(B):
        rest = need[s] - len(owned[s])
        owned[s].extend(perm[cursor: cursor + rest].tolist())
        cursor += rest
    bt = _tables_from_perm(owned, max(need) if need else 1)
    return PagedWorkload(name=name, q_lens=q_lens, kv_lens=kv_lens, block_tables=bt,
                         num_blocks=int(num_blocks), seed=seed, num_layers=num_layers,
                         shared_groups=shared_groups or None, **shp)


# ---------------------------------------------------------------------------
# The five reference workloads.  Data seed = 1000 + index of the workload.
# ---------------------------------------------------------------------------

TINY_KV_LENS = (37, 256, 300, 511)


def tiny_prefill(seed: int = 1001) -> PagedWorkload:
    """Tiny single-layer check, step 1: a prefill of all tokens, no prefix hit.

    Pool of 16 physical blocks; every sequence owns blocks for one more token
    than its prompt so that the following decode step fits."""
    kl = np.array(TINY_KV_LENS, dtype=np.int32)
    return build_workload("tiny-prefill", kl, kl, seed, num_blocks=16, capacity_tokens=kl + 1)


def tiny_decode(seed: int = 1001) -> PagedWorkload:
    """Tiny single-layer check, step 2: one decode token per sequence on top of
    :func:`tiny_prefill` (same block tables), context lengths 38/257/301/512."""
    pre = tiny_prefill(seed)
    kl = pre.kv_lens + 1
    return dataclasses.replace(pre, name="tiny-decode", q_lens=np.ones_like(kl), kv_lens=kl)


def decode_b64(seed: int = 1002, batch: int = 64, lo: int = 512, hi: int = 4096) -> PagedWorkload:
    """Decode attention, one layer: batch 64, context lengths uniform in [512, 4096],
    pool = 1.25x the blocks used, block ids a random permutation of the pool."""
    rng = np.random.default_rng(seed)
    kl = rng.integers(lo, hi + 1, size=batch).astype(np.int32)
    return build_workload(f"decode-b{batch}", np.ones(batch, np.int32), kl, seed + 7)


def prefill_prefix(seed: int = 1003, batch: int = 32, lo: int = 100, hi: int = 1024,
                   group_size: int = 4) -> PagedWorkload:
    """Varlen prefill with prefix-cache hits: 32 prompts, lengths uniform in [100, 1024].

    Groups of 4 consecutive sequences share 0-2 whole leading 256-token blocks
    (same physical ids, so those blocks have reference count 4).  The shared
    count is clamped so every sequence keeps at least one new token; the new
    tokens are the ones after the shared prefix."""
    rng = np.random.default_rng(seed)
    bs = QWEN3_0_6B["block_size"]
    kl = rng.integers(lo, hi + 1, size=batch).astype(np.int32)
    n_groups = -(-batch // group_size)
    shared = []
    for g in range(n_groups):
        members = kl[g * group_size:(g + 1) * group_size]
        c = int(rng.integers(0, 3))
        c = min(c, (int(members.min()) - 1) // bs)
        shared.append(c)
    ql = kl.copy()
    for g, c in enumerate(shared):
        ql[g * group_size:(g + 1) * group_size] -= c * bs
    return build_workload(f"prefill-prefix-b{batch}", ql, kl, seed + 7,
                          shared_prefix_blocks=shared, group_size=group_size)


def long_decode(seed: int = 1004, batch: int = 8, lo: int = 16384, hi: int = 40960,
                pool: int = 1400) -> PagedWorkload:
    """Long-context decode: batch 8, context lengths uniform in [16384, 40960],
    physical blocks permuted across a pool of 1400 blocks."""
    rng = np.random.default_rng(seed)
    kl = rng.integers(lo, hi + 1, size=batch).astype(np.int32)
    return build_workload(f"long-decode-b{batch}", np.ones(batch, np.int32), kl, seed + 7,
                          num_blocks=pool)


def full_step(seed: int = 1005, batch: int = 256, lo: int = 128, hi: int = 2048,
              num_layers: int = 28) -> PagedWorkload:
    """Full decode step, Qwen3-0.6B-shaped: 28 layers of paged decode attention,
    batch 256, context lengths uniform in [128, 2048] (the same for every
    layer).  Every layer has its own K/V pool of 1.25x the blocks used; as in
    the engine, one block table per sequence indexes every layer's pool."""
    rng = np.random.default_rng(seed)
    kl = rng.integers(lo, hi + 1, size=batch).astype(np.int32)
    return build_workload(f"full-step-b{batch}-l{num_layers}", np.ones(batch, np.int32), kl,
                          seed + 7, num_layers=num_layers)


ALL = {
    "tiny-prefill": tiny_prefill,
    "tiny-decode": tiny_decode,
    "decode-b64": decode_b64,
    "prefill-prefix": prefill_prefix,
    "long-decode": long_decode,
    "full-step": full_step,
}


# ---------------------------------------------------------------------------
# Values.  All draws are N(0, 1) rounded to bf16 unless stated.
# ---------------------------------------------------------------------------

def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, seed: int, device="cpu", std: float = 1.0) -> torch.Tensor:
    """N(0, std^2) drawn in fp32 with a seeded generator on ``device``, rounded to bf16.

    The same seed gives different values on CPU and CUDA generators; callers
    that compare against the oracle either draw on the CPU and copy, or copy
    the drawn tensor back before any kernel touches it."""
    shape = tuple(int(s) for s in shape)
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    if out.numel() == 0:
        return out
    g = _gen(seed, device)
    flat = out.view(-1)
    step = 1 << 27
    for i in range(0, flat.numel(), step):
        n = min(step, flat.numel() - i)
        flat[i:i + n] = (torch.randn(n, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)
    return out


@dataclasses.dataclass
class PagedValues:
    q: torch.Tensor          # [total_q, Hq, d] bf16
    k_new: torch.Tensor      # [total_q, Hkv, d] bf16: this step's keys
    v_new: torch.Tensor      # [total_q, Hkv, d] bf16
    k_cache: torch.Tensor    # [num_blocks, bs, Hkv, d] bf16: history (stale where unused)
    v_cache: torch.Tensor


def paged_values(wl: PagedWorkload, device="cpu", layer: int = 0,
                 poison_unreferenced: bool = False) -> PagedValues:
    """Seeded Q / new K / new V and a pool holding the cached history.

    The pool is filled entirely with N(0,1) draws: slots a sequence has not
    reached yet simply hold stale values, as a reused block does.  With
    ``poison_unreferenced`` every block no sequence references is NaN."""
    base = wl.seed * 1000 + layer * 10
    Hq, Hkv, d, bs = wl.num_heads, wl.num_kv_heads, wl.head_dim, wl.block_size
    T = wl.total_q
    q = normal_bf16((T, Hq, d), base + 1, device)
    k_new = normal_bf16((T, Hkv, d), base + 2, device)
    v_new = normal_bf16((T, Hkv, d), base + 3, device)
    k_cache = normal_bf16((wl.num_blocks, bs, Hkv, d), base + 4, device)
    v_cache = normal_bf16((wl.num_blocks, bs, Hkv, d), base + 5, device)
    if poison_unreferenced:
        unused = torch.as_tensor(wl.unreferenced_blocks(), dtype=torch.long, device=device)
        if unused.numel():
            k_cache[unused] = float("nan")
            v_cache[unused] = float("nan")
    return PagedValues(q, k_new, v_new, k_cache, v_cache)


@dataclasses.dataclass
class SamplerInputs:
    logits: torch.Tensor        # [B, V] fp32, N(0, 3^2)
    temperatures: torch.Tensor  # [B] fp32, uniform in [0.5, 1.0]
    seed: int                   # noise seed
    offset: int                 # noise row offset


def sampler_inputs(batch: int = 256, vocab: int = VOCAB_QWEN3, seed: int = 1005, step: int = 0,
                   device="cpu", std: float = 3.0, t_lo: float = 0.5, t_hi: float = 1.0) -> SamplerInputs:
    """Logits N(0, std^2) fp32, per-request temperature uniform in [t_lo, t_hi],
    exponential-noise seed 2000 + step."""
    g = _gen(seed * 1000 + 7, device)
    logits = torch.randn((batch, vocab), generator=g, device=device, dtype=torch.float32) * std
    gt = _gen(seed * 1000 + 8, "cpu")
    temps = (t_lo + (t_hi - t_lo) * torch.rand((batch,), generator=gt, dtype=torch.float32)).to(device)
    return SamplerInputs(logits, temps, 2000 + step, 0)
