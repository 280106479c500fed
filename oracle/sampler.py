"""Oracle: exponential noise and the temperature sampler's exponential race.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Sources:

* Visual atlas (diomchen.github.io/reference/visual-atlas.html), fig. 23:
  the engine implements temperature sampling only, as an exponential race:
  the winner is argmin(e/p), equivalently argmax(p/e), with e ~ Exp(1) drawn
  per vocabulary entry and p = softmax(logits / T).  It is not argmax(p).
* nano-vLLM interactive guide (blog-mushroom.pages.dev), chapter 09
  (sampling): temperature reshapes the distribution the draw is made from.

Reading where the pages are silent: the engine draws its Exp(1) noise from the
framework's RNG, which is not portable.  Both this oracle and the CUDA sampler
instead derive it from Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel
random numbers: as easy as 1, 2, 3", SC'11), keyed by the seed, counting over
(row, column):

    counter = (column // 4, row + offset (low 32 bits), (row + offset) >> 32, 0)
    key     = (seed low 32 bits, seed high 32 bits)
    x       = Philox4x32-10(counter, key)[column % 4]
    u       = (2 * (x >> 9) + 1) * 2**-24          # odd multiple of 2**-24, in (0, 1)
    e       = -ln(u)

``u`` is exact in float32 and never 0 or 1, so ``e`` is finite and positive.
The race itself is evaluated here in float64 exactly as the figure states it.
"""
from __future__ import annotations

import numpy as np

MASK32 = np.uint64(0xFFFFFFFF)
# Philox4x32 round multipliers and Weyl key increments (SC'11, Philox4x32).
PHILOX_M0 = np.uint64(0xD2511F53)
PHILOX_M1 = np.uint64(0xCD9E8D57)
PHILOX_W0 = np.uint64(0x9E3779B9)
PHILOX_W1 = np.uint64(0xBB67AE85)
PHILOX_ROUNDS = 10


def philox4x32(counter, key, rounds: int = PHILOX_ROUNDS) -> np.ndarray:
    """Philox4x32-R on arrays of counters.

    counter: uint [..., 4]; key: uint [..., 2] (broadcast).  Each round takes
    the 64-bit products of counter words 0 and 2 with the two multipliers and
    mixes their high and low halves with words 1, 3 and the key; the key is
    bumped by the Weyl constants between rounds."""
    c = np.asarray(counter, dtype=np.uint64) & MASK32
    k = np.asarray(key, dtype=np.uint64) & MASK32
    c0, c1, c2, c3 = (c[..., i].copy() for i in range(4))
    k0 = np.broadcast_to(k[..., 0], c0.shape).copy()
    k1 = np.broadcast_to(k[..., 1], c0.shape).copy()
    for r in range(rounds):
        if r:
            k0 = (k0 + PHILOX_W0) & MASK32
            k1 = (k1 + PHILOX_W1) & MASK32
        p0 = PHILOX_M0 * c0            # < 2**64: exact in uint64
        p1 = PHILOX_M1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & MASK32
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return np.stack([c0, c1, c2, c3], axis=-1).astype(np.uint32)


def noise_bits(seed: int, offset: int, rows, vocab: int) -> np.ndarray:
    """Raw 32-bit Philox word for every (row, column): uint32 [len(rows), vocab]."""
    rows = np.asarray(list(rows), dtype=np.uint64)
    n_quads = -(-vocab // 4)
    r = rows + np.uint64(offset)
    ctr = np.zeros((len(rows), n_quads, 4), dtype=np.uint64)
    ctr[..., 0] = np.arange(n_quads, dtype=np.uint64)[None, :]      # column // 4
    ctr[..., 1] = (r & MASK32)[:, None]
    ctr[..., 2] = (r >> np.uint64(32))[:, None]
    key = np.array([seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF], dtype=np.uint64)
    words = philox4x32(ctr.reshape(-1, 4), key).reshape(len(rows), n_quads * 4)
    return words[:, :vocab]                                          # word column % 4


def uniforms(seed: int, offset: int, rows, vocab: int) -> np.ndarray:
    """u = (2 * (x >> 9) + 1) / 2**24 in float64 (exact; also exact in float32)."""
    x = noise_bits(seed, offset, rows, vocab).astype(np.uint64)
    return (2.0 * (x >> np.uint64(9)).astype(np.float64) + 1.0) * 2.0 ** -24


def exponential_noise(seed: int, offset: int, rows, vocab: int) -> np.ndarray:
    """e = -ln(u) ~ Exp(1), float64 [len(rows), vocab]."""
    return -np.log(uniforms(seed, offset, rows, vocab))


def exponential_race(logits, temperatures, noise):
    """Winner of each row's exponential race (atlas fig. 23), float64.

    p = softmax(logits / T); winner = argmax_v p_v / e_v, lowest index on ties.
    Returns (ids int64 [B], log_margin float64 [B]) where log_margin is
    ln(r_best / r_second), the row's distance from a tie."""
    logits = np.asarray(logits, dtype=np.float64)
    noise = np.asarray(noise, dtype=np.float64)
    B = logits.shape[0]
    ids = np.empty(B, dtype=np.int64)
    margin = np.empty(B, dtype=np.float64)
    for b in range(B):
        z = logits[b] / float(temperatures[b])
        z = z - z.max()
        p = np.exp(z)
        p = p / p.sum()
        r = p / noise[b]
        best = int(np.argmax(r))
        ids[b] = best
        if r.shape[0] > 1:
            second = np.partition(r, -2)[-2]
            margin[b] = np.log(r[best]) - np.log(second) if second > 0 else np.inf
        else:
            margin[b] = np.inf
    return ids, margin


def sample(logits, temperatures, seed: int, offset: int = 0):
    """Exponential race with the Philox noise for rows 0..B-1."""
    logits = np.asarray(logits)
    B, V = logits.shape
    e = exponential_noise(seed, offset, range(B), V)
    return exponential_race(logits, temperatures, e)
