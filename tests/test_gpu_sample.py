"""a5 exponential-race sampler on the GPU against the oracle.

The kernel decides the argmax in fp32 on the monotone form logits/T - ln e;
the oracle evaluates the race literally in fp64.  Ids must be identical on
every row whose oracle log-margin between the two best candidates exceeds
NEAR_TIE (far above fp32 rounding of the key); on a near-tie row either of the
oracle's two best candidates is accepted, and such rows are counted."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import sampler as sm
from pkv_testutil import NEAR_TIE, check_sampler_ids as _check_ids

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("vocab", [1000, 1001, 7])
def test_sample_small_vs_oracle(pkv, vocab):
    s = W.sampler_inputs(batch=96, vocab=vocab, seed=31, device="cpu")
    ids = pkv.pkv_sample(s.logits.cuda(), s.temperatures.cuda(), s.seed, s.offset)
    _check_ids(ids, s.logits, s.temperatures, s.seed, s.offset)
    code, _ = pkv.pkv_get_device_error(clear=True)
    assert code == 0


@pytest.mark.parametrize("step", [0, 1, 3])
def test_sample_full_vocab_vs_oracle(pkv, step):
    """The full decode step's sampler, [256, 151936] logits, with the noise of several steps
    (steps 1 and 3 each held rows whose winner's noise u sits within a few 2^-24 of 1)."""
    s = W.sampler_inputs(batch=256, vocab=W.VOCAB_QWEN3, seed=1005, step=step, device="cpu")
    ids = pkv.pkv_sample(s.logits.cuda(), s.temperatures.cuda(), s.seed, s.offset)
    _check_ids(ids, s.logits, s.temperatures, s.seed, s.offset)


def test_sample_noise_next_to_one_is_ranked_exactly(pkv):
    """An element whose noise u lies within a few 2^-24 of 1 has a tiny e = -ln u and so a key
    about 16 above its scaled logit: the elements most likely to win.  Its key must come out
    exact.  The oracle's generator finds such an element; its row is rebuilt so that this
    element's exact key sits 0.3 below, then 0.3 above, one competitor in another slice of
    the row (every other logit far below), and the ids must follow the oracle both times."""
    V, seed = W.VOCAB_QWEN3, 9001
    found = None
    for r0 in range(0, 512, 32):
        x = sm.noise_bits(seed, 0, range(r0, r0 + 32), V) >> np.uint32(9)
        hits = np.argwhere(x >= np.uint32((1 << 23) - 4))
        if len(hits):
            found = (r0 + int(hits[0][0]), int(hits[0][1]))
            break
    assert found is not None
    row, v = found
    c = (v + V // 2) % V                                   # a competitor in another eighth of the row
    e = sm.exponential_noise(seed, row, [0], V)[0]          # the noise of that row (offset = row)
    assert e[v] < 1e-6
    for delta in (-0.3, 0.3):
        lg = np.full(V, -60.0)
        lg[c] = 0.0
        key_c = lg[c] + np.log(1.0 / e[c])
        lg[v] = key_c + delta + np.log(e[v])                 # exact key of v = key_c + delta
        logits = torch.tensor(lg, dtype=torch.float32).reshape(1, V)
        temps = torch.ones(1)
        ids = pkv.pkv_sample(logits.cuda(), temps.cuda(), seed, offset=row)
        ref, margin = sm.exponential_race(logits.double().numpy(), temps.double().numpy(), e[None, :])
        assert margin[0] > 0.1
        assert int(ids.item()) == int(ref[0]) == (v if delta > 0 else c)
    code, _ = pkv.pkv_get_device_error(clear=True)
    assert code == 0


def test_sample_row_offset_and_strided_rows(pkv):
    s = W.sampler_inputs(batch=16, vocab=3000, seed=32, device="cpu")
    wide = torch.zeros(16, 3100)
    wide[:, :3000] = s.logits
    view = wide.cuda()[:, :3000]
    ids = pkv.pkv_sample(view, s.temperatures.cuda(), seed=77, offset=1000)
    _check_ids(ids, s.logits, s.temperatures, 77, 1000)


def test_sample_rows_not_16_byte_aligned(pkv):
    """Rows that start off a 16-byte boundary (a view one column in, row stride 3002 floats)
    take the scalar-load path for every quad; ids must not change."""
    s = W.sampler_inputs(batch=16, vocab=3000, seed=33, device="cpu")
    wide = torch.zeros(16, 3002)
    wide[:, 1:3001] = s.logits
    view = wide.cuda()[:, 1:3001]
    assert view.data_ptr() % 16 != 0 and view.stride(0) % 4 != 0
    ids = pkv.pkv_sample(view, s.temperatures.cuda(), s.seed, s.offset)
    _check_ids(ids, s.logits, s.temperatures, s.seed, s.offset)


def test_sample_cold_temperature_is_argmax(pkv):
    g = torch.Generator().manual_seed(33)
    logits = torch.randn(64, 512, generator=g) * 3
    temps = torch.full((64,), 1e-4)
    ids = pkv.pkv_sample(logits.cuda(), temps.cuda(), seed=5)
    top2 = torch.topk(logits, 2, dim=1).values
    clear = (top2[:, 0] - top2[:, 1]) > 0.01
    assert torch.equal(ids.cpu()[clear], logits.argmax(dim=1)[clear])


def test_sample_invalid_temperature_flags_row(pkv):
    logits = torch.randn(3, 100).cuda()
    temps = torch.tensor([1.0, 0.0, 0.7]).cuda()
    ids = pkv.pkv_sample(logits, temps, seed=1)
    code, info = pkv.pkv_get_device_error(clear=True)
    assert ids.cpu()[1].item() == -1 and code == 4 and info == 1
    assert ids.cpu()[0].item() >= 0 and ids.cpu()[2].item() >= 0


def test_sample_frequencies_follow_softmax(pkv):
    """Many rows of one 4-token distribution: winner frequencies match p within 4 sigma."""
    p = np.array([0.1, 0.2, 0.3, 0.4])
    T = 0.7
    n = 20000
    logits = torch.from_numpy(np.log(p) * T).float().expand(n, 4).contiguous().cuda()
    ids = pkv.pkv_sample(logits, torch.full((n,), T).cuda(), seed=99)
    freq = np.bincount(ids.cpu().numpy(), minlength=4) / n
    assert np.all(np.abs(freq - p) < 4 * np.sqrt(p * (1 - p) / n)), freq


def test_sample_masked_and_nan_logits(pkv):
    """-inf logits (a masked vocabulary) never win and NaN logits never win; a row with a
    single finite logit returns it, a row with none returns -1.  The other rows match the
    oracle run on the same logits with NaN replaced by -inf."""
    s = W.sampler_inputs(batch=64, vocab=5000, seed=34, device="cpu")
    lg = s.logits.clone()
    g = torch.Generator().manual_seed(35)
    lg[torch.rand(lg.shape, generator=g) < 0.9] = -float("inf")
    lg[0, :] = -float("inf")
    lg[0, 17] = 2.0
    lg[1, :] = -float("inf")
    nan_at = torch.rand(lg.shape, generator=g) < 0.01
    nan_at[0, 17] = False
    lg[nan_at] = float("nan")
    ids = pkv.pkv_sample(lg.cuda(), s.temperatures.cuda(), s.seed, s.offset).cpu().numpy()
    assert ids[0] == 17 and ids[1] == -1
    rows = np.array([b for b in range(64) if b != 1])
    ref_in = lg.double().numpy()
    ref_in[np.isnan(ref_in)] = -np.inf
    e = sm.exponential_noise(s.seed, s.offset, range(64), lg.shape[1])
    ref, margin = sm.exponential_race(ref_in[rows], s.temperatures.double().numpy()[rows], e[rows])
    clear = margin >= NEAR_TIE
    assert np.array_equal(ids[rows][clear], ref[clear])
    assert np.all(np.isfinite(ref_in[rows, ids[rows]]))


def test_sample_offset_across_the_32_bit_boundary(pkv):
    """Counter word 2 is (row + offset) >> 32: an offset just below 2^32 puts the first rows at
    c2 = 0 and the rest at c2 = 1, and a seed with both halves set drives both key words."""
    s = W.sampler_inputs(batch=24, vocab=2051, seed=36, device="cpu")
    seed, offset = 0x123456789ABCDEF0, 2 ** 32 - 3
    ids = pkv.pkv_sample(s.logits.cuda(), s.temperatures.cuda(), seed, offset)
    _check_ids(ids, s.logits, s.temperatures, seed, offset)
