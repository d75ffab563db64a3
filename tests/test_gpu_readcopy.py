"""GPU parity of the low-precision read copy (FP8 per-row, NVFP4).

* The copy quantised from an initial checkpoint, and the copy re-quantised at
  every fold (decode flush steps, commits that fold), are compared code by
  code and scale by scale with the oracle's codecs applied to the device's
  own FP32 checkpoint (both sides take the rounding decisions in float32).
* Decode outputs with the copy are compared element by element, within
  2e-4 * max(|ref|, 1e-3), with the oracle's read-copy output (the copy
  replaces S_ckpt only in the decayed S_ckpt q term).  Where the oracle's copy
  (quantised from its float64 checkpoint rounded to FP32) rounds an element
  differently from the device's copy, the expected output is shifted by the
  decayed product of the two copies' difference with q (tests/harness.py).
* Per window, the output error against the exact FP32-recurrence output must
  stay below 1% (FP8) / 6% (NVFP4) rel-L2 from the second window on and must
  not grow with the window index, because the copy never feeds the recurrence.
"""

import numpy as np
import pytest
import torch

from oracle import codecs
from tests.harness import Pair, assert_close
from workloads import configs
from workloads.configs import MAMBA2, LayerShape

pytestmark = pytest.mark.gpu


def _check_initial_copy(pair, mode, seqs):
    S0 = pair.wl.S0()[seqs]
    v = pair.cache.read_copy_views()
    if mode == "fp8":
        codes, sc = codecs.fp8_rows_quantize(S0)
        np.testing.assert_array_equal(v["codes"][seqs].cpu().numpy(), codes)
        np.testing.assert_array_equal(v["row_scale"][seqs].cpu().numpy(), sc)
    else:
        packed, bs, s = codecs.nvfp4_quantize(S0)
        np.testing.assert_array_equal(v["matrix_scale"][seqs].cpu().numpy(), s)
        np.testing.assert_array_equal(v["block_scale"][seqs].cpu().numpy(), bs)
        np.testing.assert_array_equal(v["codes"][seqs].cpu().numpy(), packed)


@pytest.mark.parametrize("mode", ["fp8", "nvfp4"])
@pytest.mark.parametrize("P,N", [(16, 16), (32, 64), (64, 128)])
def test_initial_quantisation_bit_exact(mode, P, N):
    shape = LayerShape(MAMBA2, batch=3, n_heads=4, n_groups=2, d_head=P, d_state=N, ring_len=4)
    pair = Pair(configs.Mamba2Workload(shape, seed=41, s0_std=0.1), read_mode=mode)
    _check_initial_copy(pair, mode, [0, 1, 2])
    assert pair.cache.device_error() == 0


def _rel_l2(a, b):
    return float(np.sqrt(np.sum((a - b) ** 2) / np.sum(b ** 2)))


@pytest.mark.parametrize("mode", ["fp8", "nvfp4"])
def test_small_read_copy_decode_matches_oracle(mode):
    shape = LayerShape(MAMBA2, batch=2, n_heads=4, n_groups=2, d_head=16, d_state=32, ring_len=4)
    pair = Pair(configs.Mamba2Workload(shape, seed=42, s0_std=0.1), read_mode=mode)
    for t in range(20):
        y, ref = pair.decode(t)
        assert_close(y, pair.last_read_expected, f"{mode} step {t}")
        pair.check_cursor(f"step {t}")
        pair.check_ring(f"step {t}")
        if pair.cursor_gpu()[:, 2].any():
            assert_close(y, ref, f"{mode} flush step {t} reads the FP32 checkpoint")
            pair.check_ckpt(f"step {t}")
    assert pair.cache.device_error() == 0


def _config4_windows(mode, steps, seqs):
    wl = configs.config4()
    pair = Pair(wl, seqs=seqs, read_mode=mode)
    _check_initial_copy(pair, mode, seqs)
    L = wl.shape.ring_len
    num = np.zeros(steps // L)
    den = np.zeros(steps // L)
    differing = 0
    for t in range(steps):
        y, ref = pair.decode(t)
        assert_close(y, pair.last_read_expected, f"{mode} step {t}")
        differing = max(differing, pair.copy_rows_differing)
        w = t // L
        num[w] += np.sum((y - ref) ** 2)
        den[w] += np.sum(ref ** 2)
    assert pair.cache.device_error() == 0
    return np.sqrt(num / den), differing, float(np.sqrt(num.sum() / den.sum()))


@pytest.mark.parametrize("mode,bound", [("fp8", 0.01), ("nvfp4", 0.06)])
def test_config4_error_per_window(mode, bound):
    """Config-4 shape (B=256, H=128, P=64, N=128, G=8, L=16), 512 steps = 32 windows,
    oracle on two sampled sequences."""
    per_window, differing, aggregate = _config4_windows(mode, 512, [0, 255])
    assert np.all(per_window[1:] <= bound), per_window
    assert aggregate <= bound
    # the copy never feeds the recurrence: no growth with the window index
    assert per_window[-8:].mean() <= 1.1 * per_window[1:9].mean(), per_window
    # rows whose two copies differ at all (most by one FP32 ulp of the row scale, when the
    # two FP32 checkpoints' row maxima differ in the last bit) are still compared element
    # by element above, against the oracle's output shifted by the copies' difference
    assert 0 <= differing <= 2 * 128 * 64


@pytest.mark.slow
@pytest.mark.parametrize("mode,bound", [("fp8", 0.01), ("nvfp4", 0.06)])
def test_config4_full_4096_steps(mode, bound):
    """All 4096 steps; the per-window rel-L2 is taken over four sequences spread
    across the batch (one sequence alone gives a noisy estimate of the batch's
    error: its FP8 windows scatter around 0.8% with single windows near 1%)."""
    per_window, differing, aggregate = _config4_windows(mode, 4096, [0, 85, 170, 255])
    assert np.all(per_window[1:] <= bound)
    assert aggregate <= bound
    assert per_window[-32:].mean() <= 1.1 * per_window[1:33].mean()


@pytest.mark.parametrize("mode", ["fp8", "nvfp4"])
def test_read_copy_d128_mixed_window_positions(mode):
    """d_state 128, heads-per-group a multiple of four: the non-flush units of a
    read-copy layer hold four heads, flush units one.  Verify + commit rounds with
    per-sequence accepted counts put the sequences at different window positions,
    so single decode launches mix both kinds of unit.  Flushing sequences must
    match the FP32 recurrence, the others the oracle's quantised-read output."""
    shape = LayerShape(MAMBA2, batch=5, n_heads=16, n_groups=2, d_head=64, d_state=128, ring_len=4, max_draft=2)
    pair = Pair(configs.Mamba2Workload(shape, seed=43, s0_std=0.1), read_mode=mode)
    _check_initial_copy(pair, mode, list(range(5)))
    for t in range(2):  # first window: the copy and the oracle's copy come from the same state
        y, ref = pair.decode(t)
        assert_close(y, pair.last_read_expected, f"{mode} step {t}")
    for s, acc in enumerate([[0, 1, 2, 1, 0], [2, 0, 1, 2, 1], [1, 2, 0, 0, 2]]):
        y, ref = pair.verify(s, 2)
        assert_close(y, ref, f"{mode} verify {s}")
        pair.check_ring(f"{mode} verify {s}")
        pair.commit(s, 2, accepted=acc)
        pair.check_cursor(f"{mode} commit {s}")
    mixed = 0
    for t in range(2, 26):
        y, ref = pair.decode(t)
        flushed = pair.cursor_gpu()[:, 2].astype(bool)
        mixed += int(0 < flushed.sum() < len(flushed))
        # flushing sequences read the FP32 checkpoint (expected = the exact output)
        assert_close(y, pair.last_read_expected, f"{mode} step {t}")
        assert_close(y[flushed], ref[flushed], f"{mode} step {t} flush rows")
        pair.check_cursor(f"{mode} step {t}")
        pair.check_ring(f"{mode} step {t}")
        if flushed.any():
            pair.check_ckpt(f"{mode} step {t}")
    assert mixed > 0  # some launches had flush and non-flush sequences together
    assert pair.cache.device_error() == 0


def _adversarial_state(shape, seed):
    """Rows whose elements sit at, or one FP32 ulp either side of, the midpoints between
    neighbouring e4m3 / e2m1 values once divided by the row's (or block's) scale: the
    cases where the quantiser's quotient decides the code."""
    rng = np.random.default_rng(seed)
    B, H, P, N = shape.batch, shape.n_heads, shape.d_head, shape.d_state
    e4m3 = np.unique(np.abs(codecs.e4m3_decode(np.arange(0, 0x7F))))
    mids = (e4m3[1:] + e4m3[:-1]) / 2
    e2m1 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    mids2 = (e2m1[1:] + e2m1[:-1]) / 2
    S = np.empty((B, H, P, N), dtype=np.float32)
    for idx in np.ndindex(B, H, P):
        scale = np.float32(np.exp(rng.uniform(-6, 2)))
        pick = mids if idx[2] % 2 == 0 else mids2
        v = rng.choice(pick, N) * scale
        v = np.nextafter(v.astype(np.float32), rng.choice([-np.inf, np.inf], N).astype(np.float32)) \
            if idx[2] % 3 == 0 else v.astype(np.float32)
        v = v * rng.choice([-1, 1], N)
        v[0] = np.float32(448.0) * scale            # row maximum fixes the FP8 scale
        S[idx] = v
    return S


@pytest.mark.parametrize("mode", ["fp8", "nvfp4"])
def test_quantiser_at_rounding_midpoints_bit_exact(mode):
    """The quantiser divides by a per-row / per-block scale with a reciprocal and one
    fused correction; at midpoints and one ulp beside them its codes must still be
    those of the oracle codec (IEEE division, round-to-nearest-even)."""
    shape = LayerShape(MAMBA2, batch=2, n_heads=4, n_groups=2, d_head=64, d_state=128, ring_len=4)
    from checkpoint_input_replay_gb300 import ReplayCache
    cache = ReplayCache.for_shape(shape, read_mode=mode)
    S = _adversarial_state(shape, 45)
    cache.ckpt.copy_(torch.from_numpy(S))
    cache.flush()
    v = cache.read_copy_views()
    if mode == "fp8":
        codes, sc = codecs.fp8_rows_quantize(S)
        np.testing.assert_array_equal(v["row_scale"].cpu().numpy(), sc)
        np.testing.assert_array_equal(v["codes"].cpu().numpy(), codes)
    else:
        packed, bs, sm = codecs.nvfp4_quantize(S)
        np.testing.assert_array_equal(v["matrix_scale"].cpu().numpy(), sm)
        np.testing.assert_array_equal(v["block_scale"].cpu().numpy(), bs)
        np.testing.assert_array_equal(v["codes"].cpu().numpy(), packed)
    assert cache.device_error() == 0
