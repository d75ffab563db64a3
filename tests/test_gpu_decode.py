"""GPU parity of the standard decode step (non-flush and flush bodies) against the oracle.

Every case runs through the C ABI (ReplayCache -> libreplayssm.so).  Outputs
and checkpoints are compared elementwise within 2e-4 * max(|ref|, 1e-3);
cursors, flush flags and the Mamba-2 ring contents bit-exactly.
"""

import dataclasses

import numpy as np
import pytest
import torch

from tests.harness import Pair, assert_close
from workloads import configs
from workloads.configs import GDN, MAMBA2, LayerShape

pytestmark = pytest.mark.gpu


def _run_decode(pair: Pair, steps: int, check_every_ckpt=True):
    flushes = 0
    for t in range(steps):
        y, ref = pair.decode(t)
        assert_close(y, ref, f"step {t} output")
        pair.check_cursor(f"step {t} cursor")
        if pair.cursor_gpu()[:, 2].any():
            flushes += 1
            if check_every_ckpt:
                pair.check_ckpt(f"step {t} checkpoint")
    assert pair.cache.device_error() == 0
    return flushes


def test_config0_tiny_mamba2_64_steps_16_flushes():
    pair = Pair(configs.config0())
    assert _run_decode(pair, 64) == 16


def test_config0_ring_contents_bit_exact():
    """Mamba-2 ring slots hold bf16 copies of the buffered inputs, at (head + j) mod C."""
    wl = configs.config0()
    pair = Pair(wl)
    hist = []
    for t in range(11):
        pair.decode(t)
        hist.append(wl.step(t))
        ring = pair.cache.ring_views()
        cur = pair.cache.cursor.cpu().numpy()
        for b in range(wl.shape.batch):
            head, count = cur[b, 0], cur[b, 1]
            for j in range(count):
                src = hist[len(hist) - count + j]
                slot = (head + j) % pair.cache.C
                got = ring["x"][b, :, slot].view(torch.int16).cpu().numpy().view(np.uint16)
                np.testing.assert_array_equal(got, src["x"][b])
                got_b = ring["B"][b, :, slot].view(torch.int16).cpu().numpy().view(np.uint16)
                np.testing.assert_array_equal(got_b, src["B"][b])


def test_mamba2_multi_tile_ragged():
    """Several heads per group, odd window, steps not a multiple of L, larger tile."""
    shape = LayerShape(MAMBA2, batch=3, n_heads=6, n_groups=3, d_head=32, d_state=64, ring_len=5)
    wl = configs.Mamba2Workload(shape, seed=11, s0_std=0.1)
    pair = Pair(wl)
    assert _run_decode(pair, 23) == 4


def test_mamba2_window_of_one_flushes_every_step():
    shape = LayerShape(MAMBA2, batch=2, n_heads=2, n_groups=1, d_head=16, d_state=16, ring_len=1)
    pair = Pair(configs.Mamba2Workload(shape, seed=12, s0_std=0.1))
    assert _run_decode(pair, 5) == 5


def test_gdn_small_64_steps():
    shape = LayerShape(GDN, batch=2, n_heads=4, n_groups=2, d_head=16, d_state=16, ring_len=4)
    pair = Pair(configs.GdnWorkload(shape, seed=13, s0_std=0.05))
    assert _run_decode(pair, 64) == 16


def test_gdn_multi_tile_ragged():
    shape = LayerShape(GDN, batch=3, n_heads=4, n_groups=2, d_head=64, d_state=128, ring_len=6)
    pair = Pair(configs.GdnWorkload(shape, seed=14, s0_std=0.05))
    assert _run_decode(pair, 20) == 3


def test_gdn_d128_long_window_split_heads():
    """d_head 128 heads computed as two 64-row parts; three heads a group (one half-warp of
    the two-head table build idle); window 20, so groups of up to 20 records take the
    full-warp table build; 5 x 6 x 2 parts spread over CTAs that start mid-head."""
    shape = LayerShape(GDN, batch=5, n_heads=6, n_groups=2, d_head=128, d_state=128, ring_len=20)
    pair = Pair(configs.GdnWorkload(shape, seed=16, s0_std=0.05))
    assert _run_decode(pair, 45) == 2


@pytest.mark.parametrize("kind,P", [(MAMBA2, 64), (MAMBA2, 128), (GDN, 64), (GDN, 128)])
def test_d128_one_head_per_group(kind, P):
    """d_state 128 with as many groups as heads: one unit per group (two for a GDN
    head of d_head 128), so the decode kernel runs with its fewest stages (units per
    group + 1) and a group buffer restaged every one or two units."""
    shape = LayerShape(kind, batch=3, n_heads=5, n_groups=5, d_head=P, d_state=128, ring_len=4)
    wl = configs.workload(shape, seed=17, s0_std=0.1 if kind == MAMBA2 else 0.05)
    assert _run_decode(Pair(wl), 13) == 3


@pytest.mark.parametrize("kind,P", [(MAMBA2, 64), (GDN, 128)])
def test_d128_single_sequence_single_head(kind, P):
    """The smallest grid: one sequence, one head (one or two units in all)."""
    shape = LayerShape(kind, batch=1, n_heads=1, n_groups=1, d_head=P, d_state=128, ring_len=2)
    wl = configs.workload(shape, seed=18, s0_std=0.1 if kind == MAMBA2 else 0.05)
    assert _run_decode(Pair(wl), 7) == 3


@pytest.mark.slow
def test_d128_grid_doubling_many_sequences():
    """10000 single-head sequences: a CTA's share would cover more sequences than its
    per-CTA cursor table holds, so the launcher doubles the grid.  Sampled sequences
    at the edges of the CTA ranges are checked against the oracle; every cursor is
    checked against the plain ring rule."""
    shape = LayerShape(MAMBA2, batch=10000, n_heads=1, n_groups=1, d_head=64, d_state=128, ring_len=3)
    pair = Pair(configs.Mamba2Workload(shape, seed=19, s0_std=0.1), seqs=[0, 1, 32, 33, 5000, 9998, 9999])
    assert _run_decode(pair, 7) == 2
    cur = pair.cache.cursor.cpu().numpy()[:10000]
    assert (cur[:, 0] == 0).all() and (cur[:, 1] == 1).all()  # 7 steps at L = 3: flushed twice (head 6 mod 3)


@pytest.mark.parametrize("N,P", [(32, 32), (128, 128), (16, 128), (128, 16)])
def test_shapes_sweep(N, P):
    for kind in (MAMBA2, GDN):
        shape = LayerShape(kind, batch=2, n_heads=4, n_groups=2, d_head=P, d_state=N, ring_len=3)
        wl = configs.workload(shape, seed=15, s0_std=0.1)
        assert _run_decode(Pair(wl), 7) == 2


def test_config1_full_batch_sampled_sequences():
    """Config 1 (B=256, H=128, P=64, N=128, G=8, L=16), 160 steps, the launch the bench
    times; the oracle follows three sequences, cursors checked for all 256."""
    wl = configs.config1()
    pair = Pair(wl, seqs=[0, 137, 255])
    for t in range(160):
        y, ref = pair.decode(t)
        assert_close(y, ref, f"step {t} output")
        cur = pair.cache.cursor.cpu().numpy()
        assert (cur[:, 1] == (t + 1) % 16).all() and (cur[:, 0] == ((t + 1) // 16 * 16) % 16).all()
        if (t + 1) % 16 == 0:
            assert cur[:, 2].all()
            pair.check_ckpt(f"step {t} checkpoint")
    assert pair.cache.device_error() == 0


def test_config2_full_batch_sampled_sequences():
    """Config 2 (GDN, B=256, Hv=32, Hk=16, d=128, L=16), 160 steps."""
    wl = configs.config2()
    pair = Pair(wl, seqs=[3, 200])
    for t in range(160):
        y, ref = pair.decode(t)
        assert_close(y, ref, f"step {t} output")
        pair.check_cursor(f"step {t}")
        if (t + 1) % 16 == 0:
            pair.check_ckpt(f"step {t} checkpoint")
    assert pair.cache.device_error() == 0


def test_flush_with_mask_and_export():
    """rs_flush folds only the masked sequences; afterwards their checkpoint is the full state."""
    shape = LayerShape(MAMBA2, batch=4, n_heads=4, n_groups=2, d_head=16, d_state=32, ring_len=8)
    wl = configs.Mamba2Workload(shape, seed=16, s0_std=0.1)
    pair = Pair(wl)
    for t in range(5):
        pair.decode(t)
    mask = np.array([1, 0, 1, 0], dtype=np.uint8)
    pair.cache.flush(torch.from_numpy(mask).cuda())
    pair.oracle.flush(mask)
    pair.check_cursor("after masked flush")
    pair.check_ckpt("after masked flush")
    for t in range(5, 12):
        y, ref = pair.decode(t)
        assert_close(y, ref, f"step {t}")
        pair.check_cursor(f"step {t}")
    pair.cache.flush()
    pair.oracle.flush()
    pair.check_ckpt("after full flush")
    assert pair.cache.device_error() == 0


def _run_layer(shape, seed, steps, rounds):
    """Decode steps, verify + commit rounds, decode steps again, through the C ABI;
    returns every output and the caches' final contents."""
    from checkpoint_input_replay_gb300 import ReplayCache
    from tests.harness import to_dev
    wl = configs.workload(shape, seed=seed, s0_std=0.1 if shape.kind == MAMBA2 else 0.05)
    cache = ReplayCache.for_shape(shape)
    cache.ckpt.copy_(torch.from_numpy(wl.S0()))
    A = torch.from_numpy(wl.A()).cuda() if shape.kind == MAMBA2 else None

    def dev(inp):
        d = to_dev(inp)
        if A is not None:
            d["A"] = A
        return d

    ys = [cache.decode_step(dev(wl.step(t))).clone() for t in range(steps)]
    for s in range(rounds):
        ys.append(cache.verify(2, dev(wl.draft(s, 2))).clone())
        cache.commit(torch.from_numpy(wl.accepted(s, 2)).cuda())
    ys += [cache.decode_step(dev(wl.step(steps + t))).clone() for t in range(steps)]
    torch.cuda.synchronize()
    out = [cache.ckpt.cpu().numpy(), cache.cursor.cpu().numpy(),
           {k: (v.view(torch.int16) if v.dtype == torch.bfloat16 else v).cpu().numpy()
            for k, v in cache.ring_views().items()}]
    assert cache.device_error() == 0
    cache.close()
    return [y.cpu().numpy() for y in ys], out


@pytest.mark.parametrize("kind,P", [(MAMBA2, 64), (GDN, 128)])
def test_cta_order_permuted_gives_identical_results(kind, P, monkeypatch):
    """The debug permutation of unit ranges over the CTAs of the persistent decode and
    commit launches (RS_DEBUG_CTA_PERMUTE) changes which CTA runs, arrives and writes
    cursors when: outputs, checkpoints, cursors and ring must stay bit for bit."""
    shape = LayerShape(kind, batch=37, n_heads=8, n_groups=2, d_head=P, d_state=128, ring_len=3, max_draft=2)
    monkeypatch.delenv("RS_DEBUG_CTA_PERMUTE", raising=False)
    ys0, st0 = _run_layer(shape, 41, 7, 3)
    monkeypatch.setenv("RS_DEBUG_CTA_PERMUTE", "5")
    ys1, st1 = _run_layer(shape, 41, 7, 3)
    for a, b in zip(ys0, ys1):
        np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(st0[0], st1[0])
    np.testing.assert_array_equal(st0[1], st1[1])
    for k in st0[2]:
        np.testing.assert_array_equal(st0[2][k], st1[2][k])
