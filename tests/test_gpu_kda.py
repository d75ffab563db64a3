"""GPU parity of the per-channel-gate layer (the Gated DeltaNet rule with a decay per
key channel) against the oracle's conventional recurrence.

Outputs, checkpoints after every fold and the ring's delta records within
2e-4 * max(|ref|, 1e-3); the ring's per-channel log decays and keys bit for
bit; cursors and flush flags bit-exactly, after every call.
"""

import numpy as np
import pytest
import torch

from tests.harness import Pair, assert_close
from workloads import configs
from workloads.configs import KDA, LayerShape

pytestmark = pytest.mark.gpu


def _run(pair, steps):
    flushes = 0
    for t in range(steps):
        y, ref = pair.decode(t)
        assert_close(y, ref, f"step {t} output")
        pair.check_cursor(f"step {t}")
        pair.check_ring(f"step {t}")
        if pair.cursor_gpu()[:, 2].any():
            flushes += 1
            pair.check_ckpt(f"step {t}")
    assert pair.cache.device_error() == 0
    return flushes


@pytest.mark.parametrize("P,N,L", [(16, 16, 4), (32, 64, 5), (64, 128, 4), (128, 128, 6), (128, 32, 1)])
def test_kda_decode_windows(P, N, L):
    shape = LayerShape(KDA, batch=3, n_heads=4, n_groups=2, d_head=P, d_state=N, ring_len=L)
    wl = configs.KdaWorkload(shape, seed=120 + P + N, s0_std=0.05)
    assert _run(Pair(wl), 3 * L + 2) == (3 * L + 2) // L


def test_kda_long_window_32():
    shape = LayerShape(KDA, batch=2, n_heads=4, n_groups=4, d_head=128, d_state=128, ring_len=32)
    assert _run(Pair(configs.KdaWorkload(shape, seed=131, s0_std=0.05)), 70) == 2


def test_kda_masked_flush_and_export():
    shape = LayerShape(KDA, batch=4, n_heads=2, n_groups=1, d_head=32, d_state=32, ring_len=8)
    pair = Pair(configs.KdaWorkload(shape, seed=132, s0_std=0.05))
    for t in range(5):
        pair.decode(t)
    mask = np.array([1, 0, 0, 1], dtype=np.uint8)
    pair.cache.flush(torch.from_numpy(mask).cuda())
    pair.oracle.flush(mask)
    pair.check_cursor("after masked flush")
    pair.check_ckpt("after masked flush")
    assert _run(pair, 11) >= 1
    pair.cache.flush()
    pair.oracle.flush()
    pair.check_ckpt("after full flush")


def test_kda_config_shape_sampled():
    """B = 256, 32 value heads over 16 key heads, d = 128, L = 16: 40 steps, two sampled sequences."""
    pair = Pair(configs.config_kda(), seqs=[0, 199])
    assert _run(pair, 40) == 2
