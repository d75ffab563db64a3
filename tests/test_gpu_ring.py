"""GPU ring contents at d_state 128 (the workloads' kernels), slot by slot.

Records appended by the decode kernel's builder warps and by the verify
kernels' draft appends must sit at slot (head + j) mod C of every sequence
("ReplaySSM caches SSM inputs instead of state" (richland.au), "What shipped":
records past the pointer are ignored and overwritten, exactly like a KV cache).
Mamba-2 records (x, dt, B as bf16, log a = dt * A in float32) are compared bit
for bit with the inputs; GDN records compare g and k bit for bit and the delta
u = b (v - a S_{t-1} k) with the oracle's step-by-step value within
2e-4 * max(|ref|, 1e-3).  Every live slot is checked after every call.
"""

import pytest

from tests.harness import Pair, assert_close
from workloads import configs
from workloads.configs import GDN, MAMBA2, LayerShape

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kind,P", [(MAMBA2, 64), (MAMBA2, 128), (GDN, 128), (GDN, 64)])
def test_d128_ring_after_every_call(kind, P):
    shape = LayerShape(kind, batch=3, n_heads=8, n_groups=2, d_head=P, d_state=128, ring_len=5, max_draft=3)
    wl = configs.workload(shape, seed=71 + P, s0_std=0.1 if kind == MAMBA2 else 0.05)
    pair = Pair(wl)
    t = 0
    for s, acc in enumerate([[3, 0, 1], [1, 3, 2], [0, 0, 3], [2, 1, 0], [3, 3, 3]]):
        for _ in range(3):
            y, ref = pair.decode(t)
            assert_close(y, ref, f"decode {t}")
            pair.check_cursor(f"decode {t}")
            pair.check_ring(f"decode {t}")
            t += 1
        y, ref = pair.verify(s, 3)
        assert_close(y, ref, f"verify {s}")
        pair.check_ring(f"verify {s}")
        pair.commit(s, 3, accepted=acc)
        pair.check_cursor(f"commit {s}")
        pair.check_ring(f"commit {s}")
    assert pair.cache.device_error() == 0


@pytest.mark.parametrize("kind", [MAMBA2, GDN])
def test_config_shape_ring_sampled_sequences(kind):
    """Config 1 / config 2 shapes (B = 256, L = 16), 40 steps: ring of three sampled
    sequences after every step (the launch the bench times)."""
    wl = configs.config1() if kind == MAMBA2 else configs.config2()
    pair = Pair(wl, seqs=[0, 131, 255])
    for t in range(40):
        y, ref = pair.decode(t)
        assert_close(y, ref, f"step {t}")
        pair.check_cursor(f"step {t}")
        pair.check_ring(f"step {t}")
    assert pair.cache.device_error() == 0


@pytest.mark.parametrize("kind", ["mamba2", "gdn"])
def test_config3_ring_sampled_sequences(kind):
    """Config 3 (B = 512, T = 4, L = 16): draft records after every verify and committed
    records after every commit, for two sampled sequences, over 24 rounds."""
    wl = configs.config3_mamba2() if kind == "mamba2" else configs.config3_gdn()
    pair = Pair(wl, seqs=[5, 400])
    for s in range(24):
        y, ref = pair.verify(s, 4)
        assert_close(y, ref, f"verify {s}")
        pair.check_ring(f"verify {s}")
        pair.commit(s, 4)
        pair.check_cursor(f"commit {s}")
        pair.check_ring(f"commit {s}")
    assert pair.cache.device_error() == 0


@pytest.mark.parametrize("kind,P,L", [(MAMBA2, 64, 32), (GDN, 128, 32), (MAMBA2, 64, 8), (GDN, 128, 4),
                                      (MAMBA2, 64, 1), (GDN, 128, 1)])
def test_d128_window_lengths_of_the_sweep(kind, P, L):
    """The window lengths the bench sweeps (1, 4, 8, 32; 16 is the workloads' own; at 1
    every step folds): two windows and a half, every output, cursor and ring slot, the
    checkpoint at each flush."""
    shape = LayerShape(kind, batch=3, n_heads=8, n_groups=2, d_head=P, d_state=128, ring_len=L)
    wl = configs.workload(shape, seed=77 + L, s0_std=0.1 if kind == MAMBA2 else 0.05)
    pair = Pair(wl)
    flushes = 0
    for t in range(2 * L + L // 2):
        y, ref = pair.decode(t)
        assert_close(y, ref, f"step {t}")
        pair.check_cursor(f"step {t}")
        pair.check_ring(f"step {t}")
        if pair.cursor_gpu()[:, 2].any():
            flushes += 1
            pair.check_ckpt(f"step {t}")
    assert flushes == 2
    assert pair.cache.device_error() == 0
