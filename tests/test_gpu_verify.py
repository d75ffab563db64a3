"""GPU parity of speculative verification (chunkwise form) and pointer-advance commit.

Drafts are appended after the committed records, outputs of every draft
position are compared with the oracle's token-by-token drafts, and commit
advances the cursor by the accepted prefix (folding when the ring fills).
Cursors and flush flags are compared bit-exactly after every call.
"""

import numpy as np
import pytest
import torch

from tests.harness import Pair, assert_close
from workloads import configs
from workloads.configs import GDN, MAMBA2, LayerShape

pytestmark = pytest.mark.gpu


def _spec_session(pair: Pair, rounds: int, T: int, decode_between=True, check_ckpt=True):
    t = 0
    for s in range(rounds):
        y, ref = pair.verify(s, T)
        assert_close(y, ref, f"verify {s}")
        pair.check_cursor(f"after verify {s}")
        pair.commit(s, T)
        pair.check_cursor(f"after commit {s}")
        if check_ckpt and pair.cursor_gpu()[:, 2].any():
            pair.check_ckpt(f"after commit {s}")
        if decode_between and s % 3 == 2:
            y, ref = pair.decode(1000 + t)
            t += 1
            assert_close(y, ref, f"decode after round {s}")
            pair.check_cursor(f"decode after round {s}")
    assert pair.cache.device_error() == 0


@pytest.mark.parametrize("T", [1, 2, 4])
def test_mamba2_small_spec_session(T):
    shape = LayerShape(MAMBA2, batch=3, n_heads=4, n_groups=2, d_head=16, d_state=32, ring_len=5, max_draft=4)
    pair = Pair(configs.Mamba2Workload(shape, seed=21, s0_std=0.1))
    _spec_session(pair, 12, T)


@pytest.mark.parametrize("T", [1, 3, 4])
def test_gdn_small_spec_session(T):
    shape = LayerShape(GDN, batch=3, n_heads=4, n_groups=2, d_head=32, d_state=16, ring_len=5, max_draft=4)
    pair = Pair(configs.GdnWorkload(shape, seed=22, s0_std=0.05))
    _spec_session(pair, 12, T)


def test_all_accepted_and_none_accepted():
    shape = LayerShape(MAMBA2, batch=2, n_heads=2, n_groups=1, d_head=16, d_state=16, ring_len=4, max_draft=3)
    pair = Pair(configs.Mamba2Workload(shape, seed=23, s0_std=0.1))
    for s, acc in enumerate([[3, 0], [3, 0], [0, 0], [1, 3], [3, 3]]):
        y, ref = pair.verify(s, 3)
        assert_close(y, ref, f"verify {s}")
        pair.commit(s, 3, accepted=acc)
        pair.check_cursor(f"commit {s}")
        pair.check_ckpt(f"commit {s}")


def test_drafts_land_after_committed_records():
    """Draft records occupy slots (head + count + tau) mod C; the cursor does not move at verify."""
    shape = LayerShape(MAMBA2, batch=2, n_heads=2, n_groups=1, d_head=16, d_state=16, ring_len=4, max_draft=2)
    wl = configs.Mamba2Workload(shape, seed=24, s0_std=0.1)
    pair = Pair(wl)
    pair.decode(0)
    before = pair.cache.cursor.cpu().numpy().copy()
    pair.verify(0, 2)
    after = pair.cache.cursor.cpu().numpy()
    np.testing.assert_array_equal(before[:, :2], after[:, :2])
    ring = pair.cache.ring_views()
    drafts = wl.draft(0, 2)
    for b in range(2):
        for tau in range(2):
            slot = (after[b, 0] + after[b, 1] + tau) % pair.cache.C
            got = ring["x"][b, :, slot].view(torch.int16).cpu().numpy().view(np.uint16)
            np.testing.assert_array_equal(got, drafts["x"][b, tau])


@pytest.mark.parametrize("kind", ["mamba2", "gdn"])
def test_config3_full_batch_sampled(kind):
    """Config 3: B=512, T=4, L=16, 64 verify steps with accepted counts U{0..4}."""
    wl = configs.config3_mamba2() if kind == "mamba2" else configs.config3_gdn()
    pair = Pair(wl, seqs=[1, 511])
    for s in range(64):
        y, ref = pair.verify(s, 4)
        assert_close(y, ref, f"verify {s}")
        acc = pair.commit(s, 4)
        pair.check_cursor(f"commit {s}")
        if pair.cursor_gpu()[:, 2].any():
            pair.check_ckpt(f"commit {s}")
    assert pair.cache.device_error() == 0


# d_state 128 with d_head 64 or 128: the tcgen05 verify kernel (128-row units:
# two heads of d_head 64 or one of d_head 128), in small shapes that the oracle
# checks element by element.
@pytest.mark.parametrize("kind,P,H,G,T", [
    ("mamba2", 64, 4, 2, 1), ("mamba2", 64, 4, 2, 4), ("mamba2", 128, 4, 1, 3),
    ("gdn", 128, 4, 2, 1), ("gdn", 128, 4, 2, 4), ("gdn", 64, 4, 2, 2),
])
def test_tensor_core_verify_small(kind, P, H, G, T):
    k = MAMBA2 if kind == "mamba2" else GDN
    shape = LayerShape(k, batch=3, n_heads=H, n_groups=G, d_head=P, d_state=128, ring_len=5, max_draft=4)
    wl = configs.workload(shape, seed=31 + P + T, s0_std=0.1 if k == MAMBA2 else 0.05)
    _spec_session(Pair(wl), 10, T)


@pytest.mark.parametrize("kind", ["mamba2", "gdn"])
def test_tensor_core_verify_many_units_per_cta(kind):
    """Several units per CTA; groups split across CTA boundaries; the ring wraps."""
    if kind == "mamba2":
        shape = LayerShape(MAMBA2, batch=24, n_heads=32, n_groups=2, d_head=64, d_state=128, ring_len=16,
                           max_draft=4)
        wl = configs.Mamba2Workload(shape, seed=41, s0_std=0.1)
        seqs = [0, 11, 23]
    else:
        shape = LayerShape(GDN, batch=40, n_heads=32, n_groups=16, d_head=128, d_state=128, ring_len=16,
                           max_draft=4)
        wl = configs.GdnWorkload(shape, seed=42, s0_std=0.05)
        seqs = [0, 19, 39]
    _spec_session(Pair(wl, seqs=seqs), 20, 4)


@pytest.mark.slow
def test_tensor_core_verify_grid_doubling_many_sequences():
    """10000 single-head sequences of d_head 128 through the tensor-core verify and the
    balanced commit: more sequences per CTA than the per-CTA cursor table holds, so the
    launchers enlarge the grid.  Sampled sequences against the oracle."""
    shape = LayerShape(MAMBA2, batch=10000, n_heads=1, n_groups=1, d_head=128, d_state=128, ring_len=4,
                       max_draft=2)
    pair = Pair(configs.Mamba2Workload(shape, seed=29, s0_std=0.1), seqs=[0, 1, 31, 32, 5000, 9999])
    for t in range(2):
        y, ref = pair.decode(t)
        assert_close(y, ref, f"decode {t}")
    for s in range(3):
        y, ref = pair.verify(s, 2)
        assert_close(y, ref, f"verify {s}")
        pair.commit(s, 2)
        pair.check_cursor(f"commit {s}")
    pair.check_ckpt("checkpoint")
    assert pair.cache.device_error() == 0
