"""GPU parity of tree-shaped speculative verification and commit by index list.

Draft tau continues draft parents[tau] (-1 = the committed records); every
draft's output must equal the oracle's recurrence along its own path, and
after a path commit the accepted drafts' records must sit, in path order,
right after the committed ones (Mamba-2 bit for bit; GDN g and k bit for bit,
u within 2e-4 * max(|ref|, 1e-3)), the cursor must have advanced by the path
length (bit-exact) and folds must match the oracle's checkpoint.  Covers the
tensor-core verify kernel (d_state 128) and the generic one (small d_state).
"""

import numpy as np
import pytest
import torch

from tests.harness import Pair, assert_close
from workloads import configs
from workloads.configs import GDN, MAMBA2, LayerShape

pytestmark = pytest.mark.gpu

TREES = [[-1, -1, 0, 1], [-1, 0, 0, 2], [-1, -1, -1, -1], [-1, 0, 1, 0], [-1, 0, 1, 2]]


def _tree_session(pair, rounds, trees, decode_between=True):
    t = 0
    for s in range(rounds):
        parents = trees[s % len(trees)]
        T = len(parents)
        y, ref = pair.verify_tree(s, T, parents)
        assert_close(y, ref, f"tree verify {s} {parents}")
        pair.check_ring(f"tree verify {s}")
        pair.commit_path(pair.tree_paths(s, T))
        pair.check_cursor(f"commit path {s}")
        pair.check_ring(f"commit path {s}")
        if pair.cursor_gpu()[:, 2].any():
            pair.check_ckpt(f"commit path {s}")
        if decode_between and s % 2 == 1:
            y, ref = pair.decode(500 + t)
            t += 1
            assert_close(y, ref, f"decode after round {s}")
            pair.check_cursor(f"decode after round {s}")
            pair.check_ring(f"decode after round {s}")
    assert pair.cache.device_error() == 0


@pytest.mark.parametrize("kind,P,N", [(MAMBA2, 64, 128), (GDN, 128, 128), (MAMBA2, 16, 32), (GDN, 32, 16),
                                      (GDN, 64, 128)])
def test_tree_verify_and_path_commit(kind, P, N):
    shape = LayerShape(kind, batch=4, n_heads=4, n_groups=2, d_head=P, d_state=N, ring_len=6, max_draft=4)
    wl = configs.workload(shape, seed=101 + P + N, s0_std=0.1 if kind == MAMBA2 else 0.05)
    _tree_session(Pair(wl), 12, TREES)


@pytest.mark.parametrize("kind", ["mamba2", "gdn"])
def test_tree_config3_shape_sampled(kind):
    """Config 3 shapes (B = 512, T = 4, L = 16), trees in turn, 12 rounds, two sampled sequences."""
    wl = configs.config3_mamba2() if kind == "mamba2" else configs.config3_gdn()
    _tree_session(Pair(wl, seqs=[7, 300]), 12, TREES, decode_between=False)


def test_path_that_is_not_a_path_is_rejected_on_the_device():
    shape = LayerShape(MAMBA2, batch=3, n_heads=2, n_groups=1, d_head=64, d_state=128, ring_len=6, max_draft=4)
    pair = Pair(configs.Mamba2Workload(shape, seed=109, s0_std=0.1))
    pair.decode(0)
    before = pair.cache.cursor.cpu().numpy().copy()
    pair.cache.verify_tree(4, [-1, -1, 0, 1], pair._dev_inputs(pair.wl.draft(0, 4)))
    plen = torch.tensor([2, 2, 1], dtype=torch.int32).cuda()
    path = torch.tensor([[0, 2, 0, 0], [0, 3, 0, 0], [3, 0, 0, 0]], dtype=torch.int32).cuda()  # 2nd, 3rd invalid
    pair.cache.commit_path(plen, path)
    cur = pair.cache.cursor.cpu().numpy()
    assert pair.cache.device_error() == 1
    assert cur[0, 1] == before[0, 1] + 2
    np.testing.assert_array_equal(cur[1:, :2], before[1:, :2])


def test_prefix_commit_of_a_branching_tree_is_refused():
    from checkpoint_input_replay_gb300 import ReplayError
    shape = LayerShape(MAMBA2, batch=2, n_heads=2, n_groups=1, d_head=16, d_state=16, ring_len=6, max_draft=4)
    pair = Pair(configs.Mamba2Workload(shape, seed=110, s0_std=0.1))
    pair.cache.verify_tree(3, [-1, -1, 0], pair._dev_inputs(pair.wl.draft(0, 3)))
    with pytest.raises(ReplayError):
        pair.cache.commit(torch.zeros(2, dtype=torch.int32).cuda())
    pair.cache.commit_path(torch.zeros(2, dtype=torch.int32).cuda(), torch.zeros(2, 4, dtype=torch.int32).cuda())
    assert pair.cache.device_error() == 0
