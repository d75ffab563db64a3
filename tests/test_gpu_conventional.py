"""GPU parity of the conventional comparison path against the oracle.

The oracle *is* the conventional recurrence, so the read-modify-write decode
step must reproduce its outputs and its state after every token, and the
snapshot-per-draft verify must reproduce the outputs of every draft and hold,
in slot (cur + 1 + tau) mod (T_max + 1), the state after draft tau; a commit
of n drafts must leave the state after the accepted prefix current.  All
within 2e-4 * max(|ref|, 1e-3); slot indices bit-exactly.
"""

import numpy as np
import pytest
import torch

from checkpoint_input_replay_gb300 import ConventionalLayer, SnapshotLayer
from oracle.layer import OracleLayer, _wide
from oracle.recurrence import gdn_step, mamba2_step
from tests.harness import assert_close, to_dev
from workloads import configs
from workloads.configs import GDN, MAMBA2, LayerShape

pytestmark = pytest.mark.gpu


def _dev(wl, inp, A):
    d = to_dev(inp)
    if A is not None:
        d["A"] = A
    return d


def _step(kind, S, tok, A):
    if kind == MAMBA2:
        return mamba2_step(S, tok["x"], tok["dt"], A, tok["B"], tok["C"])
    return gdn_step(S, tok["q"], tok["k"], tok["v"], tok["g"], tok["beta"])


def _decode_session(wl, steps, seqs):
    s = wl.shape
    layer = ConventionalLayer.for_shape(s)
    S0 = wl.S0()
    layer.state.copy_(torch.from_numpy(S0))
    A = wl.A() if s.kind == MAMBA2 else None
    A_dev = torch.from_numpy(A).cuda() if A is not None else None
    S = S0[seqs].astype(np.float64)
    idx = torch.tensor(seqs).cuda()
    for t in range(steps):
        inp = wl.step(t)
        y = layer.decode_step(_dev(wl, inp, A_dev))
        S, ref = _step(s.kind, S, _wide({k: v[seqs] for k, v in inp.items()}), A)
        assert_close(y.index_select(0, idx).cpu().numpy(), ref, f"step {t} output")
        assert_close(layer.state.index_select(0, idx).cpu().numpy(), S, f"step {t} state")


@pytest.mark.parametrize("kind,P,N", [(MAMBA2, 16, 16), (MAMBA2, 32, 64), (MAMBA2, 64, 128), (MAMBA2, 128, 128),
                                      (GDN, 16, 16), (GDN, 64, 32), (GDN, 128, 128), (GDN, 64, 128)])
def test_conventional_decode_small(kind, P, N):
    shape = LayerShape(kind, batch=3, n_heads=4, n_groups=2, d_head=P, d_state=N, ring_len=1)
    wl = configs.workload(shape, seed=81 + P + N, s0_std=0.1 if kind == MAMBA2 else 0.05)
    _decode_session(wl, 12, [0, 1, 2])


@pytest.mark.parametrize("kind", [MAMBA2, GDN])
def test_conventional_decode_config_shapes_sampled(kind):
    """Config 1 / config 2 shapes at B = 256 (the launch the bench times), 20 tokens."""
    wl = configs.config1() if kind == MAMBA2 else configs.config2()
    _decode_session(wl, 20, [0, 200])


def _snapshot_session(wl, rounds, T, seqs):
    s = wl.shape
    layer = SnapshotLayer.for_shape(s)
    S0 = wl.S0()
    layer.pool[:, 0].copy_(torch.from_numpy(S0))
    A = wl.A() if s.kind == MAMBA2 else None
    A_dev = torch.from_numpy(A).cuda() if A is not None else None
    oracle = OracleLayer(s, seqs, S0[seqs], A=A)
    idx = torch.tensor(seqs).cuda()
    n_slots = s.max_draft + 1
    for r in range(rounds):
        inp = wl.draft(r, T)
        cur = layer.slots.cpu().numpy()[seqs]
        S_before = oracle.S.copy()
        y = layer.verify(T, _dev(wl, inp, A_dev))
        ref = oracle.verify({k: v[seqs] for k, v in inp.items()}, T)
        assert_close(y.index_select(0, idx).cpu().numpy(), ref, f"round {r} outputs")
        # the snapshot after every draft, in its slot
        pool = layer.pool.index_select(0, idx).cpu().numpy()
        Sd = S_before
        tok = _wide({k: v[seqs] for k, v in inp.items()})
        for tau in range(T):
            Sd, _ = _step(s.kind, Sd, {k: v[:, tau] for k, v in tok.items()}, A)
            for i in range(len(seqs)):
                assert_close(pool[i, (cur[i] + 1 + tau) % n_slots], Sd[i], f"round {r} snapshot {tau} seq {i}")
        acc = wl.accepted(r, T)
        layer.commit(torch.from_numpy(acc).cuda())
        oracle.commit(acc[seqs])
        np.testing.assert_array_equal(layer.slots.cpu().numpy()[seqs], (cur + acc[seqs]) % n_slots)
        cur_state = layer.pool[idx, layer.slots.index_select(0, idx).long()]
        assert_close(cur_state.cpu().numpy(), oracle.S, f"round {r} committed")
    assert layer.device_error() == 0


@pytest.mark.parametrize("kind,P,N,T", [(MAMBA2, 16, 16, 2), (MAMBA2, 64, 128, 4), (GDN, 32, 16, 3),
                                        (GDN, 128, 128, 4), (GDN, 64, 128, 1)])
def test_snapshot_verify_small(kind, P, N, T):
    shape = LayerShape(kind, batch=3, n_heads=4, n_groups=2, d_head=P, d_state=N, ring_len=1, max_draft=4)
    wl = configs.workload(shape, seed=91 + P + T, s0_std=0.1 if kind == MAMBA2 else 0.05)
    _snapshot_session(wl, 6, T, [0, 1, 2])


@pytest.mark.parametrize("kind", ["mamba2", "gdn"])
def test_snapshot_verify_config3_sampled(kind):
    """Config 3 shapes (B = 512, T = 4), 6 rounds, two sampled sequences."""
    wl = configs.config3_mamba2() if kind == "mamba2" else configs.config3_gdn()
    _snapshot_session(wl, 6, 4, [3, 509])


def test_snapshot_commit_rejects_out_of_range_counts():
    shape = LayerShape(MAMBA2, batch=4, n_heads=2, n_groups=1, d_head=16, d_state=16, ring_len=1, max_draft=2)
    wl = configs.Mamba2Workload(shape, seed=99, s0_std=0.1)
    layer = SnapshotLayer.for_shape(shape)
    layer.verify(2, _dev(wl, wl.draft(0, 2), torch.from_numpy(wl.A()).cuda()))
    layer.commit(torch.tensor([1, 3, 0, -1], dtype=torch.int32).cuda())
    assert layer.device_error() == 1                       # accepted count out of range
    np.testing.assert_array_equal(layer.slots.cpu().numpy(), [1, 0, 0, 0])  # bad sequences unchanged
