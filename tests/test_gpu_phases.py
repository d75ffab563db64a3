"""Mixed window positions in one decode launch, and whole windows replayed as CUDA graphs.

* Sequences at different window positions (staggered by masked flushes) make
  every decode launch mix flush and non-flush sequences; the launch splits the
  work by weight (a folding unit costs about 2.25 non-flush units), so CTA
  ranges no longer follow the unit count.  Outputs, checkpoints, cursors and
  ring slots are checked against the oracle after every step, also with the
  debug permutation of the CTA order.
* A window of decode steps captured once in a CUDA graph and replayed must give
  bit for bit what the same calls give when launched one by one: the cursor is
  device-resident, so a replay advances it like a live call.
"""

import numpy as np
import pytest
import torch

from checkpoint_input_replay_gb300 import ReplayCache
from tests.harness import Pair, assert_close, to_dev
from workloads import configs
from workloads.configs import GDN, MAMBA2, LayerShape

pytestmark = pytest.mark.gpu


def _stagger(pair, L):
    """After step k, fold the sequences with b % L == k: every window position occurs."""
    B = pair.shape.batch
    for k in range(L):
        y, ref = pair.decode(k)
        assert_close(y, ref, f"stagger step {k}")
        mask = np.array([1 if b % L == k else 0 for b in range(B)], dtype=np.uint8)
        pair.cache.flush(torch.from_numpy(mask).cuda())
        pair.oracle.flush(mask[pair.seqs])
        pair.check_cursor(f"stagger flush {k}")


@pytest.mark.parametrize("kind,P,permute,even", [(MAMBA2, 64, None, False), (GDN, 128, None, False),
                                                 (MAMBA2, 64, "7", False), (GDN, 128, None, True)])
def test_mixed_window_positions_every_step(kind, P, permute, even, monkeypatch):
    """Also with the CTA order permuted, and with the even split (the debug comparison)."""
    if permute is None:
        monkeypatch.delenv("RS_DEBUG_CTA_PERMUTE", raising=False)
    else:
        monkeypatch.setenv("RS_DEBUG_CTA_PERMUTE", permute)
    if even:
        monkeypatch.setenv("RS_DEBUG_UNIFORM_SPLIT", "1")
    else:
        monkeypatch.delenv("RS_DEBUG_UNIFORM_SPLIT", raising=False)
    L = 6
    shape = LayerShape(kind, batch=37, n_heads=8, n_groups=2, d_head=P, d_state=128, ring_len=L)
    wl = configs.workload(shape, seed=141 + P, s0_std=0.1 if kind == MAMBA2 else 0.05)
    pair = Pair(wl)
    _stagger(pair, L)
    for t in range(L, 4 * L):
        y, ref = pair.decode(t)
        assert_close(y, ref, f"step {t}")
        pair.check_cursor(f"step {t}")
        flags = pair.cursor_gpu()[:, 2]
        assert 0 < flags.sum() < len(flags)          # a mixed launch
        pair.check_ring(f"step {t}")
        pair.check_ckpt(f"step {t}")
    assert pair.cache.device_error() == 0


def test_config1_shape_mixed_positions_sampled():
    """B = 256 at 16 staggered window positions: about one sequence in 16 folds per step."""
    wl = configs.config1()
    pair = Pair(wl, seqs=[0, 5, 130, 255])
    _stagger(pair, 16)
    for t in range(16, 40):
        y, ref = pair.decode(t)
        assert_close(y, ref, f"step {t}")
        pair.check_cursor(f"step {t}")
        if pair.cursor_gpu()[:, 2].any():
            pair.check_ckpt(f"step {t}")
    cur = pair.cache.cursor.cpu().numpy()[:256]
    assert len(set(cur[:, 1].tolist())) == 16      # all 16 positions present
    assert pair.cache.device_error() == 0


def _graph_vs_eager(shape, seed, windows):
    wl = configs.workload(shape, seed=seed, s0_std=0.1 if shape.kind == MAMBA2 else 0.05)
    L = shape.ring_len
    A = torch.from_numpy(wl.A()).cuda() if shape.kind == MAMBA2 else None

    def dev(t):
        d = to_dev(wl.step(t))
        if A is not None:
            d["A"] = A
        return d

    inputs = [dev(t) for t in range(L)]
    outs = {}
    for mode in ("eager", "graph"):
        cache = ReplayCache.for_shape(shape)
        cache.ckpt.copy_(torch.from_numpy(wl.S0()))
        ys = [torch.empty(shape.batch, shape.n_heads, shape.d_head, device="cuda") for _ in range(L)]
        # one eager step first (also warms the library up before any capture), then
        # `windows` windows of L steps: eager calls, or replays of one captured window
        cache.decode_step(inputs[0], ys[0])
        torch.cuda.synchronize()
        if mode == "eager":
            for _ in range(windows):
                for t in range(L):
                    cache.decode_step(inputs[t], ys[t])
        else:
            g = torch.cuda.CUDAGraph()
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                with torch.cuda.graph(g, stream=s):
                    for t in range(L):
                        cache.decode_step(inputs[t], ys[t], stream=s)
            torch.cuda.current_stream().wait_stream(s)
            for _ in range(windows):
                g.replay()
        torch.cuda.synchronize()
        outs[mode] = ([y.cpu().numpy() for y in ys], cache.ckpt.cpu().numpy(), cache.cursor.cpu().numpy(),
                      {k: (v.view(torch.int16) if v.dtype == torch.bfloat16 else v).cpu().numpy()
                       for k, v in cache.ring_views().items()})
        assert cache.device_error() == 0
        cache.close()
    e, g = outs["eager"], outs["graph"]
    for a, b in zip(e[0], g[0]):
        np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(e[1], g[1])
    np.testing.assert_array_equal(e[2], g[2])
    for k in e[3]:
        np.testing.assert_array_equal(e[3][k], g[3][k])


@pytest.mark.parametrize("kind,P", [(MAMBA2, 64), (GDN, 128)])
def test_window_captured_as_cuda_graph_replays_like_live_calls(kind, P):
    shape = LayerShape(kind, batch=6, n_heads=8, n_groups=2, d_head=P, d_state=128, ring_len=5)
    _graph_vs_eager(shape, 151 + P, windows=3)
