"""Host-buffer decode steps (rs_pipe_decode_step) against the device-buffer call.

Both run the same kernels on the same inputs, so outputs, checkpoints and
cursors must match bit for bit; the host path only moves the copies onto
streams of its own (input copies overlap the previous step's kernel, the y
copy the next step's), which must not change a value.  One output tensor per
step, so every step's read-back is checked, flush steps included.
"""

import numpy as np
import pytest
import torch

from checkpoint_input_replay_gb300 import ReplayCache
from tests.harness import assert_close, to_dev
from oracle.layer import OracleLayer
from workloads import configs
from workloads.configs import GDN, MAMBA2, LayerShape

pytestmark = pytest.mark.gpu


def _pinned(inp: dict) -> dict:
    return {k: v.cpu().pin_memory() for k, v in to_dev(inp, "cpu").items()}


def _run(wl, steps: int):
    s = wl.shape
    dev_cache = ReplayCache.for_shape(s)
    host_cache = ReplayCache.for_shape(s)
    S0 = torch.from_numpy(wl.S0())
    dev_cache.ckpt.copy_(S0)
    host_cache.ckpt.copy_(S0)
    A = torch.from_numpy(wl.A()) if s.kind == MAMBA2 else None
    oracle = OracleLayer(s, [0, s.batch - 1], wl.S0()[[0, s.batch - 1]], A=wl.A() if A is not None else None)
    stream = torch.cuda.current_stream()
    ys_dev, ys_host, host_inputs, refs = [], [], [], []
    for t in range(steps):
        inp = wl.step(t)
        d = to_dev(inp)
        h = _pinned(inp)
        if A is not None:
            d["A"] = A.cuda()
            h["A"] = A.pin_memory()
        ys_dev.append(dev_cache.decode_step(d).clone())
        y_h = torch.empty(s.batch, s.n_heads, s.d_head, dtype=torch.float32).pin_memory()
        host_cache.decode_step_from_host(h, y_h, stream=stream)
        host_inputs.append(h)  # unchanged until the pipe is synchronised
        ys_host.append(y_h)
        refs.append(oracle.decode({k: v[[0, s.batch - 1]] for k, v in inp.items()}))
    host_cache.host_sync(stream)
    torch.cuda.synchronize()
    for t in range(steps):
        np.testing.assert_array_equal(ys_host[t].numpy(), ys_dev[t].cpu().numpy(), err_msg=f"step {t} y")
        assert_close(ys_host[t].numpy()[[0, s.batch - 1]], refs[t], f"step {t} output vs oracle")
    np.testing.assert_array_equal(host_cache.ckpt.cpu().numpy(), dev_cache.ckpt.cpu().numpy())
    np.testing.assert_array_equal(host_cache.cursor.cpu().numpy(), dev_cache.cursor.cpu().numpy())
    assert host_cache.device_error() == 0 and dev_cache.device_error() == 0
    host_cache.close()
    dev_cache.close()


def test_host_pipe_mamba2_matches_device_path():
    shape = LayerShape(MAMBA2, batch=5, n_heads=16, n_groups=2, d_head=64, d_state=128, ring_len=4)
    _run(configs.Mamba2Workload(shape, seed=21, s0_std=0.1), 11)


def test_host_pipe_gdn_matches_device_path():
    shape = LayerShape(GDN, batch=3, n_heads=4, n_groups=2, d_head=128, d_state=128, ring_len=3)
    _run(configs.GdnWorkload(shape, seed=22, s0_std=0.05), 8)
