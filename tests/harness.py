"""Shared helpers of the GPU parity tests: upload generated inputs, drive a
ReplayCache and the oracle side by side, compare with the stated tolerance."""

from __future__ import annotations

import numpy as np
import torch

from checkpoint_input_replay_gb300 import ReplayCache
from oracle.layer import OracleLayer
from workloads.configs import MAMBA2

# |gpu - ref| <= RTOL * max(|ref|, FLOOR), elementwise, for FP32-state paths
RTOL = 2e-4
FLOOR = 1e-3


def to_dev(inp: dict, device="cuda") -> dict:
    out = {}
    for k, v in inp.items():
        if v.dtype == np.uint16:
            out[k] = torch.from_numpy(v.view(np.int16).copy()).to(device).view(torch.bfloat16)
        else:
            out[k] = torch.from_numpy(np.ascontiguousarray(v)).to(device)
    return out


def assert_close(gpu, ref, what="", rtol=RTOL, floor=FLOOR):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    bound = rtol * np.maximum(np.abs(ref), floor)
    err = np.abs(gpu - ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err / bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; worst at {i}: "
                             f"gpu={gpu[i]!r} ref={ref[i]!r} err={err[i]:.3e} bound={bound[i]:.3e}")


class Pair:
    """A device cache over the full batch and an oracle over sampled sequences."""

    def __init__(self, wl, seqs=None, read_mode=None):
        self.wl = wl
        s = wl.shape
        self.shape = s
        self.seqs = list(range(s.batch)) if seqs is None else list(seqs)
        self.cache = ReplayCache.for_shape(s, read_mode=read_mode)
        S0 = wl.S0()
        self.cache.ckpt.copy_(torch.from_numpy(S0))
        self.A = wl.A() if s.kind == MAMBA2 else None
        self.A_dev = torch.from_numpy(self.A).cuda() if self.A is not None else None
        self.oracle = OracleLayer(s, self.seqs, S0[self.seqs], A=self.A, read_mode=read_mode)
        if read_mode is not None:
            self.cache.flush()           # quantise the initial checkpoint

    def _dev_inputs(self, inp):
        d = to_dev(inp)
        if self.A_dev is not None:
            d["A"] = self.A_dev
        return d

    def decode(self, t: int):
        inp = self.wl.step(t)
        y = self.cache.decode_step(self._dev_inputs(inp))
        ref = self.oracle.decode({k: v[self.seqs] for k, v in inp.items()})
        return y[self.seqs].cpu().numpy(), ref

    def verify(self, s: int, T: int):
        inp = self.wl.draft(s, T)
        y = self.cache.verify(T, self._dev_inputs(inp))
        ref = self.oracle.verify({k: v[self.seqs] for k, v in inp.items()}, T)
        return y[self.seqs].cpu().numpy(), ref

    def commit(self, s: int, T: int, accepted=None):
        acc = self.wl.accepted(s, T) if accepted is None else np.asarray(accepted, dtype=np.int32)
        self.cache.commit(torch.from_numpy(acc).cuda())
        self.oracle.commit(acc[self.seqs])
        return acc

    def cursor_gpu(self):
        return self.cache.cursor.cpu().numpy()[self.seqs, :3]

    def check_cursor(self, what=""):
        np.testing.assert_array_equal(self.cursor_gpu(), self.oracle.cursor(), err_msg=what)

    def check_ckpt(self, what=""):
        ck = self.cache.ckpt[self.seqs].cpu().numpy()
        assert_close(ck, self.oracle.checkpoint(), what)
