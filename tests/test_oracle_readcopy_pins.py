"""Pins of the oracle's low-precision read-copy branch (``OracleLayer`` with
``read_mode``), against facts the branch does not compute the same way.

The copy only serves the checkpoint read of non-flush decode steps; the
full-precision checkpoint drives the recurrence and the flush step reads it,
and every fold re-quantises the copy from the new checkpoint ("ReplaySSM
caches SSM inputs instead of state" (richland.au), "What shipped", the
paragraph on quantization; ai-jitan-hub.com, "何がどれだけ速くなったのか",
item 3).  The oracle computes the read-copy output through a shortcut (the
exact output plus the decayed copy error).  Here it is checked against:

* a hand-derived dyadic worked example (tests/golden/readcopy_dyadic.json);
* an independent route: a second plain conventional recurrence restarted
  from the dequantised copy at every fold, fed the same tokens; because the
  recurrence is linear in the state, its output S' q is the read-copy output.
  The fold timing comes from the plain window rule written out here, not
  from the oracle's ring model.
"""

import json
import os

import numpy as np
import pytest

from oracle import codecs
from oracle.layer import OracleLayer
from oracle.recurrence import mamba2_step
from workloads import configs
from workloads.configs import MAMBA2, LayerShape

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _copy_of(S: np.ndarray, mode: str) -> np.ndarray:
    """Dequantised read copy of float64 states [..][P][N], quantised from their float32 rounding."""
    S32 = np.asarray(S, dtype=np.float32)
    if mode == "fp8":
        return codecs.fp8_rows_dequantize(*codecs.fp8_rows_quantize(S32))
    return codecs.nvfp4_dequantize(*codecs.nvfp4_quantize(S32))


def _wide(inp):
    from workloads import rng
    return {k: (rng.bf16_bits_to_float(v) if v.dtype == np.uint16 else v.astype(np.float64)) for k, v in inp.items()}


def test_fp8_read_copy_dyadic_hand_values():
    case = json.load(open(os.path.join(GOLDEN, "readcopy_dyadic.json")))
    shape = LayerShape(MAMBA2, batch=1, n_heads=1, n_groups=1, d_head=1, d_state=2, ring_len=case["L"])
    S0 = np.array(case["S0"], dtype=np.float32).reshape(1, 1, 1, 2)
    lay = OracleLayer(shape, [0], S0, A=np.array([-np.log(2.0)]), read_mode="fp8")
    assert np.array_equal(lay.read_copy[0, 0, 0], np.array(case["R0"]))
    for st in case["steps"]:
        inp = {"x": np.array([[st["x"]]]), "dt": np.array([[st["dt"]]]), "B": np.array([[st["B"]]]),
               "C": np.array([[st["C"]]])}
        y = lay.decode(inp)
        assert lay.cursor()[0, 2] == int(st["flush"])
        np.testing.assert_allclose(y[0, 0, 0], st["y"], rtol=1e-15, atol=0)
        np.testing.assert_allclose(lay.last_read_out[0, 0, 0], st["y_read"], rtol=1e-15, atol=0)
        if "R" in st:
            assert np.array_equal(lay.read_copy[0, 0, 0], np.array(st["R"]))


class _Restarted:
    """The read-copy output by the independent route: a conventional Mamba-2
    recurrence over the true state and a second one over the copy-started
    state, folded by the plain window rule (decode: fold on the L-th record;
    commit: fold once count >= L)."""

    def __init__(self, shape, S0, A, mode):
        self.shape, self.A, self.mode = shape, A, mode
        self.S = np.asarray(S0, dtype=np.float64).copy()
        self.Sr = _copy_of(self.S, mode)
        self.count = np.zeros(len(S0), dtype=int)

    def _fold(self, i):
        self.count[i] = 0
        self.Sr[i] = _copy_of(self.S[i], self.mode)

    def decode(self, tok):
        self.S, y = mamba2_step(self.S, tok["x"], tok["dt"], self.A, tok["B"], tok["C"])
        self.Sr, yr = mamba2_step(self.Sr, tok["x"], tok["dt"], self.A, tok["B"], tok["C"])
        for i in range(len(self.S)):
            self.count[i] += 1
            if self.count[i] == self.shape.ring_len:
                yr[i] = y[i]          # the flush step reads the full-precision state
                self._fold(i)
        return y, yr

    def commit(self, drafts, acc):
        for t in range(drafts["x"].shape[1]):
            m = acc > t
            if m.any():
                tk = {k: v[m, t] for k, v in drafts.items()}
                self.S[m], _ = mamba2_step(self.S[m], tk["x"], tk["dt"], self.A, tk["B"], tk["C"])
                self.Sr[m], _ = mamba2_step(self.Sr[m], tk["x"], tk["dt"], self.A, tk["B"], tk["C"])
        for i in range(len(self.S)):
            self.count[i] += acc[i]
            if self.count[i] >= self.shape.ring_len:
                self._fold(i)


@pytest.mark.parametrize("mode", ["fp8", "nvfp4"])
def test_read_copy_output_equals_recurrence_restarted_from_the_copy(mode):
    shape = LayerShape(MAMBA2, batch=3, n_heads=4, n_groups=2, d_head=4, d_state=16, ring_len=4)
    wl = configs.Mamba2Workload(shape, seed=61, s0_std=0.1)
    S0, A = wl.S0(), wl.A().astype(np.float64)
    lay = OracleLayer(shape, [0, 1, 2], S0, A=A, read_mode=mode)
    ref = _Restarted(shape, S0, A, mode)
    for t in range(14):
        inp = wl.step(t)
        y = lay.decode(inp)
        y_exact, y_read = ref.decode(_wide(inp))
        np.testing.assert_allclose(y, y_exact, rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(lay.last_read_out, y_read, rtol=1e-11, atol=1e-14)
        # the copy must differ from the state, or the test would not see a wrong copy
        assert np.max(np.abs(lay.last_read_out - y)) > 1e-6 or t % 4 == 3


@pytest.mark.parametrize("mode", ["fp8", "nvfp4"])
def test_read_copy_output_after_commits_equals_restarted_recurrence(mode):
    """Verify + commit rounds (commits with and without a fold) between decode steps:
    decodes after a commit continue the copy-started recurrence through the committed drafts."""
    shape = LayerShape(MAMBA2, batch=3, n_heads=2, n_groups=1, d_head=4, d_state=16, ring_len=5, max_draft=3)
    wl = configs.Mamba2Workload(shape, seed=62, s0_std=0.1)
    S0, A = wl.S0(), wl.A().astype(np.float64)
    lay = OracleLayer(shape, [0, 1, 2], S0, A=A, read_mode=mode)
    ref = _Restarted(shape, S0, A, mode)
    t = 0
    for s, acc in enumerate([[3, 0, 1], [2, 3, 0], [1, 1, 3], [0, 2, 2]]):
        lay.verify(wl.draft(s, 3), 3)
        acc = np.array(acc)
        lay.commit(acc)
        ref.commit(_wide(wl.draft(s, 3)), acc)
        for _ in range(2):
            inp = wl.step(t)
            t += 1
            y = lay.decode(inp)
            y_exact, y_read = ref.decode(_wide(inp))
            np.testing.assert_allclose(y, y_exact, rtol=1e-12, atol=1e-15)
            np.testing.assert_allclose(lay.last_read_out, y_read, rtol=1e-11, atol=1e-14)
