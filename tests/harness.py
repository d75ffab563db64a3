"""Shared helpers of the GPU parity tests: upload generated inputs, drive a
ReplayCache and the oracle side by side, compare with the stated tolerance."""

from __future__ import annotations

import numpy as np
import torch

from checkpoint_input_replay_gb300 import ReplayCache
from oracle import codecs
from oracle.layer import OracleLayer
from workloads import rng
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
    """A device cache over the full batch and an oracle over sampled sequences.

    Besides the oracle, it keeps a model of the ring slots of the sampled
    sequences: every record the calls append, at the slot the cursor rule puts
    it, built from the generated inputs (Mamba-2: the bf16 x, dt, B and the
    float32 product dt A; GDN: the float32 g, the bf16 k and the oracle's delta
    record u from its step-by-step state), so ``check_ring`` can compare every
    live slot of the device ring with them."""

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
        self.read_mode = read_mode
        self.slots = [dict() for _ in self.seqs]
        self.pending = 0
        if read_mode is not None:
            self.cache.flush()           # quantise the initial checkpoint
            self.copy_delta = np.zeros_like(self.oracle.read_copy)
            self.copy_rows_differing = 0
            self._sync_copy(np.ones(len(self.seqs), dtype=bool), "initial copy")
        self.last_read_expected = None

    # --- read copy ---------------------------------------------------------------
    def _sync_copy(self, folded, what):
        """At a fold of sampled sequences: (1) the device's re-quantised copy must equal,
        code for code and scale for scale, the oracle codec applied to the device's own
        FP32 checkpoint; (2) where the oracle's copy (quantised from its own float64
        checkpoint rounded to FP32) rounds an element differently, remember the difference
        of the two dequantised copies, which shifts the read-copy output of the following
        non-flush steps by exactly its decayed product with q."""
        idx = [i for i in range(len(self.seqs)) if folded[i]]
        if not idx:
            return
        sel = torch.tensor([self.seqs[i] for i in idx], device=self.cache.device)
        ck = self.cache.ckpt.index_select(0, sel).cpu().numpy()
        v = {k: t.index_select(0, sel).cpu().numpy() for k, t in self.cache.read_copy_views().items()}
        if self.read_mode == "fp8":
            codes, sc = codecs.fp8_rows_quantize(ck)
            np.testing.assert_array_equal(v["codes"], codes, err_msg=what + ": FP8 codes")
            np.testing.assert_array_equal(v["row_scale"], sc, err_msg=what + ": FP8 row scales")
            deq = codecs.fp8_rows_dequantize(codes, sc)
        else:
            packed, bs, sm = codecs.nvfp4_quantize(ck)
            np.testing.assert_array_equal(v["matrix_scale"], sm, err_msg=what + ": NVFP4 matrix scales")
            np.testing.assert_array_equal(v["block_scale"], bs, err_msg=what + ": NVFP4 block scales")
            np.testing.assert_array_equal(v["codes"], packed, err_msg=what + ": NVFP4 codes")
            deq = codecs.nvfp4_dequantize(packed, bs, sm)
        for n, i in enumerate(idx):
            self.copy_delta[i] = deq[n] - self.oracle.read_copy[i]
        self.copy_rows_differing = int(np.count_nonzero(np.any(self.copy_delta != 0, axis=-1)))

    def _read_expected(self, tok):
        """Read-copy output of the last decode for the device's copy: the oracle's
        read-copy output plus the decayed effect of any element the two copies round
        differently (zero where they agree code for code)."""
        grp = (np.arange(self.shape.n_heads) * self.shape.n_groups) // self.shape.n_heads
        q = rng.bf16_bits_to_float(tok["C"][self.seqs])[:, grp, :]
        shift = np.exp(self.oracle.logdecay)[:, :, None] * np.einsum("bhpn,bhn->bhp", self.copy_delta, q)
        flushed = self.oracle.cursor()[:, 2].astype(bool)
        shift[flushed] = 0.0
        return self.oracle.last_read_out + shift

    def _dev_inputs(self, inp):
        d = to_dev(inp)
        if self.A_dev is not None:
            d["A"] = self.A_dev
        return d

    def _record(self, inp, i, lead=(), u=None):
        """The ring record of sampled sequence i for the token at index ``lead`` of its inputs."""
        b = self.seqs[i]
        if self.shape.kind == MAMBA2:
            dt = inp["dt"][(b,) + lead]
            la = (rng.bf16_bits_to_float(dt).astype(np.float32) * self.A.astype(np.float32)).astype(np.float32)
            return {"x": inp["x"][(b,) + lead], "dt": dt, "la": la, "B": inp["B"][(b,) + lead]}
        return {"u": u, "g": inp["g"][(b,) + lead], "k": inp["k"][(b,) + lead]}

    def decode(self, t: int):
        inp = self.wl.step(t)
        before = self.oracle.cursor()
        y = self.cache.decode_step(self._dev_inputs(inp))
        ref = self.oracle.decode({k: v[self.seqs] for k, v in inp.items()})
        C = self.cache.C
        for i in range(len(self.seqs)):
            u = None if self.oracle.last_deltas is None else self.oracle.last_deltas[i]
            self.slots[i][(before[i, 0] + before[i, 1]) % C] = self._record(inp, i, (), u)
        if self.read_mode is not None:
            # expected values before the copy is refreshed by this step's folds
            self.last_read_expected = self._read_expected(inp)
            self._sync_copy(self.oracle.cursor()[:, 2].astype(bool), f"decode {t}")
        return y[self.seqs].cpu().numpy(), ref

    def verify(self, s: int, T: int):
        inp = self.wl.draft(s, T)
        before = self.oracle.cursor()
        y = self.cache.verify(T, self._dev_inputs(inp))
        ref = self.oracle.verify({k: v[self.seqs] for k, v in inp.items()}, T)
        C = self.cache.C
        for i in range(len(self.seqs)):
            for tau in range(T):
                u = None if self.oracle.last_deltas is None else self.oracle.last_deltas[i, tau]
                self.slots[i][(before[i, 0] + before[i, 1] + tau) % C] = self._record(inp, i, (tau,), u)
        self.pending = T
        return y[self.seqs].cpu().numpy(), ref

    def verify_tree(self, s: int, T: int, parents):
        inp = self.wl.draft(s, T)
        before = self.oracle.cursor()
        y = self.cache.verify_tree(T, parents, self._dev_inputs(inp))
        ref = self.oracle.verify_tree({k: v[self.seqs] for k, v in inp.items()}, T, parents)
        C = self.cache.C
        for i in range(len(self.seqs)):
            for tau in range(T):
                u = None if self.oracle.last_deltas is None else self.oracle.last_deltas[i, tau]
                self.slots[i][(before[i, 0] + before[i, 1] + tau) % C] = self._record(inp, i, (tau,), u)
        self.pending = T
        self.tree = list(parents)
        return y[self.seqs].cpu().numpy(), ref

    def tree_paths(self, s: int, T: int):
        """Accepted root-to-draft path of every sequence of the batch after tree verify s:
        the path to draft accepted - 1 (none when the draw is 0)."""
        acc = self.wl.accepted(s, T)
        paths = []
        for a in acc:
            node, path = int(a) - 1, []
            while node >= 0:
                path.append(node)
                node = self.tree[node]
            paths.append(path[::-1])
        return paths

    def commit_path(self, paths):
        """paths: one list of draft indices per sequence of the batch."""
        B, Tm = self.shape.batch, self.shape.max_draft
        plen = np.array([len(p) for p in paths], dtype=np.int32)
        parr = np.zeros((B, Tm), dtype=np.int32)
        for b, p in enumerate(paths):
            parr[b, :len(p)] = p
        before = self.oracle.cursor()
        self.cache.commit_path(torch.from_numpy(plen).cuda(), torch.from_numpy(parr).cuda())
        self.oracle.commit_path([paths[b] for b in self.seqs])
        C = self.cache.C
        for i, b in enumerate(self.seqs):
            moved = [self.slots[i].get((before[i, 0] + before[i, 1] + node) % C) for node in paths[b]]
            for j, rec in enumerate(moved):
                self.slots[i][(before[i, 0] + before[i, 1] + j) % C] = rec
        self.pending = 0
        if self.read_mode is not None:
            self._sync_copy(self.oracle.cursor()[:, 2].astype(bool), "commit path")

    def commit(self, s: int, T: int, accepted=None):
        acc = self.wl.accepted(s, T) if accepted is None else np.asarray(accepted, dtype=np.int32)
        self.cache.commit(torch.from_numpy(acc).cuda())
        self.oracle.commit(acc[self.seqs])
        self.pending = 0
        if self.read_mode is not None:
            self._sync_copy(self.oracle.cursor()[:, 2].astype(bool), f"commit {s}")
        return acc

    def check_ring(self, what=""):
        """Every live slot of the sampled sequences (committed records, and the drafts
        of a pending verify) against the records the calls appended: Mamba-2 bit for
        bit; GDN g and k bit for bit, u within the FP32-path tolerance."""
        idx = torch.tensor(self.seqs, device=self.cache.device)
        ring = {k: v.index_select(0, idx) for k, v in self.cache.ring_views().items()}
        ring = {k: (v.view(torch.int16).cpu().numpy().view(np.uint16) if v.dtype == torch.bfloat16
                    else v.cpu().numpy()) for k, v in ring.items()}
        cur = self.cursor_gpu()
        C = self.cache.C
        G, H = self.shape.n_groups, self.shape.n_heads
        for i in range(len(self.seqs)):
            head, count = int(cur[i, 0]), int(cur[i, 1])
            for j in range(count + self.pending):
                sl = (head + j) % C
                rec = self.slots[i].get(sl)
                assert rec is not None, (what, i, sl)
                w = f"{what}: seq {self.seqs[i]} record {j} (slot {sl})"
                if self.shape.kind == MAMBA2:
                    np.testing.assert_array_equal(ring["x"][i, :, sl], rec["x"], err_msg=w + " x")
                    np.testing.assert_array_equal(ring["dt"][i, :, sl], rec["dt"], err_msg=w + " dt")
                    np.testing.assert_array_equal(ring["la"][i, :, sl], rec["la"], err_msg=w + " log a")
                    np.testing.assert_array_equal(ring["B"][i, :, sl], rec["B"], err_msg=w + " B")
                else:
                    np.testing.assert_array_equal(ring["g"][i, :, sl], rec["g"], err_msg=w + " g")
                    np.testing.assert_array_equal(ring["k"][i, :, sl], rec["k"], err_msg=w + " k")
                    assert_close(ring["u"][i, :, sl], rec["u"], w + " u")

    def cursor_gpu(self):
        return self.cache.cursor.cpu().numpy()[self.seqs, :3]

    def check_cursor(self, what=""):
        np.testing.assert_array_equal(self.cursor_gpu(), self.oracle.cursor(), err_msg=what)

    def check_ckpt(self, what=""):
        ck = self.cache.ckpt[self.seqs].cpu().numpy()
        assert_close(ck, self.oracle.checkpoint(), what)
