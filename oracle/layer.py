"""Expected results of the decode-path calls on a subset of sequences (test infrastructure only).

``OracleLayer`` mirrors one SSM layer of the C-ABI -- decode step, speculative
verify, commit, flush -- for the sequences listed in ``seqs``.  It never uses
the checkpoint-plus-buffer form: it runs the conventional per-token recurrence
in float64 (``recurrence``) and tracks the cursor with ``RingModel``.  What it
exposes is what ReplaySSM must reproduce:

* the output of every decode step and of every draft position of a verify
  ([richland] What shipped: outputs match conventional decoding up to
  floating-point differences; drafts are appended, verification runs);
* the checkpoint, which equals the conventional state at the last flush
  ([richland] What shipped: the flush folds the records into the checkpoint;
  [ai-jitan] ReplaySSMは何をする手法か, third bullet);
* the cursor (head, count) and the per-call flush flag of every sequence.

Speculative commit advances the committed state by the first n drafts, which
the oracle recomputes token by token from the stored draft inputs (plain
snapshots are fine here).  Inputs arrive as the workload generators produce
them (bfloat16 bit patterns, float32) and are widened exactly to float64.
"""

from __future__ import annotations

import numpy as np

from workloads import rng
from workloads.configs import GDN, KDA, MAMBA2, LayerShape

from . import codecs
from .recurrence import gdn_delta, gdn_step, kda_delta, kda_step, mamba2_step
from .ring import RingModel


def _wide(inp: dict) -> dict:
    """Exact float64 view of one token's inputs (bf16 bits or float32)."""
    out = {}
    for k, v in inp.items():
        v = np.asarray(v)
        out[k] = rng.bf16_bits_to_float(v) if v.dtype == np.uint16 else v.astype(np.float64)
    return out


class OracleLayer:
    """One layer, sequences ``seqs`` of the batch.

    shape   the layer's LayerShape (batch = full batch)
    seqs    sorted list of sequence indices this oracle follows
    S0      float32 initial states of those sequences [len(seqs)][H][P][N]
    A       Mamba-2 per-head A (float32 [H]); None for GDN
    """

    def __init__(self, shape: LayerShape, seqs, S0, A=None, read_mode=None):
        self.shape = shape
        if read_mode not in (None, "fp8", "nvfp4"):
            raise ValueError(read_mode)
        if read_mode is not None and shape.kind != MAMBA2:
            raise ValueError("read copy is modelled for Mamba-2 layers")
        self.read_mode = read_mode
        self.seqs = list(seqs)
        self.S = np.asarray(S0, dtype=np.float64).copy()
        self.ckpt = self.S.copy()
        self.A = None if A is None else np.asarray(A, dtype=np.float64)
        C = shape.ring_len + shape.max_draft
        self.rings = [RingModel(shape.ring_len, C) for _ in self.seqs]
        self._drafts = None
        self._tree = None  # parents of the pending tree verify (None: chain-shaped drafts)
        # sum of log decays applied to the state since the last flush, per head
        self.logdecay = np.zeros((len(self.seqs), shape.n_heads) + ((shape.d_state,) if shape.kind == KDA else ()))
        # dequantised read copy (float64) of each followed sequence's checkpoint
        self.read_copy = np.zeros_like(self.S) if read_mode else None
        for i in range(len(self.seqs)):
            self._refresh_read_copy(i)
        self.last_read_out = None
        # GDN: delta records u of the tokens of the last decode ([b][H][P]) or verify ([b][T][H][P])
        self.last_deltas = None

    # --- one token ---------------------------------------------------------
    def _token(self, S, tok: dict):
        """Advance states S by one token; returns (S_new, out, log decay per head)."""
        if self.shape.kind == MAMBA2:
            S_new, y = mamba2_step(S, tok["x"], tok["dt"], self.A, tok["B"], tok["C"])
            return S_new, y, tok["dt"] * self.A[None, :]
        if self.shape.kind == KDA:
            S_new, o = kda_step(S, tok["q"], tok["k"], tok["v"], tok["g"], tok["beta"])
            return S_new, o, tok["g"]
        S_new, o = gdn_step(S, tok["q"], tok["k"], tok["v"], tok["g"], tok["beta"])
        return S_new, o, tok["g"]

    def _delta(self, S, tok: dict):
        """GDN / per-channel gate: the token's delta record u from the state before it
        (None for Mamba-2)."""
        if self.shape.kind == MAMBA2:
            return None
        if self.shape.kind == KDA:
            return kda_delta(S, tok["k"], tok["v"], tok["g"], tok["beta"])
        return gdn_delta(S, tok["k"], tok["v"], tok["g"], tok["beta"])

    # --- calls ---------------------------------------------------------------
    def decode(self, inp: dict) -> np.ndarray:
        """Decode step; ``inp`` holds this oracle's rows.  Returns the outputs [b][H][P].

        With a read copy, ``last_read_out`` receives the output the decoder
        gives when the checkpoint term is read from the low-precision copy:
        the copy replaces the checkpoint only where the checkpoint is read,
        the decayed S_ckpt q term; buffered and current records stay exact,
        and a flush step reads the full-precision checkpoint it folds
        ([ai-jitan] 何がどれだけ速くなったのか, item 3; [richland] What shipped,
        the paragraph on quantization).  So y_q = y + exp(sum of log a since
        the checkpoint, this token included) (R - S_ckpt) q.
        """
        tok = _wide(inp)
        S_prev_ckpt = self.ckpt.copy() if self.read_mode else None
        self.last_deltas = self._delta(self.S, tok)
        self.S, y, ld = self._token(self.S, tok)
        self.logdecay += ld
        if self.read_mode:
            grp = (np.arange(self.shape.n_heads) * self.shape.n_groups) // self.shape.n_heads
            q = tok["C"][:, grp, :]
            err = np.einsum("bhpn,bhn->bhp", self.read_copy - S_prev_ckpt, q)
            self.last_read_out = y + np.exp(self.logdecay)[:, :, None] * err
        for i, r in enumerate(self.rings):
            if r.decode():
                self.ckpt[i] = self.S[i]
                self.logdecay[i] = 0.0
                if self.read_mode:
                    self.last_read_out[i] = y[i]
                    self._refresh_read_copy(i)
        return y

    def verify(self, drafts: dict, T: int) -> np.ndarray:
        """Outputs of all T draft positions [b][T][H][P]; the committed state is unchanged."""
        tok = {k: v[:, :T] for k, v in _wide(drafts).items()}
        Sd = self.S.copy()
        outs, deltas = [], []
        for t in range(T):
            tk = {k: v[:, t] for k, v in tok.items()}
            deltas.append(self._delta(Sd, tk))
            Sd, y, _ = self._token(Sd, tk)
            outs.append(y)
        # GDN: delta record of every draft, from the draft chain's own states [b][T][H][P]
        self.last_deltas = None if deltas[0] is None else np.stack(deltas, axis=1)
        for r in self.rings:
            r.verify(T)
        self._drafts = (tok, T)
        self._tree = None
        return np.stack(outs, axis=1)

    def verify_tree(self, drafts: dict, T: int, parents) -> np.ndarray:
        """Tree-shaped drafts: draft tau continues draft parents[tau] (-1: the last
        committed record; otherwise an earlier draft, so parents[tau] < tau).  Each
        draft's output is the conventional recurrence run along its root-to-draft path
        from the committed state; the committed state is unchanged.  Draft records
        still take the slots after the committed ones, in draft order, so accepted
        records need not be contiguous in the buffer ([warp-studio]
        推測デコーディングにおける革新と実装詳細, the sentence on tree-based
        speculative decoding).  Returns [b][T][H][P]."""
        par = [int(p) for p in parents]
        if len(par) != T or any(not -1 <= p < t for t, p in enumerate(par)):
            raise ValueError("parents[tau] must lie in -1..tau-1")
        tok = {k: v[:, :T] for k, v in _wide(drafts).items()}
        node_states, outs, deltas = [], [], []
        for t in range(T):
            base = self.S if par[t] < 0 else node_states[par[t]]
            tk = {k: v[:, t] for k, v in tok.items()}
            deltas.append(self._delta(base, tk))
            St, y, _ = self._token(base, tk)
            node_states.append(St)
            outs.append(y)
        for r in self.rings:
            r.verify(T)
        self.last_deltas = None if deltas[0] is None else np.stack(deltas, axis=1)
        self._drafts = (tok, T)
        self._tree = par
        return np.stack(outs, axis=1)

    def commit_path(self, paths) -> None:
        """Commit, per sequence, the drafts listed in paths[i]: a root-to-draft path of the
        last tree verify, in order (empty: none).  The committed state advances token by
        token along the path; the cursor advances by its length."""
        tok, T = self._drafts
        par = self._tree if self._tree is not None else list(range(-1, T - 1))
        for i, path in enumerate(paths):
            prev = -1
            for node in path:
                if not 0 <= node < T or par[node] != prev:
                    raise ValueError("not a root-to-draft path of the last verify")
                prev = node
                S_new, _, ld = self._token(self.S[i:i + 1], {k: v[i:i + 1, node] for k, v in tok.items()})
                self.S[i] = S_new[0]
                self.logdecay[i] += ld[0]
        for i, r in enumerate(self.rings):
            if r.commit(len(paths[i])):
                self.ckpt[i] = self.S[i]
                self.logdecay[i] = 0.0
                self._refresh_read_copy(i)
        self._drafts = None
        self._tree = None

    def commit(self, accepted) -> None:
        """Commit the first accepted[i] drafts of each sequence."""
        if self._tree is not None and self._tree != list(range(-1, len(self._tree) - 1)):
            raise RuntimeError("a prefix commit needs chain-shaped drafts; use commit_path")
        self._tree = None
        tok, T = self._drafts
        n = np.asarray(accepted)
        for t in range(T):
            m = n > t
            if m.any():
                S_new, _, ld = self._token(self.S[m], {k: v[m, t] for k, v in tok.items()})
                self.S[m] = S_new
                self.logdecay[m] += ld
        for i, r in enumerate(self.rings):
            if r.commit(int(n[i])):
                self.ckpt[i] = self.S[i]
                self.logdecay[i] = 0.0
                self._refresh_read_copy(i)
        self._drafts = None

    def flush(self, mask=None) -> None:
        """Fold the buffered records of the masked sequences (all when mask is None)."""
        for i, r in enumerate(self.rings):
            if mask is None or mask[i]:
                r.flush()
                self.ckpt[i] = self.S[i]
                self.logdecay[i] = 0.0
                self._refresh_read_copy(i)
            else:
                r.last_flush = 0
                r.folded = 0

    # --- what the device holds ----------------------------------------------
    def cursor(self) -> np.ndarray:
        """[b][3] int32: head, count, flush flag of the last call."""
        return np.array([[r.head, r.count, r.last_flush] for r in self.rings], dtype=np.int32)

    def checkpoint(self) -> np.ndarray:
        return self.ckpt

    # --- read copy -----------------------------------------------------------
    def _refresh_read_copy(self, i: int) -> None:
        """Re-quantise sequence i's read copy from its float32-rounded checkpoint."""
        if self.read_mode is None:
            return
        S32 = self.ckpt[i].astype(np.float32)
        if self.read_mode == "fp8":
            codes, sc = codecs.fp8_rows_quantize(S32)
            self.read_copy[i] = codecs.fp8_rows_dequantize(codes, sc)
        else:
            packed, bs, s = codecs.nvfp4_quantize(S32)
            self.read_copy[i] = codecs.nvfp4_dequantize(packed, bs, s)
