"""The conventional decode path on the same GPU, for comparison (argument marshalling only).

``ConventionalLayer`` holds one layer's recurrent state and runs the plain
per-token read-update-write decode step; ``SnapshotLayer`` holds T_max + 1
state slots per sequence and runs snapshot-per-draft speculative verify and
rollback by slot select.  Both call the C ABI (rs_conventional_decode_step,
rs_snapshot_verify, rs_snapshot_commit); PyTorch only provides the memory
and the stream.
"""

from __future__ import annotations

import torch

from . import _lib
from ._lib import check
from .cache import _KIND, marshal_inputs


def _stream(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


class ConventionalLayer:
    """Recurrent state f32 [B][H][P][N] updated in place by every decode step."""

    def __init__(self, kind, batch, n_heads, n_groups, d_head, d_state, device=None):
        kind = _KIND.get(kind, kind)
        self.cfg = _lib.rs_config(kind, batch, n_heads, n_groups, d_head, d_state, 1, 0, _lib.RS_READ_NONE)
        self.kind, self.B, self.H, self.G, self.P, self.N = kind, batch, n_heads, n_groups, d_head, d_state
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.state = torch.zeros(batch, n_heads, d_head, d_state, dtype=torch.float32, device=self.device)

    @classmethod
    def for_shape(cls, shape, device=None) -> "ConventionalLayer":
        return cls(shape.kind, shape.batch, shape.n_heads, shape.n_groups, shape.d_head, shape.d_state, device)

    def decode_step(self, inputs: dict, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        if y is None:
            y = torch.empty(self.B, self.H, self.P, dtype=torch.float32, device=self.device)
        inp = marshal_inputs(self.kind, self.H, self.G, self.P, self.N, inputs, (self.B,), self.device)
        check(_lib.rs_conventional_decode_step(self.cfg, self.state.data_ptr(), inp, y.data_ptr(),
                                               _stream(stream, self.device)), "rs_conventional_decode_step")
        return y


class SnapshotLayer:
    """State slots f32 [B][T_max+1][H][P][N] and the current slot of every sequence."""

    def __init__(self, kind, batch, n_heads, n_groups, d_head, d_state, max_draft, device=None):
        kind = _KIND.get(kind, kind)
        self.cfg = _lib.rs_config(kind, batch, n_heads, n_groups, d_head, d_state, 1, max_draft,
                                  _lib.RS_READ_NONE)
        st, sizes = _lib.rs_snapshot_query_sizes(self.cfg)
        check(st, "rs_snapshot_query_sizes")
        self.kind, self.B, self.H, self.G, self.P, self.N = kind, batch, n_heads, n_groups, d_head, d_state
        self.T_max = max_draft
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.pool = torch.zeros(batch, max_draft + 1, n_heads, d_head, d_state, dtype=torch.float32,
                                device=self.device)
        assert self.pool.numel() * 4 == sizes[0]
        self._slots = torch.zeros(sizes[1] // 4, dtype=torch.int32, device=self.device)
        self._T = 0

    @classmethod
    def for_shape(cls, shape, device=None) -> "SnapshotLayer":
        return cls(shape.kind, shape.batch, shape.n_heads, shape.n_groups, shape.d_head, shape.d_state,
                   shape.max_draft, device)

    @property
    def slots(self) -> torch.Tensor:
        """int32 [B]: the slot holding each sequence's current state."""
        return self._slots[: self.B]

    def current_state(self) -> torch.Tensor:
        """f32 [B][H][P][N] gathered from the current slots (a copy, for checks)."""
        idx = self.slots.long()
        return self.pool[torch.arange(self.B, device=self.device), idx]

    def device_error(self) -> int:
        torch.cuda.synchronize(self.device)
        return int(self._slots[self.B].item())

    def verify(self, T: int, inputs: dict, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        if y is None:
            y = torch.empty(self.B, T, self.H, self.P, dtype=torch.float32, device=self.device)
        inp = marshal_inputs(self.kind, self.H, self.G, self.P, self.N, inputs, (self.B, T), self.device)
        check(_lib.rs_snapshot_verify(self.cfg, self.pool.data_ptr(), self._slots.data_ptr(), T, inp, y.data_ptr(),
                                      _stream(stream, self.device)), "rs_snapshot_verify")
        self._T = T
        return y

    def commit(self, accepted: torch.Tensor, stream=None) -> None:
        if accepted.dtype != torch.int32 or tuple(accepted.shape) != (self.B,) or accepted.device != self.device:
            raise ValueError("accepted must be int32 [B] on the layer's device")
        check(_lib.rs_snapshot_commit(self.cfg, self._slots.data_ptr(), accepted.data_ptr(), self._T,
                                      _stream(stream, self.device)), "rs_snapshot_commit")
