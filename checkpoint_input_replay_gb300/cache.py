"""``ReplayCache``: one SSM layer's ReplaySSM cache on one GPU.

PyTorch provides the device memory and the stream; every step of the decode
path runs in the CUDA library through the C ABI (``_lib``).  Buffers follow
the layout documented in include/replayssm.h.
"""

from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import check

_KIND = {"mamba2": _lib.RS_MAMBA2, "gdn": _lib.RS_GDN, "kda": _lib.RS_KDA}
_READ = {None: _lib.RS_READ_NONE, "none": _lib.RS_READ_NONE, "fp8": _lib.RS_READ_FP8_ROW,
         "nvfp4": _lib.RS_READ_NVFP4}

_M2_KEYS = ("x", "dt", "A", "B", "C")
_GDN_KEYS = ("q", "k", "v", "g", "beta")


def _a256(x: int) -> int:
    return (x + 255) & ~255


def marshal_inputs(kind: int, H: int, G: int, P: int, N: int, inputs: dict, lead: tuple, device) -> _lib.rs_inputs:
    """rs_inputs for one call's token tensors (checked: dtype, shape, contiguity, device)."""
    if kind == _lib.RS_MAMBA2:
        spec = {"x": (torch.bfloat16, lead + (H, P)), "dt": (torch.bfloat16, lead + (H,)),
                "A": (torch.float32, (H,)), "B": (torch.bfloat16, lead + (G, N)),
                "C": (torch.bfloat16, lead + (G, N))}
    else:
        g_shape = lead + ((H, N) if kind == _lib.RS_KDA else (H,))
        spec = {"q": (torch.bfloat16, lead + (G, N)), "k": (torch.bfloat16, lead + (G, N)),
                "v": (torch.bfloat16, lead + (H, P)), "g": (torch.float32, g_shape),
                "beta": (torch.float32, lead + (H,))}
    ptrs = {}
    for name, (dtype, shape) in spec.items():
        t = inputs[name]
        if t.dtype != dtype or tuple(t.shape) != shape or not t.is_contiguous() or t.device != device:
            raise ValueError(f"input {name}: want contiguous {dtype} {shape} on {device}, "
                             f"got {t.dtype} {tuple(t.shape)} on {t.device}")
        ptrs[name] = t.data_ptr()
    if kind == _lib.RS_MAMBA2:
        return _lib.rs_inputs(ptrs["x"], ptrs["dt"], ptrs["A"], ptrs["B"], ptrs["C"], None, None, None, None, None)
    return _lib.rs_inputs(None, None, None, None, None, ptrs["q"], ptrs["k"], ptrs["v"], ptrs["g"], ptrs["beta"])


class ReplayCache:
    """A ReplaySSM cache for one layer.

    kind       "mamba2" or "gdn" (or 0 / 1)
    batch, n_heads, n_groups, d_head, d_state, ring_len, max_draft
               as rs_config (n_groups: Mamba-2 ngroups | GDN key heads)
    read_mode  None, "fp8" or "nvfp4" (Mamba-2 only)
    """

    def __init__(self, kind, batch, n_heads, n_groups, d_head, d_state, ring_len, max_draft=0,
                 read_mode=None, device=None):
        kind = _KIND.get(kind, kind)
        self.cfg = _lib.rs_config(kind, batch, n_heads, n_groups, d_head, d_state, ring_len, max_draft,
                                  _READ[read_mode])
        st, sizes = _lib.rs_query_sizes(self.cfg)
        check(st, "rs_query_sizes")
        self.sizes = sizes
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self._mem = [torch.zeros(max(s, 16), dtype=torch.uint8, device=self.device) if s else None for s in sizes]
        ptr = lambda m: m.data_ptr() if m is not None else None
        self.bufs = _lib.rs_buffers(*(ptr(m) for m in self._mem))
        st, self.handle = _lib.rs_create_cache(self.cfg, self.bufs)
        check(st, "rs_create_cache")
        self.kind = kind
        self.B, self.H, self.G, self.P, self.N = batch, n_heads, n_groups, d_head, d_state
        self.L, self.T_max, self.C = ring_len, max_draft, ring_len + max_draft
        self.read_mode = _READ[read_mode]

    @classmethod
    def for_shape(cls, shape, read_mode=None, device=None) -> "ReplayCache":
        """From any object with kind, batch, n_heads, n_groups, d_head, d_state, ring_len, max_draft."""
        return cls(shape.kind, shape.batch, shape.n_heads, shape.n_groups, shape.d_head, shape.d_state,
                   shape.ring_len, shape.max_draft, read_mode, device)

    def close(self) -> None:
        if getattr(self, "_pipe", None):
            _lib.rs_pipe_destroy(self._pipe)
            self._pipe = None
        if getattr(self, "handle", None):
            _lib.rs_destroy_cache(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # --- views of the caller-owned buffers ---------------------------------------
    @property
    def ckpt(self) -> torch.Tensor:
        """FP32 checkpoint [B][H][P][N] (a view; write the initial state here)."""
        return self._mem[0][: self.sizes[0]].view(torch.float32).view(self.B, self.H, self.P, self.N)

    @property
    def cursor(self) -> torch.Tensor:
        """int32 [B][4]: head, count, last_flush, 0."""
        return self._mem[2][: 16 * self.B].view(torch.int32).view(self.B, 4)

    def ring_views(self) -> dict:
        """Views of the ring sections; per-head scalar rows have Cp = C rounded up to 8 slots."""
        B, H, G, P, N, C = self.B, self.H, self.G, self.P, self.N, self.C
        Cp = (C + 7) // 8 * 8
        m = self._mem[1]
        if self.kind == _lib.RS_MAMBA2:
            o1 = _a256(B * H * C * P * 2)
            o2 = o1 + _a256(B * H * Cp * 2)
            o3 = o2 + _a256(B * H * Cp * 4)
            return {
                "x": m[0:B * H * C * P * 2].view(torch.bfloat16).view(B, H, C, P),
                "dt": m[o1:o1 + B * H * Cp * 2].view(torch.bfloat16).view(B, H, Cp),
                "la": m[o2:o2 + B * H * Cp * 4].view(torch.float32).view(B, H, Cp),
                "B": m[o3:o3 + B * G * C * N * 2].view(torch.bfloat16).view(B, G, C, N),
            }
        o1 = _a256(B * H * C * P * 4)
        if self.kind == _lib.RS_KDA:   # g: a log decay per key channel
            o2 = o1 + _a256(B * H * C * N * 4)
            g = m[o1:o1 + B * H * C * N * 4].view(torch.float32).view(B, H, C, N)
        else:
            o2 = o1 + _a256(B * H * Cp * 4)
            g = m[o1:o1 + B * H * Cp * 4].view(torch.float32).view(B, H, Cp)
        return {
            "u": m[0:B * H * C * P * 4].view(torch.float32).view(B, H, C, P),
            "g": g,
            "k": m[o2:o2 + B * G * C * N * 2].view(torch.bfloat16).view(B, G, C, N),
        }

    def read_copy_views(self) -> dict:
        B, H, P, N = self.B, self.H, self.P, self.N
        m = self._mem[3]
        if self.read_mode == _lib.RS_READ_FP8_ROW:
            o1 = _a256(B * H * P * N)
            return {"codes": m[0:B * H * P * N].view(B, H, P, N),
                    "row_scale": m[o1:o1 + B * H * P * 4].view(torch.float32).view(B, H, P)}
        if self.read_mode == _lib.RS_READ_NVFP4:
            o1 = _a256(B * H * P * N // 2)
            o2 = o1 + _a256(B * H * P * (N // 16))
            return {"codes": m[0:B * H * P * N // 2].view(B, H, P, N // 2),
                    "block_scale": m[o1:o1 + B * H * P * (N // 16)].view(B, H, P, N // 16),
                    "matrix_scale": m[o2:o2 + B * H * 4].view(torch.float32).view(B, H)}
        return {}

    # --- calls ---------------------------------------------------------------------
    def _stream(self, stream) -> int:
        if stream is None:
            stream = torch.cuda.current_stream(self.device)
        return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)

    def _inputs(self, inputs: dict, lead: tuple, device=None) -> _lib.rs_inputs:
        device = self.device if device is None else device
        return marshal_inputs(self.kind, self.H, self.G, self.P, self.N, inputs, lead, device)

    def decode_step(self, inputs: dict, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """One decode token per sequence; returns y f32 [B][H][P]."""
        if y is None:
            y = torch.empty(self.B, self.H, self.P, dtype=torch.float32, device=self.device)
        check(_lib.rs_decode_step(self.handle, self._inputs(inputs, (self.B,)), y.data_ptr(), self._stream(stream)),
              "rs_decode_step")
        return y

    def verify(self, T: int, inputs: dict, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """Outputs of T draft tokens per sequence, y f32 [B][T][H][P]; commit must follow."""
        if y is None:
            y = torch.empty(self.B, T, self.H, self.P, dtype=torch.float32, device=self.device)
        check(_lib.rs_verify(self.handle, T, self._inputs(inputs, (self.B, T)), y.data_ptr(), self._stream(stream)),
              "rs_verify")
        return y

    def verify_tree(self, T: int, parents, inputs: dict, y: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
        """Tree-shaped drafts (draft tau continues draft parents[tau], -1 = the committed
        records); y f32 [B][T][H][P]; commit_path (or, for a chain, commit) must follow."""
        if y is None:
            y = torch.empty(self.B, T, self.H, self.P, dtype=torch.float32, device=self.device)
        check(_lib.rs_verify_tree(self.handle, T, list(parents), self._inputs(inputs, (self.B, T)), y.data_ptr(),
                                  self._stream(stream)), "rs_verify_tree")
        return y

    def commit_path(self, path_len: torch.Tensor, path: torch.Tensor, stream=None) -> None:
        """path_len int32 [B], path int32 [B][T_max] on the device: each sequence's accepted
        root-to-draft path of the pending verify."""
        if path_len.dtype != torch.int32 or tuple(path_len.shape) != (self.B,) or path_len.device != self.device:
            raise ValueError("path_len must be int32 [B] on the cache's device")
        if path.dtype != torch.int32 or tuple(path.shape) != (self.B, self.T_max) or path.device != self.device \
                or not path.is_contiguous():
            raise ValueError("path must be contiguous int32 [B][T_max] on the cache's device")
        check(_lib.rs_commit_path(self.handle, path_len.data_ptr(), path.data_ptr(), self._stream(stream)),
              "rs_commit_path")

    def commit(self, accepted: torch.Tensor, stream=None) -> None:
        """accepted: int32 [B] on the device."""
        if accepted.dtype != torch.int32 or tuple(accepted.shape) != (self.B,) or accepted.device != self.device:
            raise ValueError("accepted must be int32 [B] on the cache's device")
        check(_lib.rs_commit(self.handle, accepted.data_ptr(), self._stream(stream)), "rs_commit")

    def flush(self, mask: torch.Tensor | None = None, stream=None) -> None:
        """Fold the buffered records of the masked sequences (uint8 [B]; None = all)."""
        ptr = None
        if mask is not None:
            if mask.dtype != torch.uint8 or tuple(mask.shape) != (self.B,) or mask.device != self.device:
                raise ValueError("mask must be uint8 [B] on the cache's device")
            ptr = mask.data_ptr()
        check(_lib.rs_flush(self.handle, ptr, self._stream(stream)), "rs_flush")

    def device_error(self, stream=None) -> int:
        """Synchronises the stream; returns the sticky device error code (0 = none)."""
        st, code = _lib.rs_get_device_error(self.handle, self._stream(stream))
        if st not in (_lib.RS_OK, _lib.RS_ERR_DEVICE):
            check(st, "rs_get_device_error")
        return code

    # --- end to end from host memory --------------------------------------------------
    def decode_step_from_host(self, host_inputs: dict, host_y: torch.Tensor, stream=None) -> torch.Tensor:
        """Decode step whose inputs live in (pinned) host memory and whose output is
        read back to host memory, through rs_pipe_decode_step: the input copies overlap
        the previous step's kernel and the y copy the next step's.  host_y (f32
        [B][H][P], pinned) is complete after host_sync() and a synchronise of the stream;
        the host inputs must stay unchanged until then."""
        if host_y.dtype != torch.float32 or tuple(host_y.shape) != (self.B, self.H, self.P) or \
                host_y.device.type != "cpu" or not host_y.is_contiguous():
            raise ValueError("host_y must be a contiguous f32 [B][H][P] host tensor")
        if getattr(self, "_pipe", None) is None:
            st, self._pipe = _lib.rs_pipe_create(self.handle)
            check(st, "rs_pipe_create")
        check(_lib.rs_pipe_decode_step(self._pipe, self._inputs(host_inputs, (self.B,), torch.device("cpu")),
                                       host_y.data_ptr(), self._stream(stream)), "rs_pipe_decode_step")
        return host_y

    def host_sync(self, stream=None) -> None:
        """Make the stream wait for every host copy issued by decode_step_from_host."""
        if getattr(self, "_pipe", None) is not None:
            check(_lib.rs_pipe_sync(self._pipe, self._stream(stream)), "rs_pipe_sync")
