"""ctypes view of include/replayssm.h: the same structs and the same function names.

Argument marshalling only: every computation happens in the CUDA library.
Loading fails loudly when the library has not been built -- there is no
fallback path.
"""

from __future__ import annotations

import ctypes
import os

from .build import LIB

RS_OK = 0
RS_ERR_NULL = 1
RS_ERR_SHAPE = 2
RS_ERR_ALIGN = 3
RS_ERR_RANGE = 4
RS_ERR_STATE = 5
RS_ERR_UNSUPPORTED = 6
RS_ERR_CUDA = 7
RS_ERR_DEVICE = 8

RS_MAMBA2 = 0
RS_GDN = 1
RS_KDA = 2
RS_READ_NONE = 0
RS_READ_FP8_ROW = 1
RS_READ_NVFP4 = 2

RS_DEVERR_NONE = 0
RS_DEVERR_ACCEPTED = 1
RS_DEVERR_CURSOR = 2
RS_DEVERR_TIMEOUT = 3

EXPORTED = ("rs_query_sizes", "rs_create_cache", "rs_destroy_cache", "rs_decode_step", "rs_verify",
            "rs_commit", "rs_flush", "rs_get_device_error", "rs_status_string", "rs_decode_step_noalloc",
            "rs_selftest_wait_timeout", "rs_pipe_create", "rs_pipe_decode_step", "rs_pipe_sync",
            "rs_pipe_destroy", "rs_conventional_decode_step", "rs_snapshot_query_sizes", "rs_snapshot_verify",
            "rs_snapshot_commit", "rs_verify_tree", "rs_commit_path")


class rs_config(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int32) for name in
                ("kind", "batch", "n_heads", "n_groups", "d_head", "d_state", "ring_len", "max_draft",
                 "read_mode")]


class rs_buffers(ctypes.Structure):
    _fields_ = [(name, ctypes.c_void_p) for name in ("ckpt", "ring", "cursor", "read_copy", "scratch")]


class rs_inputs(ctypes.Structure):
    _fields_ = [(name, ctypes.c_void_p) for name in ("x", "dt", "A", "Bm", "Cm", "q", "k", "v", "g", "beta")]


class ReplayError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


_lib = None


def load() -> ctypes.CDLL:
    """The loaded library; raises if it was not built (run ``build()`` first)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"libreplayssm.so is not built ({LIB}); run checkpoint_input_replay_gb300.build")
        lib = ctypes.CDLL(LIB)
        vp, sz = ctypes.c_void_p, ctypes.POINTER(ctypes.c_size_t)
        lib.rs_query_sizes.argtypes = [ctypes.POINTER(rs_config), sz]
        lib.rs_create_cache.argtypes = [ctypes.POINTER(rs_config), ctypes.POINTER(rs_buffers), ctypes.POINTER(vp)]
        lib.rs_destroy_cache.argtypes = [vp]
        lib.rs_destroy_cache.restype = None
        lib.rs_decode_step.argtypes = [vp, ctypes.POINTER(rs_inputs), vp, vp]
        lib.rs_verify.argtypes = [vp, ctypes.c_int32, ctypes.POINTER(rs_inputs), vp, vp]
        lib.rs_commit.argtypes = [vp, vp, vp]
        lib.rs_verify_tree.argtypes = [vp, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(rs_inputs),
                                       vp, vp]
        lib.rs_commit_path.argtypes = [vp, vp, vp, vp]
        lib.rs_flush.argtypes = [vp, vp, vp]
        lib.rs_get_device_error.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int32)]
        lib.rs_selftest_wait_timeout.argtypes = [ctypes.c_int32, ctypes.POINTER(ctypes.c_int32), vp]
        lib.rs_decode_step_noalloc.argtypes = [ctypes.POINTER(rs_config), ctypes.POINTER(rs_buffers),
                                               ctypes.POINTER(rs_inputs), vp, vp]
        lib.rs_pipe_create.argtypes = [vp, ctypes.POINTER(vp)]
        lib.rs_pipe_decode_step.argtypes = [vp, ctypes.POINTER(rs_inputs), vp, vp]
        lib.rs_pipe_sync.argtypes = [vp, vp]
        lib.rs_pipe_destroy.argtypes = [vp]
        lib.rs_pipe_destroy.restype = None
        lib.rs_conventional_decode_step.argtypes = [ctypes.POINTER(rs_config), vp, ctypes.POINTER(rs_inputs), vp,
                                                    vp]
        lib.rs_snapshot_query_sizes.argtypes = [ctypes.POINTER(rs_config), sz]
        lib.rs_snapshot_verify.argtypes = [ctypes.POINTER(rs_config), vp, vp, ctypes.c_int32,
                                           ctypes.POINTER(rs_inputs), vp, vp]
        lib.rs_snapshot_commit.argtypes = [ctypes.POINTER(rs_config), vp, vp, ctypes.c_int32, vp]
        lib.rs_status_string.argtypes = [ctypes.c_int]
        lib.rs_status_string.restype = ctypes.c_char_p
        for name in EXPORTED:
            if name not in ("rs_destroy_cache", "rs_status_string", "rs_pipe_destroy"):
                getattr(lib, name).restype = ctypes.c_int
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().rs_status_string(int(status)).decode()


def check(status: int, what: str) -> None:
    if status != RS_OK:
        raise ReplayError(status, what)


# --- same-name wrappers (return the rs_status, like the C calls) ---------------

def rs_query_sizes(cfg: rs_config):
    """Returns (status, [ckpt, ring, cursor, read_copy, scratch] bytes)."""
    out = (ctypes.c_size_t * 5)()
    st = load().rs_query_sizes(ctypes.byref(cfg), out)
    return st, list(out)


def rs_create_cache(cfg: rs_config, bufs: rs_buffers):
    """Returns (status, handle)."""
    h = ctypes.c_void_p()
    st = load().rs_create_cache(ctypes.byref(cfg), ctypes.byref(bufs), ctypes.byref(h))
    return st, h


def rs_destroy_cache(handle) -> None:
    load().rs_destroy_cache(handle)


def rs_decode_step(handle, inputs: rs_inputs, y_ptr: int, stream: int) -> int:
    return load().rs_decode_step(handle, ctypes.byref(inputs), ctypes.c_void_p(y_ptr), ctypes.c_void_p(stream))


def rs_verify(handle, T: int, inputs: rs_inputs, y_ptr: int, stream: int) -> int:
    return load().rs_verify(handle, int(T), ctypes.byref(inputs), ctypes.c_void_p(y_ptr), ctypes.c_void_p(stream))


def rs_commit(handle, accepted_ptr: int, stream: int) -> int:
    return load().rs_commit(handle, ctypes.c_void_p(accepted_ptr), ctypes.c_void_p(stream))


def rs_verify_tree(handle, T: int, parents, inputs: rs_inputs, y_ptr: int, stream: int) -> int:
    """parents: T ints (host), parents[tau] in -1..tau-1."""
    arr = (ctypes.c_int32 * max(len(parents), 1))(*[int(p) for p in parents])
    return load().rs_verify_tree(handle, int(T), arr, ctypes.byref(inputs), ctypes.c_void_p(y_ptr),
                                 ctypes.c_void_p(stream))


def rs_commit_path(handle, path_len_ptr: int, path_ptr: int, stream: int) -> int:
    return load().rs_commit_path(handle, ctypes.c_void_p(path_len_ptr), ctypes.c_void_p(path_ptr),
                                 ctypes.c_void_p(stream))


def rs_flush(handle, mask_ptr: int | None, stream: int) -> int:
    return load().rs_flush(handle, ctypes.c_void_p(mask_ptr or 0), ctypes.c_void_p(stream))


def rs_get_device_error(handle, stream: int):
    """Returns (status, code)."""
    code = ctypes.c_int32(0)
    st = load().rs_get_device_error(handle, ctypes.c_void_p(stream), ctypes.byref(code))
    return st, code.value


def rs_status_string(status: int) -> str:
    return status_string(status)


def rs_decode_step_noalloc(cfg: rs_config, bufs: rs_buffers, inputs: rs_inputs, y_ptr: int, stream: int) -> int:
    """Decode step with the library's fixed arrival-counter array (no handle, no scratch buffer)."""
    return load().rs_decode_step_noalloc(ctypes.byref(cfg), ctypes.byref(bufs), ctypes.byref(inputs),
                                         ctypes.c_void_p(y_ptr), ctypes.c_void_p(stream))


def rs_selftest_wait_timeout(limit_us: int, stream: int):
    """Returns (status, device code); see the header."""
    code = ctypes.c_int32(-1)
    st = load().rs_selftest_wait_timeout(ctypes.c_int32(limit_us), ctypes.byref(code), ctypes.c_void_p(stream))
    return st, code.value


def rs_pipe_create(handle):
    """Returns (status, pipe handle) for host-buffer decode steps on this cache."""
    p = ctypes.c_void_p()
    st = load().rs_pipe_create(handle, ctypes.byref(p))
    return st, p


def rs_pipe_decode_step(pipe, host_inputs: rs_inputs, host_y_ptr: int, stream: int) -> int:
    return load().rs_pipe_decode_step(pipe, ctypes.byref(host_inputs), ctypes.c_void_p(host_y_ptr),
                                      ctypes.c_void_p(stream))


def rs_pipe_sync(pipe, stream: int) -> int:
    return load().rs_pipe_sync(pipe, ctypes.c_void_p(stream))


def rs_pipe_destroy(pipe) -> None:
    load().rs_pipe_destroy(pipe)


# --- the conventional path (comparison) ------------------------------------------

def rs_conventional_decode_step(cfg: rs_config, state_ptr: int, inputs: rs_inputs, y_ptr: int, stream: int) -> int:
    return load().rs_conventional_decode_step(ctypes.byref(cfg), ctypes.c_void_p(state_ptr), ctypes.byref(inputs),
                                              ctypes.c_void_p(y_ptr), ctypes.c_void_p(stream))


def rs_snapshot_query_sizes(cfg: rs_config):
    """Returns (status, [pool, slots] bytes)."""
    out = (ctypes.c_size_t * 2)()
    st = load().rs_snapshot_query_sizes(ctypes.byref(cfg), out)
    return st, list(out)


def rs_snapshot_verify(cfg: rs_config, pool_ptr: int, slots_ptr: int, T: int, inputs: rs_inputs, y_ptr: int,
                       stream: int) -> int:
    return load().rs_snapshot_verify(ctypes.byref(cfg), ctypes.c_void_p(pool_ptr), ctypes.c_void_p(slots_ptr),
                                     int(T), ctypes.byref(inputs), ctypes.c_void_p(y_ptr), ctypes.c_void_p(stream))


def rs_snapshot_commit(cfg: rs_config, slots_ptr: int, accepted_ptr: int, T: int, stream: int) -> int:
    return load().rs_snapshot_commit(ctypes.byref(cfg), ctypes.c_void_p(slots_ptr), ctypes.c_void_p(accepted_ptr),
                                     int(T), ctypes.c_void_p(stream))
