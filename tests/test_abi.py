"""The C-ABI library without a GPU: it loads, exports every function the
header declares, sizes buffers per the documented layout and rejects bad
arguments on the host before touching the device."""

import ctypes
import os
import re

import pytest

import checkpoint_input_replay_gb300 as rs
from checkpoint_input_replay_gb300 import _lib

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "replayssm.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rs_[a-z_]+)\s*\(", text)))


def test_every_declared_function_is_exported():
    lib = _lib.load()
    names = _declared()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(names) == sorted(_lib.EXPORTED)


def test_query_sizes_config1_and_config2():
    st, sz = rs.rs_query_sizes(rs.rs_config(0, 256, 128, 8, 64, 128, 16, 0, 0))
    assert st == rs.RS_OK
    assert sz[0] == 256 * 128 * 64 * 128 * 4                 # 1 GiB checkpoint
    ring = (256 * 128 * 16 * 64 * 2) + (256 * 128 * 16 * 2) + (256 * 128 * 16 * 4) + (256 * 8 * 16 * 128 * 2)
    assert sz[1] == ring                                      # sections already 256-aligned here
    assert sz[2] == 256 * 16 + 16 and sz[3] == 0 and sz[4] == 256 * 4
    st, sz = rs.rs_query_sizes(rs.rs_config(1, 256, 32, 16, 128, 128, 16, 0, 0))
    assert st == rs.RS_OK and sz[0] == 512 * 1024 * 1024
    st, sz = rs.rs_query_sizes(rs.rs_config(0, 256, 128, 8, 64, 128, 16, 0, 2))
    assert st == rs.RS_OK and sz[3] == 256 * 128 * 64 * 64 + 256 * 128 * 64 * 8 + 256 * 128 * 4


def test_query_sizes_scratch_with_drafts():
    """max_draft > 0 adds the verify coefficient tables after the arrival counters."""
    st, sz = rs.rs_query_sizes(rs.rs_config(0, 512, 128, 8, 64, 128, 16, 4, 0))
    C = 16 + 4
    assert st == rs.RS_OK and sz[4] == 512 * 4 + 512 * 128 * (4 * C + 4) * 4
    st, sz = rs.rs_query_sizes(rs.rs_config(1, 3, 32, 16, 128, 128, 16, 4, 0))
    assert st == rs.RS_OK and sz[4] == 256 + 3 * 32 * (8 * C + 48) * 4


@pytest.mark.parametrize("fields,status", [
    ((3, 1, 4, 1, 16, 16, 4, 0, 0), rs.RS_ERR_RANGE),        # kind
    ((2, 1, 4, 1, 16, 16, 4, 2, 0), rs.RS_ERR_UNSUPPORTED),  # per-channel gate: no drafts
    ((0, 1, 4, 1, 16, 16, 4, 0, 7), rs.RS_ERR_RANGE),        # read mode
    ((0, 0, 4, 1, 16, 16, 4, 0, 0), rs.RS_ERR_SHAPE),        # batch
    ((0, 1, 4, 3, 16, 16, 4, 0, 0), rs.RS_ERR_SHAPE),        # heads not a multiple of groups
    ((0, 1, 4, 1, 16, 16, 0, 0, 0), rs.RS_ERR_SHAPE),        # ring_len
    ((0, 1, 4, 1, 16, 24, 4, 0, 0), rs.RS_ERR_UNSUPPORTED),  # d_state not a power of two
    ((0, 1, 4, 1, 256, 128, 4, 0, 0), rs.RS_ERR_UNSUPPORTED),  # tile above 64 KiB
    ((0, 1, 4, 1, 16, 16, 30, 3, 0), rs.RS_ERR_UNSUPPORTED),   # L + T_max > 32
    ((0, 1, 4, 1, 16, 16, 4, 5, 0), rs.RS_ERR_UNSUPPORTED),    # T_max > 4
    ((1, 1, 4, 1, 16, 16, 4, 0, 1), rs.RS_ERR_UNSUPPORTED),    # read copy on GDN
])
def test_invalid_configs(fields, status):
    st, _ = rs.rs_query_sizes(rs.rs_config(*fields))
    assert st == status


def test_null_and_alignment_errors_need_no_device():
    cfg = rs.rs_config(0, 2, 4, 1, 16, 16, 4, 0, 0)
    st, h = rs.rs_create_cache(cfg, rs.rs_buffers(None, None, None, None, None))
    assert st == rs.RS_ERR_NULL
    st, h = rs.rs_create_cache(cfg, rs.rs_buffers(4096, 4096 + 8, 8192, None, 12288))
    assert st == rs.RS_ERR_ALIGN
    st, h = rs.rs_create_cache(rs.rs_config(0, 2, 4, 1, 16, 16, 4, 0, 1),
                               rs.rs_buffers(4096, 8192, 8192, None, 12288))
    assert st == rs.RS_ERR_NULL                     # read copy buffer required
    assert rs.rs_decode_step(None, rs.rs_inputs(), 0, 0) == rs.RS_ERR_NULL
    assert rs.rs_verify(None, 1, rs.rs_inputs(), 0, 0) == rs.RS_ERR_NULL
    assert rs.rs_commit(None, 0, 0) == rs.RS_ERR_NULL
    assert rs.rs_flush(None, None, 0) == rs.RS_ERR_NULL
    # tree-shaped drafts: null handle, parents or path are rejected before any CUDA call
    assert rs.rs_verify_tree(None, 2, [-1, 0], rs.rs_inputs(), 0, 0) == rs.RS_ERR_NULL
    assert rs.rs_commit_path(None, 4096, 8192, 0) == rs.RS_ERR_NULL
    st, code = rs.rs_get_device_error(None, 0)
    assert st == rs.RS_ERR_NULL
    rs.rs_destroy_cache(None)
    # host-buffer pipe: null handles are rejected before any CUDA call
    st, pipe = rs.rs_pipe_create(None)
    assert st == rs.RS_ERR_NULL
    assert rs.rs_pipe_decode_step(None, rs.rs_inputs(), 0, 0) == rs.RS_ERR_NULL
    assert rs.rs_pipe_sync(None, 0) == rs.RS_ERR_NULL
    rs.rs_pipe_destroy(None)
    assert rs.rs_decode_step_noalloc(cfg, rs.rs_buffers(None, None, None, None, None), rs.rs_inputs(), 0, 0) \
        == rs.RS_ERR_NULL


def test_status_strings():
    for s in range(9):
        assert rs.rs_status_string(s) and rs.rs_status_string(s) != "unknown status"
    assert rs.rs_status_string(42) == "unknown status"


def test_conventional_path_host_checks_need_no_device():
    """The comparison path's calls size the snapshot pool and reject bad arguments on the host."""
    cfg = rs.rs_config(0, 512, 128, 8, 64, 128, 16, 4, 0)
    st, sz = rs.rs_snapshot_query_sizes(cfg)
    assert st == rs.RS_OK
    assert sz[0] == 512 * 5 * 128 * 64 * 128 * 4 and sz[1] == 512 * 4 + 16
    assert rs.rs_snapshot_query_sizes(rs.rs_config(0, 4, 4, 1, 16, 16, 4, 0, 0))[0] == rs.RS_ERR_RANGE
    assert rs.rs_snapshot_query_sizes(rs.rs_config(0, 4, 4, 1, 16, 16, 4, 5, 0))[0] == rs.RS_ERR_RANGE
    assert rs.rs_snapshot_query_sizes(rs.rs_config(0, 4, 4, 1, 16, 16, 4, 2, 1))[0] == rs.RS_ERR_UNSUPPORTED
    small = rs.rs_config(0, 2, 4, 1, 16, 16, 4, 2, 0)
    assert rs.rs_conventional_decode_step(small, 0, rs.rs_inputs(), 4096, 0) == rs.RS_ERR_NULL
    assert rs.rs_conventional_decode_step(small, 4096 + 4, rs.rs_inputs(), 4096, 0) == rs.RS_ERR_ALIGN
    assert rs.rs_conventional_decode_step(small, 4096, rs.rs_inputs(), 4096, 0) == rs.RS_ERR_NULL  # inputs
    assert rs.rs_snapshot_verify(small, 4096, 4096, 3, rs.rs_inputs(), 4096, 0) == rs.RS_ERR_RANGE  # T > T_max
    assert rs.rs_snapshot_verify(small, 4096, 4096, 0, rs.rs_inputs(), 4096, 0) == rs.RS_ERR_RANGE
    assert rs.rs_snapshot_verify(small, 4096, 4096 + 8, 1, rs.rs_inputs(), 4096, 0) == rs.RS_ERR_ALIGN
    assert rs.rs_snapshot_commit(small, 0, 4096, 1, 0) == rs.RS_ERR_NULL
    assert rs.rs_snapshot_commit(small, 4096, 4096, 3, 0) == rs.RS_ERR_RANGE


def test_query_sizes_per_channel_gate_ring():
    """The per-channel-gate layer's ring keeps a log decay per key channel."""
    B, H, G, P, N, L = 4, 8, 2, 32, 64, 6
    st, sz = rs.rs_query_sizes(rs.rs_config(2, B, H, G, P, N, L, 0, 0))
    a = lambda x: (x + 255) // 256 * 256
    assert st == rs.RS_OK
    assert sz[1] == a(B * H * L * P * 4) + a(B * H * L * N * 4) + a(B * G * L * N * 2)
