"""ReplaySSM decode hot path for one GPU (sm_103a): checkpoint + input ring buffer.

The compute lives in ``libreplayssm.so`` (CUDA kernels behind the C ABI of
include/replayssm.h); this package only marshals arguments (``_lib``) and
provides device memory and streams through PyTorch (``ReplayCache``).
"""

from . import _lib
from ._lib import (EXPORTED, RS_ERR_ALIGN, RS_ERR_CUDA, RS_ERR_DEVICE, RS_ERR_NULL, RS_ERR_RANGE, RS_ERR_SHAPE,
                   RS_ERR_STATE, RS_ERR_UNSUPPORTED, RS_GDN, RS_MAMBA2, RS_OK, RS_READ_FP8_ROW, RS_READ_NONE,
                   RS_READ_NVFP4, ReplayError, rs_buffers, rs_commit, rs_config, rs_create_cache, rs_decode_step,
                   rs_decode_step_noalloc, rs_destroy_cache, rs_flush, rs_get_device_error, rs_inputs, rs_pipe_create,
                   rs_pipe_decode_step, rs_pipe_destroy, rs_pipe_sync, rs_query_sizes, rs_selftest_wait_timeout,
                   rs_status_string, rs_verify)
from ._lib import (rs_commit_path, rs_conventional_decode_step, rs_snapshot_commit, rs_snapshot_query_sizes,
                   rs_snapshot_verify, rs_verify_tree)
from .cache import ReplayCache
from .conventional import ConventionalLayer, SnapshotLayer

__all__ = ["ReplayCache", "ReplayError", "EXPORTED", "rs_config", "rs_buffers", "rs_inputs", "rs_query_sizes",
           "rs_create_cache", "rs_destroy_cache", "rs_decode_step", "rs_verify", "rs_commit", "rs_flush",
           "rs_get_device_error", "rs_status_string", "rs_decode_step_noalloc", "rs_selftest_wait_timeout",
           "rs_pipe_create", "rs_pipe_decode_step", "rs_pipe_sync", "rs_pipe_destroy",
           "ConventionalLayer", "SnapshotLayer", "rs_conventional_decode_step", "rs_snapshot_query_sizes",
           "rs_snapshot_verify", "rs_snapshot_commit", "rs_verify_tree", "rs_commit_path"]
