"""rs_decode_step_noalloc: the decode step for callers that cannot allocate.

Callers that run where they may not allocate device memory (a server or
plugin whose device memory is pre-allocated and owned by someone else) get a
decode step that takes the buffers directly and keeps its arrival counters in
a fixed array inside the library.  This file checks, through the C ABI, that
two calls in a row (a non-flush step, then a flush step) give the same outputs,
cursors and checkpoint as the regular rs_decode_step on an identical cache.

It is named so that pytest collects it last; it also passes on its own in a
fresh process.
"""

import numpy as np
import pytest
import torch

import checkpoint_input_replay_gb300 as rs
from checkpoint_input_replay_gb300 import ReplayCache, _lib
from tests.harness import assert_close, to_dev
from workloads import configs
from workloads.configs import GDN, MAMBA2, LayerShape

pytestmark = pytest.mark.gpu


_SHAPES = {
    # d_state 128: the persistent grouped kernel
    "mamba2_d128": LayerShape(MAMBA2, batch=5, n_heads=8, n_groups=2, d_head=64, d_state=128, ring_len=2),
    "gdn_d128": LayerShape(GDN, batch=5, n_heads=4, n_groups=2, d_head=128, d_state=128, ring_len=2),
    # a small d_state: the generic decode kernel
    "mamba2_d16": LayerShape(MAMBA2, batch=2, n_heads=4, n_groups=1, d_head=16, d_state=16, ring_len=2),
}


@pytest.mark.parametrize("name,read_mode,permute", [
    ("mamba2_d128", None, None), ("gdn_d128", None, None), ("mamba2_d16", None, None),
    ("mamba2_d128", "fp8", None), ("mamba2_d128", None, "5"),
])
def test_noalloc_matches_rs_decode_step_on_two_calls(name, read_mode, permute, monkeypatch):
    """Two calls in a row (a non-flush step, then a flush step at L = 2) give the same
    outputs, cursors and checkpoint (and read copy) as rs_decode_step on an identical
    cache; also with the debug CTA permutation, which this call reads too."""
    shape = _SHAPES[name]
    kind = shape.kind
    if permute is None:
        monkeypatch.delenv("RS_DEBUG_CTA_PERMUTE", raising=False)
    else:
        monkeypatch.setenv("RS_DEBUG_CTA_PERMUTE", permute)
    wl = configs.workload(shape, seed=51, s0_std=0.1)
    S0 = torch.from_numpy(wl.S0())
    regular = ReplayCache.for_shape(shape, read_mode=read_mode)
    static = ReplayCache.for_shape(shape, read_mode=read_mode)
    regular.ckpt.copy_(S0)
    static.ckpt.copy_(S0)
    if read_mode is not None:
        regular.flush()
        static.flush()
    A = torch.from_numpy(wl.A()).cuda() if kind == MAMBA2 else None
    stream = torch.cuda.current_stream().cuda_stream
    no_scratch = _lib.rs_buffers(static.bufs.ckpt, static.bufs.ring, static.bufs.cursor, static.bufs.read_copy,
                                 None)
    for t in range(2):                      # step 0: non-flush, step 1: flush (L = 2)
        inp = to_dev(wl.step(t))
        if A is not None:
            inp["A"] = A
        y_regular = regular.decode_step(inp)
        y_static = torch.empty_like(y_regular)
        st = _lib.rs_decode_step_noalloc(static.cfg, no_scratch, static._inputs(inp, (shape.batch,)),
                                         y_static.data_ptr(), stream)
        assert st == rs.RS_OK, rs.rs_status_string(st)
        torch.cuda.synchronize()
        assert_close(y_static.cpu().numpy(), y_regular.cpu().numpy(), f"call {t} output")
        np.testing.assert_array_equal(static.cursor.cpu().numpy(), regular.cursor.cpu().numpy())
    assert static.cursor.cpu().numpy()[:, 2].all()            # the second call folded
    assert_close(static.ckpt.cpu().numpy(), regular.ckpt.cpu().numpy(), "checkpoint after the flush")
    for k, v in static.read_copy_views().items():            # the copy re-quantised by the flush step
        np.testing.assert_array_equal(v.cpu().numpy(), regular.read_copy_views()[k].cpu().numpy())
    assert static.device_error() == 0 and regular.device_error() == 0


def test_noalloc_rejects_batch_above_its_array():
    cfg = rs.rs_config(MAMBA2, 16385, 4, 1, 16, 16, 4, 0, 0)
    bufs = rs.rs_buffers(4096, 4096, 4096, None, None)
    st = _lib.rs_decode_step_noalloc(cfg, bufs, rs.rs_inputs(), 4096, 0)
    assert st == rs.RS_ERR_UNSUPPORTED
