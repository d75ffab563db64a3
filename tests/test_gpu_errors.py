"""Failure detection without a GPU fault: API misuse is refused on the host,
and bad device-side data (an accepted count out of range, a corrupt cursor)
sets the sticky device error word instead of trapping."""

import numpy as np
import pytest
import torch

import checkpoint_input_replay_gb300 as rs
from checkpoint_input_replay_gb300 import _lib
from tests.harness import Pair, assert_close
from workloads import configs
from workloads.configs import MAMBA2, LayerShape

pytestmark = pytest.mark.gpu


def _pair():
    shape = LayerShape(MAMBA2, batch=3, n_heads=2, n_groups=1, d_head=16, d_state=16, ring_len=4, max_draft=2)
    return Pair(configs.Mamba2Workload(shape, seed=31, s0_std=0.1))


def test_call_order_rules():
    pair = _pair()
    with pytest.raises(rs.ReplayError) as e:
        pair.cache.commit(torch.zeros(3, dtype=torch.int32, device="cuda"))
    assert e.value.status == rs.RS_ERR_STATE
    pair.verify(0, 2)
    with pytest.raises(rs.ReplayError) as e:
        pair.decode(0)
    assert e.value.status == rs.RS_ERR_STATE
    with pytest.raises(rs.ReplayError) as e:
        pair.cache.flush()
    assert e.value.status == rs.RS_ERR_STATE
    with pytest.raises(rs.ReplayError) as e:
        pair.verify(1, 2)
    assert e.value.status == rs.RS_ERR_STATE
    pair.commit(0, 2)
    with pytest.raises(rs.ReplayError) as e:
        pair.verify(1, 3)                 # T > max_draft
    assert e.value.status == rs.RS_ERR_RANGE
    assert pair.cache.device_error() == 0


def test_accepted_out_of_range_sets_error_and_keeps_sequence():
    pair = _pair()
    pair.decode(0)
    pair.verify(0, 2)
    before = pair.cache.cursor.cpu().numpy().copy()
    ckpt_before = pair.cache.ckpt.clone()
    acc = torch.tensor([1, 5, -1], dtype=torch.int32, device="cuda")
    pair.cache.commit(acc)
    assert pair.cache.device_error() == rs._lib.RS_DEVERR_ACCEPTED
    after = pair.cache.cursor.cpu().numpy()
    assert after[0, 1] == before[0, 1] + 1            # valid sequence committed
    np.testing.assert_array_equal(after[1:, :2], before[1:, :2])
    assert torch.equal(pair.cache.ckpt[1:], ckpt_before[1:])


def test_corrupt_cursor_sets_error():
    pair = _pair()
    pair.decode(0)
    cur = pair.cache.cursor
    cur[1, 1] = 99                                     # count beyond the ring
    torch.cuda.synchronize()
    pair.cache.decode_step(pair._dev_inputs(pair.wl.step(1)))
    assert pair.cache.device_error() == rs._lib.RS_DEVERR_CURSOR
    after = pair.cache.cursor.cpu().numpy()
    assert after[1, 1] == 99 and after[0, 1] == 2 and after[2, 1] == 2


def test_bounded_wait_gives_up_without_a_fault():
    """The bounded mbarrier wait of the kernels, on a barrier nothing completes:
    it gives up after the limit, reports RS_DEVERR_TIMEOUT, and the context
    stays usable (a decode step afterwards still matches the oracle)."""
    import time
    stream = torch.cuda.current_stream().cuda_stream
    t0 = time.perf_counter()
    st, code = _lib.rs_selftest_wait_timeout(2000, stream)
    dt = time.perf_counter() - t0
    assert st == _lib.RS_OK and code == _lib.RS_DEVERR_TIMEOUT
    assert 0.002 <= dt < 1.0
    assert _lib.rs_selftest_wait_timeout(0, stream)[0] == _lib.RS_ERR_RANGE
    pair = Pair(configs.config0())
    y, ref = pair.decode(0)
    assert_close(y, ref, "decode after the timeout self-test")
    assert pair.cache.device_error() == 0
