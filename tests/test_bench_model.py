"""The bench's algorithmic byte model (the numerator of roofline.achieved), pinned
to the library's own buffer sizes and to hand-summed totals for config 1 / 2."""

import bench
import checkpoint_input_replay_gb300 as rs
from workloads import configs


def _ring_bytes_per_slot(shape):
    cfg = rs.rs_config(shape.kind, shape.batch, shape.n_heads, shape.n_groups, shape.d_head, shape.d_state,
                       shape.ring_len, 0, 0)
    st, sz = rs.rs_query_sizes(cfg)
    assert st == rs.RS_OK
    return sz[1] / (shape.batch * shape.ring_len)  # C = L, Cp = L (16 is a multiple of 8)


def test_record_bytes_equal_the_ring_layout():
    for wl, fn in ((configs.config1(), bench.m2_bytes), (configs.config2(), bench.gdn_bytes)):
        s = wl.shape
        rec = fn(s, 1, False) - fn(s, 0, False)  # one more buffered record read
        assert rec == _ring_bytes_per_slot(s)
        # a non-flush step appends exactly one record; a flush step writes the state instead
        appended = fn(s, 0, False) - (fn(s, 0, True) - s.n_heads * s.d_head * s.d_state * 4)
        assert appended == rec


def test_config1_window_totals():
    s = configs.config1().shape
    state = 128 * 64 * 128 * 4                          # 4 MiB
    record = 128 * 64 * 2 + 128 * 2 + 128 * 4 + 8 * 128 * 2   # x, dt, log a, B = 19,200
    inputs = 128 * 64 * 2 + 128 * 2 + 2 * 8 * 128 * 2   # x, dt, B, C
    out = 128 * 64 * 4
    assert bench.m2_bytes(s, 0, False) == state + inputs + out + record == 4_267_008
    assert bench.m2_bytes(s, 15, True) == 2 * state + 15 * record + inputs + out == 8_730_112
    window = sum(bench.m2_bytes(s, h, h == 15) for h in range(16)) / 16
    assert abs(window - 4_671_952) < 1                  # 4.67 MB per sequence-step


def test_gdn_config2_step():
    s = configs.config2().shape
    state = 32 * 128 * 128 * 4                          # 2 MiB
    record = 32 * 128 * 4 + 32 * 4 + 16 * 128 * 2      # u, g, k
    inputs = 2 * 16 * 128 * 2 + 32 * 128 * 2 + 2 * 32 * 4
    out = 32 * 128 * 4
    assert bench.gdn_bytes(s, 3, False) == state + 3 * record + inputs + out + record
