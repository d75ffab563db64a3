"""A schedule model of the d_state-128 decode kernel's roles, checking the rule its
launcher uses for the number of stages.

Roles, as in the kernel: the producer issues unit i into stage i mod S after unit
i - S has been released, and stages group g + 1's buffer (of three, g + 1 mod 3)
at the first unit of group g; the builder finishes group g's tables after the
buffer's copies land; the prologue hands unit i over once its copies landed and,
at a group's first unit, once the group's tables are in place; computing teams
take units in turn and release them.  With random copy and compute times, every
restage of a group buffer must come after all units of the group that used it
were released and its tables were read, for S = min(cap, units per group + 1) --
the launcher's rule -- and the walk over units and over groups must agree.
"""

import random

import numpy as np

import pytest


def _units(u0, u1, H, hpg, spl, step_of):
    out, ui = [], u0
    b = u0 // (H * spl)
    r = u0 - b * H * spl
    h, sp = r // spl, r % spl
    g, hh = h // hpg, h % hpg
    while ui < u1:
        out.append((b, g, hh, sp))
        st = step_of(b)
        if spl > 1:
            ui += 1
            sp += 1
            if sp < spl:
                continue
            sp, st = 0, 1
        else:
            ui += st
        h += st
        hh += st
        if hh == hpg:
            hh, g = 0, g + 1
        if h == H:
            h, g, b = 0, 0, b + 1
    return out


def _groups(u0, u1, H, G, hpg, spl):
    b = u0 // (H * spl)
    r = u0 - b * H * spl
    h, sp0 = r // spl, r % spl
    g, hh0, ui0 = h // hpg, h % hpg, u0
    out = []
    while ui0 < u1:
        out.append((b, g, hh0, sp0))
        g += 1
        if g == G:
            g, b = 0, b + 1
        hh0, sp0, ui0 = 0, 0, (b * H + g * hpg) * spl
    return out


def _simulate(B, H, G, spl, hr, cap, teams, grid, flushing, rnd, extra_stages=0):
    hpg = H // G
    total = B * H * spl
    per = ((total + grid - 1) // grid + hr - 1) // hr * hr
    grid = (total + per - 1) // per
    stages = min(cap + extra_stages, hpg * spl // hr + 1 + extra_stages)
    for c in range(grid):
        u0, u1 = c * per, min((c + 1) * per, total)
        if u0 >= u1:
            continue
        units = _units(u0, u1, H, hpg, spl, lambda b: 1 if (hr == 1 or b in flushing) else hr)
        groups = _groups(u0, u1, H, G, hpg, spl)
        gi_of, gi = [], -1
        for i, (b, g, hh, sp) in enumerate(units):
            if i == 0 or (hh == 0 and sp == 0):
                gi += 1
                assert groups[gi] == (b, g, hh, sp)  # the two walks agree
            gi_of.append(gi)
        assert gi + 1 == len(groups)
        n = len(units)
        release = [0.0] * n
        tready, owner = {}, {}
        t_prod = t_build = t_pro = 0.0
        team_free = [0.0] * teams

        def stage(g, t):
            nonlocal t_build
            x = g % 3
            if x in owner:
                prev = owner[x]
                assert all(release[j] <= t for j in range(n) if gi_of[j] == prev), "restaged before release"
                assert tready[prev] <= t
            owner[x] = g
            t_build = max(t_build, t + rnd.uniform(0.5, 3.0)) + rnd.uniform(0.2, 4.0)
            tready[g] = t_build

        for i in range(n):
            t = max(t_prod + 0.01, release[i - stages] if i >= stages else 0.0)
            first = i == 0 or (units[i][2] == 0 and units[i][3] == 0)
            if i == 0:
                stage(0, t)
            full = t + rnd.uniform(0.5, 4.0)
            if first and gi_of[i] + 1 < len(groups):
                stage(gi_of[i] + 1, t)
            t_prod = t
            t_pro = max(t_pro + 0.01, full, tready[gi_of[i]] if first else 0.0)
            tm = i % teams
            release[i] = max(team_free[tm], t_pro) + rnd.uniform(0.5, 3.0)
            team_free[tm] = release[i]


@pytest.mark.parametrize("B,H,G,spl,hr,teams,grid", [
    (256, 32, 16, 2, 1, 2, 152),   # GDN d_head 128: half-head units
    (5, 6, 2, 2, 1, 2, 152),
    (256, 128, 8, 1, 1, 2, 152),   # Mamba-2 FP32
    (3, 6, 3, 1, 1, 2, 5),
    (256, 128, 8, 1, 4, 1, 152),   # read copy: four-head non-flush units
    (9, 16, 4, 1, 4, 1, 11),
    (7, 5, 5, 1, 1, 2, 4),         # one head per group
    (1, 2, 1, 2, 1, 2, 3),
])
def test_group_buffer_restage_never_precedes_release(B, H, G, spl, hr, teams, grid):
    rnd = random.Random(B * 1000 + H)
    for _ in range(10):
        flushing = {b for b in range(B) if rnd.random() < 0.2}
        _simulate(B, H, G, spl, hr, 5, teams, grid, flushing, rnd)


def test_the_model_catches_one_stage_too_many():
    """With one stage more than the rule a group buffer is restaged while a unit of
    the group that used it is still being computed."""
    rnd = random.Random(1)
    with pytest.raises(AssertionError, match="restaged before release"):
        for _ in range(20):
            _simulate(256, 32, 16, 2, 1, 8, 2, 152, {b for b in range(256) if rnd.random() < 0.2}, rnd,
                      extra_stages=1)


# --- weighted work split of the decode launch ------------------------------------

def _split(weights, upseq, grid, hr=1):
    """Unit range of every CTA: units whose weight interval starts in
    [c ceil(W / grid), (c + 1) ceil(W / grid)), rounded down to multiples of hr (the
    launch's rule)."""
    W = sum(weights) * upseq
    def units_before(T):
        cum, n = 0, 0
        for w in weights:
            if T > cum:
                n += min(upseq, -(-(T - cum) // w))
            cum += w * upseq
        return n - n % hr
    per_w = -(-W // grid)
    bounds = [units_before(min(W, c * per_w)) for c in range(grid)] + [len(weights) * upseq]
    return list(zip(bounds[:-1], bounds[1:]))


@pytest.mark.parametrize("flush_every", [0, 1, 16, 5])
def test_weighted_split_covers_every_unit_once_and_balances(flush_every):
    rng = np.random.default_rng(flush_every)
    B, upseq, grid = 256, 128, 152
    flush = (rng.integers(0, flush_every, B) == 0) if flush_every else np.zeros(B, bool)
    weights = [9 if f else 4 for f in flush]
    ranges = _split(weights, upseq, grid)
    assert ranges[0][0] == 0 and ranges[-1][1] == B * upseq
    assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
    assert all(lo <= hi for lo, hi in ranges)
    unit_w = np.repeat(weights, upseq)
    cost = np.array([unit_w[lo:hi].sum() for lo, hi in ranges])
    assert cost.max() <= cost.mean() + 9          # within one unit of an even share
    seqs = [(hi - 1) // upseq - lo // upseq + 1 for lo, hi in ranges if hi > lo]
    assert max(seqs) + 2 <= 64                    # the per-CTA cursor table


def test_weighted_split_keeps_read_copy_units_whole():
    weights = [9 if b % 7 == 0 else 4 for b in range(40)]
    for lo, hi in _split(weights, 16, 152, hr=4):
        assert lo % 4 == 0 and hi % 4 == 0


def test_weighted_split_with_equal_weights_is_the_even_split():
    B, upseq, grid = 256, 64, 152
    per = -(-B * upseq // grid)
    ranges = _split([4] * B, upseq, grid)
    assert ranges == [(min(c * per, B * upseq), min((c + 1) * per, B * upseq)) for c in range(grid)]
