"""CPU models of the decode kernel's lane layouts (no GPU).

The d_state-128 decode kernel's non-flush read-copy units and its Gated DeltaNet
non-flush units give each lane a 16-channel block of a state row and sum a row
over eight lanes by a transpose-reduce that leaves each total in one lane.
These tests replay that index arithmetic in numpy, the way the kernel writes
it, and check that every (head, row) output comes out exactly once, with the
right value, and that the shared-memory reads of a quarter-warp are
conflict-free where the layout claims so.
"""

import numpy as np
import pytest


def reduce8_lanes3(v):
    """v[lane][8] -> out[lane]: the total of v[.][lane & 7] over the eight lanes that
    share lane >> 3 (three butterfly levels, each lane keeping one half)."""
    v = np.asarray(v, dtype=np.float64)
    w = np.zeros((32, 4))
    for L in range(32):
        b2, P = (L >> 2) & 1, L ^ 4
        for i in range(4):
            send_p = v[P][i] if (P >> 2) & 1 else v[P][i + 4]
            w[L][i] = (v[L][i + 4] if b2 else v[L][i]) + send_p
    x = np.zeros((32, 2))
    for L in range(32):
        b1, P = (L >> 1) & 1, L ^ 2
        for i in range(2):
            send_p = w[P][i] if (P >> 1) & 1 else w[P][i + 2]
            x[L][i] = (w[L][i + 2] if b1 else w[L][i]) + send_p
    out = np.zeros(32)
    for L in range(32):
        b0, P = L & 1, L ^ 1
        send_p = x[P][0] if P & 1 else x[P][1]
        out[L] = (x[L][1] if b0 else x[L][0]) + send_p
    return out


def test_reduce8_lanes3_is_a_segmented_transpose_sum():
    rng = np.random.default_rng(1)
    v = rng.standard_normal((32, 8))
    out = reduce8_lanes3(v)
    for L in range(32):
        grp = [8 * (L >> 3) + c for c in range(8)]
        assert np.isclose(out[L], sum(v[g][L & 7] for g in grp))


@pytest.mark.parametrize("RW", [8, 16])
def test_read_copy_unit_covers_every_head_row_once(RW):
    """Four heads of a unit, warp tw of eight takes rows RW tw .. RW tw + RW - 1; in pass
    f lane 8 rq + cb decodes channels 16 cb .. 16 cb + 15 of row RW tw + 4 f + rq."""
    HR, NPASS = 4, RW // 4
    NV = NPASS * HR
    rows = 8 * RW
    rng = np.random.default_rng(RW)
    codes = rng.standard_normal((HR, rows, 128))
    q = rng.standard_normal(128)
    got = np.full((HR, rows), np.nan)
    seen = np.zeros((HR, rows), dtype=int)
    for tw in range(8):
        V = np.zeros((32, NV))
        for L in range(32):
            rq, cb = L >> 3, L & 7
            for f in range(NPASS):
                R = RW * tw + 4 * f + rq
                for hu in range(HR):
                    V[L][f * HR + hu] = codes[hu, R, 16 * cb:16 * cb + 16] @ q[16 * cb:16 * cb + 16]
        for g in range(NV // 8):
            tot = reduce8_lanes3(V[:, 8 * g:8 * g + 8])
            for L in range(32):
                rq, cb = L >> 3, L & 7
                hu, R = cb & 3, RW * tw + 4 * (2 * g + (cb >> 2)) + rq
                got[hu, R] = tot[L]
                seen[hu, R] += 1
    assert (seen == 1).all()
    assert np.allclose(got, codes @ q)


def test_read_copy_record_reads_hit_distinct_banks():
    """The lane that writes (head cb mod 4, row R) reads that row of every buffered record;
    with the heads' record blocks 16 bytes off the 128-byte period (2048 + 16 bytes apart
    for C = 16, P = 64) the 32 lanes touch 16 distinct 4-byte banks (two bf16 per word)."""
    P, C = 64, 16
    stride = C * P * 2 + 16
    for tw in range(8):
        for j in range(C):
            words = set()
            for L in range(32):
                rq, cb = L >> 3, L & 7
                hu, R = cb & 3, 8 * tw + 4 * (cb >> 2) + rq
                byte = hu * stride + (j * P + R) * 2
                words.add(byte // 4)
            assert len({w % 32 for w in words}) == len(words) == 16


def test_gdn_row_pairs_cover_every_row_and_pair_the_two_dots():
    """GDN: warp tw of a team of four takes rows 16 tw .. 16 tw + 15; lane 8 rq + cb holds
    channels 4 (8 i + cb) .. + 3 (i < 4); values 2 f + d (d = 0: S k, 1: S q) of pass f are
    reduced together, so lanes cb = 2 f', 2 f' + 1 end with S k and S q of one row."""
    RW, TW = 16, 4
    rng = np.random.default_rng(7)
    S = rng.standard_normal((RW * TW, 128))
    k, q = rng.standard_normal(128), rng.standard_normal(128)
    res = {}
    for tw in range(TW):
        V = np.zeros((32, 8))
        for L in range(32):
            rq, cb = L >> 3, L & 7
            ch = np.concatenate([np.arange(4 * (8 * i + cb), 4 * (8 * i + cb) + 4) for i in range(4)])
            for f in range(4):
                R = RW * tw + 4 * f + rq
                V[L][2 * f] = S[R, ch] @ k[ch]
                V[L][2 * f + 1] = S[R, ch] @ q[ch]
        tot = reduce8_lanes3(V)
        for L in range(32):
            rq, cb = L >> 3, L & 7
            R = RW * tw + 4 * (cb >> 1) + rq
            other = tot[L ^ 1]
            sk, sq = (other, tot[L]) if cb & 1 else (tot[L], other)
            if cb & 1 == 0:
                assert R not in res
                res[R] = (sk, sq)
            else:
                assert np.isclose(res[R][0], sk) and np.isclose(res[R][1], sq)
    assert sorted(res) == list(range(RW * TW))
    for R, (sk, sq) in res.items():
        assert np.isclose(sk, S[R] @ k) and np.isclose(sq, S[R] @ q)


def test_gdn_tile_loads_are_conflict_free_per_quarter_warp():
    """Per 16-byte load i, the eight lanes of a row (one quarter-warp phase) read chunks
    8 i + cb of that row: 128 contiguous bytes."""
    SEG = 32
    for i in range(4):
        for rq in range(4):
            chunks = [(rq * SEG + 8 * i + cb) for cb in range(8)]
            banks = {(c * 16 // 4) % 32 // 4 for c in chunks}
            assert len(banks) == 8


@pytest.mark.parametrize("ncol", [4, 8])
@pytest.mark.parametrize("T", [1, 3, 4])
@pytest.mark.parametrize("n", [0, 5, 15, 28])
def test_verify_prep_dots_cover_every_record_and_column_once(ncol, T, n):
    """Verify prep (d_state 128): a pass takes 4 RPL records (RPL = 8 / ncol); lane
    8 rq + cb holds channels 4 (8 i + cb) .. + 3 of record jb + 4 r + rq (clamped to the
    last record) and forms value r ncol + col; after the transpose-reduce lane cb holds
    record jb + 4 (cb // ncol) + rq, column cb % ncol.  Columns 0..3 are the queries,
    4..7 the drafts' keys; those with tau >= T are not written."""
    nr = n + T
    if nr > 32:
        pytest.skip("more records than a ring holds")
    RPL = 8 // ncol
    rng = np.random.default_rng(ncol * 100 + n * 10 + T)
    keys = rng.standard_normal((nr, 128))
    cols = rng.standard_normal((ncol, 128))
    written = {}
    npass = (nr + 4 * RPL - 1) // (4 * RPL)
    for p in range(npass):
        jb = p * 4 * RPL
        V = np.zeros((32, 8))
        for L in range(32):
            rq, cb = L >> 3, L & 7
            ch = np.concatenate([np.arange(4 * (8 * i + cb), 4 * (8 * i + cb) + 4) for i in range(4)])
            for r in range(RPL):
                j = min(jb + 4 * r + rq, nr - 1)
                for c in range(ncol):
                    V[L][r * ncol + c] = keys[j, ch] @ cols[c, ch]
        tot = reduce8_lanes3(V)
        for L in range(32):
            rq, cb = L >> 3, L & 7
            j, c = jb + 4 * (cb // ncol) + rq, cb % ncol
            if j < nr and (c % 4) < T:
                assert (j, c) not in written
                written[(j, c)] = tot[L]
    want = {(j, c) for j in range(nr) for c in range(ncol) if c % 4 < T}
    assert set(written) == want
    for (j, c), v in written.items():
        assert np.isclose(v, keys[j] @ cols[c])


def test_verify_prep_key_rows_fill_both_bank_halves():
    """Key rows padded to 320 bytes: the four consecutive records one pass reads (64
    contiguous bytes each, chunk i) fall on alternate 64-byte halves of the 128-byte bank
    period, so the warp's 256 bytes need the minimum two wavefronts."""
    row = 320
    for j0 in range(29):
        for i in range(4):
            per_bank = {}
            for L in range(32):
                rq, cb = L >> 3, L & 7
                byte = (j0 + rq) * row + 8 * (8 * i + cb)
                for w in (byte // 4, byte // 4 + 1):
                    per_bank.setdefault(w % 32, set()).add(w)
            assert max(len(v) for v in per_bank.values()) == 2


def _anc_mask(parents):
    """Row tau (bits 4 tau .. 4 tau + 3): draft tau and its draft ancestors."""
    anc = 0
    for tau, p in enumerate(parents):
        row = 1 << tau
        if p >= 0:
            row |= (anc >> (4 * p)) & 0xF
        anc |= row << (4 * tau)
    return anc


@pytest.mark.parametrize("parents", [[-1, 0, 1, 2], [-1, 0, 0, 1], [-1, -1, 1, 0], [-1, 0, 0, 0], [-1], [-1, 0, 0]])
@pytest.mark.parametrize("n", [0, 1, 9, 28])
def test_verify_prep_path_sums_match_the_path(parents, n):
    """Verify prep: sc_j = sum of the committed log decays l_j..l_{n-1} (a suffix scan, 0 past
    n-1); for draft tau (record m = n + tau) and lane j = n + sigma, ex_q = sc_{j+1} (committed
    lanes only) + the path drafts s > sigma up to tau, ex_k the same without tau, a_q / a_k
    the path drafts' totals.  For j on the path these must be the sums over the path records
    j+1..m and j+1..m-1, and sc_0 + a_q (a_k) the sum over the path up to m (m-1)."""
    T = len(parents)
    anc = _anc_mask(parents)
    on = lambda tau, s: 0 <= s < 4 and 0 <= tau < 4 and (anc >> (4 * tau + s)) & 1
    rng = np.random.default_rng(n + 7 * T)
    l = np.zeros(32)
    l[:n + T] = -rng.uniform(0.01, 30.0, n + T)
    sc = np.where(np.arange(32) < n, l, 0.0)
    o = 1
    while o < 32:  # Hillis-Steele inclusive suffix scan, as the shuffles do it
        sc = sc + np.concatenate([sc[o:], np.zeros(o)])
        o *= 2
    tot_c = sc[0]
    ld = [l[min(n + s, 31)] for s in range(4)]
    for tau in range(T):
        m = n + tau
        path = [i for i in range(m + 1) if i < n or on(tau, i - n)]
        assert path[-1] == m
        aq = sum(ld[s] for s in range(4) if s < T and on(tau, s))
        ak = sum(ld[s] for s in range(4) if s < T and on(tau, s) and s != tau)
        assert np.isclose(tot_c + aq, sum(l[i] for i in path))
        assert np.isclose(tot_c + ak, sum(l[i] for i in path if i < m))
        for j in path:
            sigma = j - n
            sc_after = sc[j + 1] if j < n else 0.0
            exq = sc_after + sum(ld[s] for s in range(4) if s < T and on(tau, s) and s > sigma)
            exk = sc_after + sum(ld[s] for s in range(4) if s < T and on(tau, s) and s > sigma and s != tau)
            assert np.isclose(exq, sum(l[i] for i in path if i > j))
            if j < m:
                assert np.isclose(exk, sum(l[i] for i in path if j < i < m))
