"""Pins of the float64 oracle against facts fixed outside the oracle itself.

Each test checks one oracle function against something it does not compute
the same way: a closed form, an invariant of the update, the pages'
unrolled / chunkwise formulas, or hand-derived exact values
(tests/golden/dyadic_cases.json).  A dropped term, a wrong sign or index or
a transposed operand in the oracle fails at least one of them.
"""

import json
import os

import numpy as np
import pytest

from oracle.layer import OracleLayer
from oracle.recurrence import gdn_step, group_of_head, mamba2_step
from workloads import rng
from workloads.configs import GDN, MAMBA2, LayerShape

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
R = np.random.default_rng(12345)


def close(a, b, tol=1e-12):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    scale = max(1.0, float(np.max(np.abs(b))) if b.size else 1.0)
    assert np.max(np.abs(a - b)) <= tol * scale, np.max(np.abs(a - b))


# --- hand-derived exact cases ------------------------------------------------

def test_mamba2_dyadic_hand_values():
    case = json.load(open(os.path.join(GOLDEN, "dyadic_cases.json")))["mamba2"]
    S = np.array(case["S0"], dtype=np.float64)[None, None]
    A = np.array([case["A"]])
    for st in case["steps"]:
        S, y = mamba2_step(S, np.array([[st["x"]]], float), np.array([[st["dt"]]]), A,
                           np.array([[st["B"]]], float), np.array([[st["C"]]], float))
        assert np.array_equal(S[0, 0], np.array(st["S"], float))
        assert np.array_equal(y[0, 0], np.array(st["y"], float))


def test_gdn_dyadic_hand_values():
    case = json.load(open(os.path.join(GOLDEN, "dyadic_cases.json")))["gdn"]
    S = np.array(case["S0"], dtype=np.float64)[None, None]
    for st in case["steps"]:
        S, o = gdn_step(S, np.array([[st["q"]]], float), np.array([[st["k"]]], float),
                        np.array([[st["v"]]], float), np.array([[st["g"]]]), np.array([[st["beta"]]]))
        assert np.array_equal(S[0, 0], np.array(st["S"], float))
        assert np.array_equal(o[0, 0], np.array(st["o"], float))


# --- Mamba-2 closed forms ----------------------------------------------------

def test_mamba2_geometric_series():
    """Constant a, v, k from S_0: S_t = a^t S_0 + (1 - a^t)/(1 - a) v k^T, y_t = S_t q."""
    H, P, N, T = 3, 5, 6, 9
    A = np.array([-0.3, -1.7, -4.0])
    dt = np.full((1, H), 0.45)
    x = R.standard_normal((1, H, P))
    Bm = R.standard_normal((1, 1, N))
    Cm = R.standard_normal((1, 1, N))
    S0 = R.standard_normal((1, H, P, N))
    S = S0.copy()
    a = np.exp(0.45 * A)
    v = 0.45 * x[0]
    for t in range(1, T + 1):
        S, y = mamba2_step(S, x, dt, A, Bm, Cm)
        geo = (1 - a ** t) / (1 - a)
        expect = a[:, None, None] ** t * S0[0] + geo[:, None, None] * v[:, :, None] * Bm[0, 0][None, None, :]
        close(S[0], expect)
        close(y[0], expect @ Cm[0, 0])


def test_mamba2_unit_decay_is_prefix_sum():
    """A = 0 gives a = 1: the state is S_0 plus the running sum of v k^T."""
    H, P, N, G, T = 4, 3, 4, 2, 7
    A = np.zeros(H)
    S0 = R.standard_normal((2, H, P, N))
    xs = R.standard_normal((T, 2, H, P))
    dts = R.uniform(0.1, 1.0, (T, 2, H))
    Bs = R.standard_normal((T, 2, G, N))
    Cs = R.standard_normal((T, 2, G, N))
    grp = [0, 0, 1, 1]
    outer = np.einsum("tbhp,tbhn->tbhpn", dts[..., None] * xs, Bs[:, :, grp, :])
    prefix = S0[None] + np.cumsum(outer, axis=0)
    S = S0.copy()
    for t in range(T):
        S, y = mamba2_step(S, xs[t], dts[t], A, Bs[t], Cs[t])
        close(S, prefix[t])
        close(y, np.einsum("bhpn,bhn->bhp", prefix[t], Cs[t][:, grp, :]))


def test_mamba2_group_mapping():
    """Heads h use group floor(h*G/H): zeroing group 1's B leaves heads 2,3 purely decayed."""
    H, P, N, G = 4, 2, 3, 2
    assert list(group_of_head(H, G)) == [0, 0, 1, 1]
    assert list(group_of_head(32, 16)) == [i // 2 for i in range(32)]
    A = np.array([-1.0, -2.0, -3.0, -4.0])
    S0 = R.standard_normal((1, H, P, N))
    Bm = R.standard_normal((1, G, N))
    Bm[0, 1] = 0.0
    S, _ = mamba2_step(S0, R.standard_normal((1, H, P)), np.full((1, H), 0.5), A, Bm, R.standard_normal((1, G, N)))
    close(S[0, 2:], np.exp(0.5 * A[2:])[:, None, None] * S0[0, 2:])
    assert np.max(np.abs(S[0, :2] - np.exp(0.5 * A[:2])[:, None, None] * S0[0, :2])) > 1e-3


def _mamba2_records(h, H, P, N, G, Bsz=2):
    xs = R.standard_normal((h, Bsz, H, P))
    dts = R.uniform(0.05, 0.6, (h, Bsz, H))
    Bs = R.standard_normal((h, Bsz, G, N)) / np.sqrt(N)
    Cs = R.standard_normal((h, Bsz, G, N)) / np.sqrt(N)
    return xs, dts, Bs, Cs


def test_mamba2_unrolled_identity():
    """The state h tokens after the checkpoint is gamma_h S_ckpt + sum_j w_j(h) v_j k_j^T,
    with w_j(h) the product of the decays after record j
    ([richland] What shipped, the paragraph on unrolling the recurrence)."""
    H, P, N, G, h = 4, 5, 6, 2, 11
    A = -R.uniform(0.5, 4.0, H)
    S0 = R.standard_normal((2, H, P, N))
    xs, dts, Bs, Cs = _mamba2_records(h, H, P, N, G)
    grp = group_of_head(H, G)
    S = S0.copy()
    for t in range(h):
        S, _ = mamba2_step(S, xs[t], dts[t], A, Bs[t], Cs[t])
    a = np.exp(dts * A)                       # [h][b][H]
    gamma = np.prod(a, axis=0)
    unrolled = gamma[..., None, None] * S0
    for j in range(h):
        w = np.prod(a[j + 1:], axis=0) if j + 1 < h else np.ones_like(gamma)
        v = dts[j][..., None] * xs[j]
        unrolled = unrolled + w[..., None, None] * v[..., :, None] * Bs[j][:, grp, None, :]
    close(S, unrolled)


def test_mamba2_chunkwise_verify_matches_oracle():
    """Verify outputs equal O = S_ckpt Q D + V (W ⊙ (K^T Q)), with D the cumulative decay of
    each draft position and W the causally masked decay matrix
    ([richland] What shipped, the paragraph on the second, subtler benefit)."""
    H, P, N, G, L, T, h = 4, 6, 8, 2, 16, 4, 5
    shape = LayerShape(MAMBA2, 2, H, G, P, N, L, T)
    A = (-R.uniform(0.5, 4.0, H)).astype(np.float32)
    S0 = (0.1 * R.standard_normal((2, H, P, N))).astype(np.float32)
    lay = OracleLayer(shape, [0, 1], S0, A=A)
    xs, dts, Bs, Cs = _mamba2_records(h + T, H, P, N, G)
    f32 = lambda z: z.astype(np.float32)
    for t in range(h):
        lay.decode({"x": f32(xs[t]), "dt": f32(dts[t]), "B": f32(Bs[t]), "C": f32(Cs[t])})
    drafts = {"x": f32(np.moveaxis(xs[h:], 0, 1)), "dt": f32(np.moveaxis(dts[h:], 0, 1)),
              "B": f32(np.moveaxis(Bs[h:], 0, 1)), "C": f32(np.moveaxis(Cs[h:], 0, 1))}
    Y = lay.verify(drafts, T)
    # chunkwise form, per sequence and head, records 0..h+T-1 (committed then drafts)
    X = f32(xs).astype(np.float64); DT = f32(dts).astype(np.float64)
    BB = f32(Bs).astype(np.float64); CC = f32(Cs).astype(np.float64)
    grp = group_of_head(H, G)
    for b in range(2):
        for hd in range(H):
            la = DT[:, b, hd] * np.float64(A[hd])              # log decays of the h+T records
            K = BB[:, b, grp[hd], :].T                         # N x (h+T)
            V = (DT[:, b, hd][:, None] * X[:, b, hd, :]).T     # P x (h+T)
            Q = CC[h:, b, grp[hd], :].T                        # N x T
            n = h + T
            Dd = np.diag([np.exp(la[:h + tau + 1].sum()) for tau in range(T)])
            W = np.zeros((n, T))
            for s in range(n):
                for tau in range(T):
                    if s <= h + tau:
                        W[s, tau] = np.exp(la[s + 1:h + tau + 1].sum())
            O = S0[b, hd].astype(np.float64) @ Q @ Dd + V @ (W * (K.T @ Q))
            close(Y[b, :, hd, :].T, O)


# --- Gated DeltaNet closed forms and invariants --------------------------------

def _unit(v):
    return v / np.linalg.norm(v, axis=-1, keepdims=True)


def test_gdn_zero_beta_is_pure_decay():
    Hv, Hk, d = 4, 2, 5
    S0 = R.standard_normal((1, Hv, d, d))
    S = S0.copy()
    g = -R.uniform(0.1, 2.0, (6, 1, Hv))
    for t in range(6):
        S, o = gdn_step(S, R.standard_normal((1, Hk, d)), R.standard_normal((1, Hk, d)),
                        R.standard_normal((1, Hv, d)), g[t], np.zeros((1, Hv)))
    close(S, np.exp(g.sum(axis=0))[..., None, None] * S0)


def test_gdn_delta_rule_writes_value_at_key():
    """a = 1, b = 1, |k| = 1: S_t k_t = v_t, and directions orthogonal to k_t are untouched."""
    Hv, Hk, d = 2, 1, 6
    S = R.standard_normal((1, Hv, d, d))
    for _ in range(5):
        k = _unit(R.standard_normal((1, Hk, d)))
        v = R.standard_normal((1, Hv, d))
        x = R.standard_normal(d)
        x = x - (x @ k[0, 0]) * k[0, 0]                 # x orthogonal to k
        S_prev = S
        S, o = gdn_step(S, k, k, v, np.zeros((1, Hv)), np.ones((1, Hv)))
        close(S[0] @ k[0, 0], v[0])
        close(o, v)                                     # q = k reads back v
        close(S[0] @ x, S_prev[0] @ x)


def test_gdn_general_step_along_and_across_key():
    """S_t k = a(1 - b|k|^2) S_{t-1} k + b|k|^2 v and S_t x = a S_{t-1} x for x orthogonal to k."""
    Hv, Hk, d = 4, 2, 7
    S = R.standard_normal((1, Hv, d, d))
    kh = group_of_head(Hv, Hk)
    for _ in range(4):
        k = R.standard_normal((1, Hk, d))
        q = R.standard_normal((1, Hk, d))
        v = R.standard_normal((1, Hv, d))
        g = -R.uniform(0.0, 2.0, (1, Hv))
        beta = R.uniform(0.0, 1.0, (1, Hv))
        S_new, o = gdn_step(S, q, k, v, g, beta)
        for h in range(Hv):
            kk = k[0, kh[h]]
            a, b, k2 = np.exp(g[0, h]), beta[0, h], kk @ kk
            close(S_new[0, h] @ kk, a * (1 - b * k2) * (S[0, h] @ kk) + b * k2 * v[0, h])
            x = R.standard_normal(d)
            x = x - (x @ kk) / k2 * kk
            close(S_new[0, h] @ x, a * (S[0, h] @ x))
            close(o[0, h], S_new[0, h] @ q[0, kh[h]])
        S = S_new


def test_gdn_from_zero_state():
    d = 4
    k = R.standard_normal((1, 1, d)); v = R.standard_normal((1, 1, d)); q = R.standard_normal((1, 1, d))
    S, o = gdn_step(np.zeros((1, 1, d, d)), q, k, v, np.array([[-0.7]]), np.array([[0.3]]))
    close(S[0, 0], 0.3 * np.outer(v[0, 0], k[0, 0]))


def test_gdn_delta_form():
    """S_t = a S_{t-1} + u k^T with u = b (v - a S_{t-1} k): the form that lets the buffer
    hold (g, u, k) records (the '(d, k, g)' records of [warp-studio]
    推測デコーディングにおける革新と実装詳細)."""
    Hv, Hk, d = 2, 1, 5
    S = R.standard_normal((1, Hv, d, d))
    k = R.standard_normal((1, Hk, d)); q = R.standard_normal((1, Hk, d)); v = R.standard_normal((1, Hv, d))
    g = np.array([[-0.4, -1.1]]); beta = np.array([[0.2, 0.9]])
    S_new, _ = gdn_step(S, q, k, v, g, beta)
    a = np.exp(g[0])
    for h in range(Hv):
        u = beta[0, h] * (v[0, h] - a[h] * S[0, h] @ k[0, 0])
        close(S_new[0, h], a[h] * S[0, h] + np.outer(u, k[0, 0]))


def test_gdn_chunkwise_verify_with_triangular_solve():
    """Verify outputs of GDN drafts from the chunkwise form: the draft deltas U_d solve a
    unit-triangular T x T system, then O = S_ckpt Q D + U (W ⊙ (K^T Q))
    ([richland] What shipped: 'a small T×T triangular solve on the GDN delta-rule path')."""
    Hv, Hk, d, L, T, h = 4, 2, 6, 16, 4, 3
    shape = LayerShape(GDN, 1, Hv, Hk, d, d, L, T)
    S0 = (0.05 * R.standard_normal((1, Hv, d, d))).astype(np.float32)
    lay = OracleLayer(shape, [0], S0)
    n = h + T
    q = _unit(R.standard_normal((n, 1, Hk, d))).astype(np.float32)
    k = _unit(R.standard_normal((n, 1, Hk, d))).astype(np.float32)
    v = R.standard_normal((n, 1, Hv, d)).astype(np.float32)
    g = (-R.uniform(0.05, 1.5, (n, 1, Hv))).astype(np.float32)
    beta = R.uniform(0.1, 0.9, (n, 1, Hv)).astype(np.float32)
    states = [S0[0].astype(np.float64)]
    for t in range(h):
        lay.decode({"q": q[t], "k": k[t], "v": v[t], "g": g[t], "beta": beta[t]})
        states.append(lay.S[0].copy())
    mv = lambda z: np.moveaxis(z[h:], 0, 1)
    Y = lay.verify({"q": mv(q), "k": mv(k), "v": mv(v), "g": mv(g), "beta": mv(beta)}, T)
    Q64, K64, V64 = q.astype(float), k.astype(float), v.astype(float)
    A64, B64 = np.exp(g.astype(float)), beta.astype(float)
    kh = group_of_head(Hv, Hk)
    for hd in range(Hv):
        a = A64[:, 0, hd]; bt = B64[:, 0, hd]
        Kc = K64[:, 0, kh[hd], :]                      # records x d
        Qc = Q64[:, 0, kh[hd], :]
        Sc = S0[0, hd].astype(np.float64)
        prod = lambda i, j: np.prod(a[i:j + 1]) if j >= i else 1.0   # a_i ... a_j
        # committed deltas from the definition u_j = b_j (v_j - a_j S_{j} k_j)
        U = np.zeros((n, d))
        for j in range(h):
            U[j] = bt[j] * (V64[j, 0, hd] - a[j] * states[j][hd] @ Kc[j])
        # right-hand sides and the unit lower-triangular system for the drafts
        Rhs = np.zeros((T, d)); M = np.eye(T)
        for tau in range(T):
            m = h + tau
            Sk = prod(0, m - 1) * (Sc @ Kc[m]) + sum(prod(j + 1, m - 1) * U[j] * (Kc[j] @ Kc[m]) for j in range(h))
            Rhs[tau] = bt[m] * (V64[m, 0, hd] - a[m] * Sk)
            for sg in range(tau):
                M[tau, sg] = bt[m] * a[m] * prod(h + sg + 1, m - 1) * (Kc[h + sg] @ Kc[m])
        U[h:] = np.linalg.solve(M, Rhs)
        # chunkwise output O = S_ckpt Q D + U (W ⊙ K^T Q) for the draft positions
        Qd = Qc[h:].T
        Dd = np.diag([prod(0, h + tau) for tau in range(T)])
        W = np.array([[prod(s + 1, h + tau) if s <= h + tau else 0.0 for tau in range(T)] for s in range(n)])
        O = Sc @ Qd @ Dd + U.T @ (W * (Kc @ Qd))
        close(Y[0, :, hd, :].T, O, tol=1e-11)


# --- layer-level facts ---------------------------------------------------------

def test_flush_timing_config0_sixteen_flushes():
    """L = 4 and 64 decode steps give 16 flushes: the flush happens on the step whose
    append fills the buffer, and the checkpoint then equals the step-by-step state."""
    from workloads.configs import config0
    w = config0()
    s = w.shape
    lay = OracleLayer(s, range(s.batch), w.S0(), A=w.A())
    S = np.zeros((s.batch, s.n_heads, s.d_head, s.d_state))
    flushes = 0
    A = w.A().astype(np.float64)
    for t in range(64):
        inp = w.step(t)
        lay.decode(inp)
        wide = {k: rng.bf16_bits_to_float(v) for k, v in inp.items()}
        S, _ = mamba2_step(S, wide["x"], wide["dt"], A, wide["B"], wide["C"])
        cur = lay.cursor()
        if cur[0, 2]:
            flushes += 1
            close(lay.checkpoint(), S)
        assert cur[0, 1] == (t + 1) % 4
    assert flushes == 16


def test_commit_advances_by_accepted_prefix():
    """Committing n drafts equals decoding those n tokens; rejected drafts leave no trace."""
    H, P, N, G, L, T = 2, 3, 4, 1, 16, 4
    shape = LayerShape(MAMBA2, 3, H, G, P, N, L, T)
    A = (-R.uniform(0.5, 2.0, H)).astype(np.float32)
    S0 = R.standard_normal((3, H, P, N)).astype(np.float32)
    spec = OracleLayer(shape, [0, 1, 2], S0, A=A)
    plain = OracleLayer(shape, [0, 1, 2], S0, A=A)
    drafts = {"x": R.standard_normal((3, T, H, P)).astype(np.float32),
              "dt": R.uniform(0.1, 0.5, (3, T, H)).astype(np.float32),
              "B": R.standard_normal((3, T, G, N)).astype(np.float32),
              "C": R.standard_normal((3, T, G, N)).astype(np.float32)}
    Y = spec.verify(drafts, T)
    spec.commit([0, 2, 4])
    for t in range(4):
        y = plain.decode({k: v[:, t] for k, v in drafts.items()})
        close(y, Y[:, t])
        if t == 1:
            S_after2 = plain.S.copy()
    close(spec.S[0], S0[0])
    close(spec.S[1], S_after2[1])
    close(spec.S[2], plain.S[2])
    assert spec.cursor()[:, 1].tolist() == [0, 2, 4]


# --- Gated DeltaNet delta record ---------------------------------------------

def test_gdn_delta_dyadic_hand_values():
    """u = b (v - a S_{t-1} k), hand-derived on the dyadic GDN case."""
    from oracle.recurrence import gdn_delta
    case = json.load(open(os.path.join(GOLDEN, "dyadic_cases.json")))["gdn"]
    S = np.array(case["S0"], dtype=np.float64)[None, None]
    for st in case["steps"]:
        args = (np.array([[st["k"]]], float), np.array([[st["v"]]], float), np.array([[st["g"]]]),
                np.array([[st["beta"]]]))
        u = gdn_delta(S, *args)
        assert np.array_equal(u[0, 0], np.array(st["u"], float))
        S, _ = gdn_step(S, np.array([[st["q"]]], float), *args)


def test_gdn_delta_reproduces_the_state_and_vanishes_without_write():
    """S_t = a S_{t-1} + u k^T for the step-by-step state; b = 0 gives u = 0."""
    from oracle.recurrence import gdn_delta
    Hv, Hk, d = 4, 2, 6
    S = R.standard_normal((2, Hv, d, d))
    q = R.standard_normal((2, Hk, d))
    k = R.standard_normal((2, Hk, d))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = R.standard_normal((2, Hv, d))
    g = -R.uniform(0.1, 2.0, (2, Hv))
    beta = R.uniform(0.1, 0.9, (2, Hv))
    u = gdn_delta(S, k, v, g, beta)
    S1, _ = gdn_step(S, q, k, v, g, beta)
    kk = k[:, group_of_head(Hv, Hk), :]
    close(S1, np.exp(g)[:, :, None, None] * S + u[:, :, :, None] * kk[:, :, None, :])
    assert np.array_equal(gdn_delta(S, k, v, g, np.zeros_like(beta)), np.zeros_like(v))


def test_oracle_layer_records_draft_deltas_along_the_draft_chain():
    """Verify's per-draft deltas come from the draft chain's own states: draft t's u
    equals gdn_delta of the state after drafts 0..t-1."""
    from oracle.recurrence import gdn_delta
    shape = LayerShape(GDN, batch=2, n_heads=2, n_groups=1, d_head=3, d_state=4, ring_len=4, max_draft=3)
    S0 = R.standard_normal((2, 2, 3, 4))
    lay = OracleLayer(shape, [0, 1], S0)
    k = R.standard_normal((2, 3, 1, 4))
    drafts = {"q": R.standard_normal((2, 3, 1, 4)), "k": k / np.linalg.norm(k, axis=-1, keepdims=True),
              "v": R.standard_normal((2, 3, 2, 3)), "g": -R.uniform(0.1, 1.0, (2, 3, 2)),
              "beta": R.uniform(0.1, 0.9, (2, 3, 2))}
    lay.verify(drafts, 3)
    S = S0.copy()
    for t in range(3):
        tk = {n: v[:, t] for n, v in drafts.items()}
        close(lay.last_deltas[:, t], gdn_delta(S, tk["k"], tk["v"], tk["g"], tk["beta"]))
        S, _ = gdn_step(S, tk["q"], tk["k"], tk["v"], tk["g"], tk["beta"])


# --- delta rule with a per-channel gate ------------------------------------------

def test_kda_dyadic_hand_values():
    from oracle.recurrence import kda_delta, kda_step
    case = json.load(open(os.path.join(GOLDEN, "dyadic_cases.json")))["kda"]
    S = np.array(case["S0"], dtype=np.float64)[None, None]
    for st in case["steps"]:
        g = np.log(np.array([[st["a"]]], float))
        args = (np.array([[st["k"]]], float), np.array([[st["v"]]], float), g, np.array([[st["beta"]]]))
        close(kda_delta(S, *args)[0, 0], st["u"], tol=1e-15)
        S, o = kda_step(S, np.array([[st["q"]]], float), *args)
        close(S[0, 0], st["S"], tol=1e-15)
        close(o[0, 0], st["o"], tol=1e-15)


def test_kda_with_equal_channels_is_gated_deltanet():
    from oracle.recurrence import kda_step
    Hv, Hk, d = 4, 2, 6
    S = R.standard_normal((2, Hv, d, d))
    q = _unit(R.standard_normal((2, Hk, d)))
    k = _unit(R.standard_normal((2, Hk, d)))
    v = R.standard_normal((2, Hv, d))
    g = -R.uniform(0.05, 2.0, (2, Hv))
    beta = R.uniform(0.1, 0.9, (2, Hv))
    S1, o1 = kda_step(S, q, k, v, np.repeat(g[:, :, None], d, axis=2), beta)
    S2, o2 = gdn_step(S, q, k, v, g, beta)
    close(S1, S2)
    close(o1, o2)


def test_kda_without_write_is_per_channel_decay():
    """b = 0: every column c of the state decays by its own a_c, token after token."""
    from oracle.recurrence import kda_step
    Hv, Hk, d, T = 2, 1, 5, 6
    S0 = R.standard_normal((1, Hv, d, d))
    S = S0.copy()
    total = np.zeros((1, Hv, d))
    for _ in range(T):
        g = -R.uniform(0.0, 1.0, (1, Hv, d))
        total += g
        S, _ = kda_step(S, _unit(R.standard_normal((1, Hk, d))), _unit(R.standard_normal((1, Hk, d))),
                        R.standard_normal((1, Hv, d)), g, np.zeros((1, Hv)))
    close(S, S0 * np.exp(total)[:, :, None, :])


def test_kda_unrolled_identity():
    """h tokens after a checkpoint: S_h = S_c Diag(G_h) + sum_j u_j (k_j * W_j(h))^T with
    G_h the channel-wise product of all decays and W_j(h) the product of the decays after
    record j -- the checkpoint-plus-buffer form the decode kernel uses for this gate."""
    from oracle.recurrence import kda_delta, kda_step
    Hv, Hk, d, h = 3, 1, 6, 7
    Sc = R.standard_normal((1, Hv, d, d))
    S = Sc.copy()
    us, ks, gs = [], [], []
    for _ in range(h):
        q, k = _unit(R.standard_normal((1, Hk, d))), _unit(R.standard_normal((1, Hk, d)))
        v, g, b = R.standard_normal((1, Hv, d)), -R.uniform(0.0, 0.8, (1, Hv, d)), R.uniform(0.1, 0.9, (1, Hv))
        us.append(kda_delta(S, k, v, g, b)[0])
        ks.append(k[0, 0])
        gs.append(g[0])
        S, _ = kda_step(S, q, k, v, g, b)
    for hd in range(Hv):
        unrolled = Sc[0, hd] * np.exp(sum(gg[hd] for gg in gs))[None, :]
        for j in range(h):
            W = np.exp(sum(gs[i][hd] for i in range(j + 1, h))) if j + 1 < h else np.ones(d)
            unrolled = unrolled + np.outer(us[j][hd], ks[j] * W)
        close(S[0, hd], unrolled)
