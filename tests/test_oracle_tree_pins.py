"""Pins of the oracle's tree-shaped speculative verify and path commit.

Tree drafts: draft tau continues draft parents[tau] (-1 = the last committed
record), so the records a draft depends on are the committed ones plus its
ancestors, which need not be contiguous in the buffer ([warp-studio]
推測デコーディングにおける革新と実装詳細, the sentence on tree-based
speculative decoding).  The chunkwise form of the chain case ([richland]
What shipped, the paragraph on the second, subtler benefit) carries over with
the causal mask of W replaced by the ancestor mask: W[s, tau] is nonzero only
for committed records and for s on the root-to-tau path, and on the Gated
DeltaNet path the T x T system couples a draft only to its ancestors.  These
tests check the oracle's verify_tree against that masked chunkwise form
(computed here independently), against the chain case, and its commit_path
against plain decode steps along the path.
"""

import numpy as np
import pytest

from oracle.layer import OracleLayer
from oracle.recurrence import gdn_step, group_of_head, mamba2_step
from workloads.configs import GDN, MAMBA2, LayerShape

R = np.random.default_rng(4242)
TREES = [[-1, 0, 1, 2], [-1, -1, 0, 1], [-1, 0, 0, 2], [-1, -1, -1, -1], [-1, 0, 1, 0]]


def close(a, b, tol=1e-11):
    a, b = np.asarray(a, float), np.asarray(b, float)
    assert np.max(np.abs(a - b)) <= tol * max(1.0, float(np.max(np.abs(b)))), np.max(np.abs(a - b))


def ancestors(parents, tau, self_too=True):
    out, p = [], (tau if self_too else parents[tau])
    while p >= 0:
        out.append(p)
        p = parents[p]
    return sorted(out)


def _m2_setup(h, T, H=3, P=4, N=6, G=1):
    shape = LayerShape(MAMBA2, 1, H, G, P, N, 16, T)
    A = (-R.uniform(0.5, 3.0, H)).astype(np.float32)
    S0 = (0.1 * R.standard_normal((1, H, P, N))).astype(np.float32)
    lay = OracleLayer(shape, [0], S0, A=A)
    n = h + T
    rec = {"x": R.standard_normal((n, 1, H, P)), "dt": R.uniform(0.05, 0.6, (n, 1, H)),
           "B": R.standard_normal((n, 1, G, N)) / np.sqrt(N), "C": R.standard_normal((n, 1, G, N)) / np.sqrt(N)}
    rec = {k: v.astype(np.float32) for k, v in rec.items()}
    for t in range(h):
        lay.decode({k: v[t] for k, v in rec.items()})
    drafts = {k: np.moveaxis(v[h:], 0, 1) for k, v in rec.items()}
    return lay, rec, drafts, A, S0


@pytest.mark.parametrize("parents", TREES)
def test_mamba2_tree_verify_is_the_ancestor_masked_chunkwise_form(parents):
    """O_tau = D_tau S_ckpt q_tau + sum over committed and ancestor records s of
    w_s(tau) v_s (k_s . q_tau), decays taken along the root-to-tau path."""
    h, T = 3, 4
    lay, rec, drafts, A, S0 = _m2_setup(h, T)
    Y = lay.verify_tree(drafts, T, parents)
    H = A.shape[0]
    X, DT, BB, CC = (rec[k].astype(np.float64) for k in ("x", "dt", "B", "C"))
    for hd in range(H):
        la = DT[:, 0, hd] * np.float64(A[hd])
        for tau in range(T):
            path = list(range(h)) + [h + s for s in ancestors(parents, tau)]   # records in order
            q = CC[h + tau, 0, 0]
            D = np.exp(sum(la[r] for r in path))
            o = D * (S0[0, hd].astype(np.float64) @ q)
            for i, sidx in enumerate(path):
                w = np.exp(sum(la[r] for r in path[i + 1:]))
                o = o + w * DT[sidx, 0, hd] * X[sidx, 0, hd] * (BB[sidx, 0, 0] @ q)
            close(Y[0, tau, hd], o)


@pytest.mark.parametrize("parents", TREES)
def test_gdn_tree_verify_is_the_ancestor_masked_triangular_solve(parents):
    """GDN: draft deltas solve U M = Rhs with M coupling a draft only to its strict
    ancestors, then O_tau = D_tau S_ckpt q_tau + sum over committed and ancestor records."""
    Hv, Hk, d, h, T = 2, 1, 5, 2, 4
    shape = LayerShape(GDN, 1, Hv, Hk, d, d, 16, T)
    S0 = (0.05 * R.standard_normal((1, Hv, d, d))).astype(np.float32)
    lay = OracleLayer(shape, [0], S0)
    n = h + T
    unit = lambda z: z / np.linalg.norm(z, axis=-1, keepdims=True)
    q = unit(R.standard_normal((n, 1, Hk, d))).astype(np.float32)
    k = unit(R.standard_normal((n, 1, Hk, d))).astype(np.float32)
    v = R.standard_normal((n, 1, Hv, d)).astype(np.float32)
    g = (-R.uniform(0.05, 1.5, (n, 1, Hv))).astype(np.float32)
    beta = R.uniform(0.1, 0.9, (n, 1, Hv)).astype(np.float32)
    states = [S0[0].astype(np.float64)]
    for t in range(h):
        lay.decode({"q": q[t], "k": k[t], "v": v[t], "g": g[t], "beta": beta[t]})
        states.append(lay.S[0].copy())
    mv = lambda z: np.moveaxis(z[h:], 0, 1)
    Y = lay.verify_tree({"q": mv(q), "k": mv(k), "v": mv(v), "g": mv(g), "beta": mv(beta)}, T, parents)
    kh = group_of_head(Hv, Hk)
    for hd in range(Hv):
        a = np.exp(g[:, 0, hd].astype(float))
        bt = beta[:, 0, hd].astype(float)
        Kc, Qc, V = k[:, 0, kh[hd]].astype(float), q[:, 0, kh[hd]].astype(float), v[:, 0, hd].astype(float)
        Sc = S0[0, hd].astype(np.float64)
        U = np.zeros((n, d))
        for j in range(h):
            U[j] = bt[j] * (V[j] - a[j] * states[j][hd] @ Kc[j])
        prodr = lambda recs: float(np.prod([a[r] for r in recs])) if recs else 1.0
        Rhs, M = np.zeros((T, d)), np.eye(T)
        for tau in range(T):
            m = h + tau
            before = list(range(h)) + [h + s for s in ancestors(parents, tau, self_too=False)]
            Sk = prodr(before) * (Sc @ Kc[m])
            for i, r in enumerate(before):
                if r < h:
                    Sk = Sk + prodr(before[i + 1:]) * U[r] * (Kc[r] @ Kc[m])
            Rhs[tau] = bt[m] * (V[m] - a[m] * Sk)
            for i, r in enumerate(before):
                if r >= h:
                    M[tau, r - h] = bt[m] * a[m] * prodr(before[i + 1:]) * (Kc[r] @ Kc[m])
        U[h:] = np.linalg.solve(M, Rhs)
        for tau in range(T):
            path = list(range(h)) + [h + s for s in ancestors(parents, tau)]
            o = prodr(path) * (Sc @ Qc[h + tau])
            for i, r in enumerate(path):
                o = o + prodr(path[i + 1:]) * U[r] * (Kc[r] @ Qc[h + tau])
            close(Y[0, tau, hd], o)


def test_chain_tree_equals_chain_verify():
    lay, rec, drafts, A, S0 = _m2_setup(2, 4)
    Y_tree = lay.verify_tree(drafts, 4, [-1, 0, 1, 2])
    lay.commit_path([[]])
    Y_chain = lay.verify(drafts, 4)
    close(Y_tree, Y_chain, tol=0)


@pytest.mark.parametrize("parents,path", [([-1, -1, 0, 1], [1, 3]), ([-1, 0, 0, 2], [0, 2, 3]),
                                          ([-1, -1, -1, -1], [2]), ([-1, 0, 1, 2], [0, 1, 2, 3]),
                                          ([-1, 0, 1, 0], [])])
def test_commit_path_equals_plain_decode_along_the_path(parents, path):
    """After commit_path, the committed state is the plain recurrence run over the path's
    tokens in order, and the cursor advanced by the path length."""
    h, T = 3, 4
    lay, rec, drafts, A, S0 = _m2_setup(h, T)
    S = lay.S.copy()
    cur0 = lay.cursor()[0, 1]
    lay.verify_tree(drafts, T, parents)
    lay.commit_path([path])
    for node in path:
        S, _ = mamba2_step(S, *(drafts[k][:, node].astype(np.float64) for k in ("x", "dt")), A.astype(np.float64),
                           drafts["B"][:, node].astype(np.float64), drafts["C"][:, node].astype(np.float64))
    close(lay.S, S, tol=1e-13)
    assert lay.cursor()[0, 1] == cur0 + len(path)


def test_commit_path_rejects_a_non_path():
    lay, rec, drafts, A, S0 = _m2_setup(1, 4)
    lay.verify_tree(drafts, 4, [-1, -1, 0, 1])
    with pytest.raises(ValueError):
        lay.commit_path([[0, 3]])        # 3's parent is 1, not 0
    lay2, rec, drafts, A, S0 = _m2_setup(1, 4)
    lay2.verify_tree(drafts, 4, [-1, -1, 0, 1])
    with pytest.raises(RuntimeError):
        lay2.commit([2])                 # prefix commit of a non-chain tree
