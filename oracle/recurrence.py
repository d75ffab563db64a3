"""Conventional per-token SSM recurrences in float64 (test infrastructure only).

Both functions take a batch of sequences and return the updated state and the
output of this token.  They are the plain definitions that ReplaySSM must
reproduce "up to floating-point differences" ([richland] What shipped, the
paragraph on unrolling the recurrence; [ai-jitan] ReplaySSMは何をする手法か).
"""

from __future__ import annotations

import numpy as np


def group_of_head(n_heads: int, n_groups: int) -> np.ndarray:
    """Group (Mamba-2 B/C group, GDN key head) used by each head: floor(h * G / H)."""
    return (np.arange(n_heads) * n_groups) // n_heads


def mamba2_step(S, x, dt, A, Bm, Cm):
    """One Mamba-2 decode token, conventional form.

    S_t = a_t S_{t-1} + v_t k_t^T and y_t = S_t q_t, per head, with
    a_t = exp(dt_t A_h), v_t = dt_t x_t, k_t = B_t and q_t = C_t of the head's
    group ([richland] What shipped: "the Mamba-2 update S_t = α_t S_{t-1} + v_t k_t^T";
    the per-token read-update-write of the conventional decoder).

    S  [b][H][P][N] float64     x  [b][H][P]      dt [b][H]
    A  [H]                      Bm, Cm [b][G][N]
    Returns (S_t, y_t) with y_t [b][H][P].
    """
    H = S.shape[1]
    G = Bm.shape[1]
    grp = group_of_head(H, G)
    a = np.exp(dt * A[None, :])                      # [b][H]
    v = dt[:, :, None] * x                           # [b][H][P]
    k = Bm[:, grp, :]                                # [b][H][N]
    q = Cm[:, grp, :]                                # [b][H][N]
    S_new = a[:, :, None, None] * S + v[:, :, :, None] * k[:, :, None, :]
    y = np.einsum("bhpn,bhn->bhp", S_new, q)
    return S_new, y


def gdn_step(S, q, k, v, g, beta):
    """One Gated DeltaNet decode token, conventional form.

    S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T and o_t = S_t q_t, per
    value head, with a_t = exp(g_t) and b_t = beta_t; q and k come from the
    head's key head.  S_{t-1}(I - b k k^T) is expanded as S_{t-1} - b (S_{t-1} k) k^T.

    S  [b][Hv][dv][dk] float64   q, k [b][Hk][dk]   v [b][Hv][dv]
    g, beta [b][Hv]
    Returns (S_t, o_t) with o_t [b][Hv][dv].
    """
    Hv = S.shape[1]
    Hk = k.shape[1]
    kh = group_of_head(Hv, Hk)
    a = np.exp(g)[:, :, None, None]
    b = beta[:, :, None, None]
    kk = k[:, kh, :]                                 # [b][Hv][dk]
    qq = q[:, kh, :]
    Sk = np.einsum("bhvk,bhk->bhv", S, kk)           # S_{t-1} k
    S_new = a * (S - b * Sk[:, :, :, None] * kk[:, :, None, :]) + b * v[:, :, :, None] * kk[:, :, None, :]
    o = np.einsum("bhvk,bhk->bhv", S_new, qq)
    return S_new, o


def gdn_delta(S, k, v, g, beta):
    """The delta record of one Gated DeltaNet token: u_t = b_t (v_t - a_t S_{t-1} k_t).

    Expanding the gated delta rule gives S_t = a_t S_{t-1} + u_t k_t^T, so u_t is
    the value-side vector a ring record must hold for the unrolled form to
    reproduce S_t ([warp-studio] 推測デコーディングにおける革新と実装詳細: the
    buffered records "(d, k, g)", read as d = u).  Computed here from the
    step-by-step state S_{t-1}, not from the unrolled form.

    S  [b][Hv][dv][dk] float64 (the state before the token)
    k [b][Hk][dk]   v [b][Hv][dv]   g, beta [b][Hv]
    Returns u [b][Hv][dv].
    """
    Hv = S.shape[1]
    kh = group_of_head(Hv, k.shape[1])
    kk = k[:, kh, :]
    Sk = np.einsum("bhvk,bhk->bhv", S, kk)
    return beta[:, :, None] * (v - np.exp(g)[:, :, None] * Sk)


def kda_step(S, q, k, v, g, beta):
    """One token of the delta rule with a per-channel gate (the gate form of Kimi
    Delta Attention), conventional form.

    S_t = S_{t-1} Diag(a_t) (I - b_t k_t k_t^T) + b_t v_t k_t^T and o_t = S_t q_t,
    per value head, with a_t = exp(g_t) a vector over the key channels (Gated
    DeltaNet is the case of equal channels).  The pages note that the method
    generalises to this rule ([richland] Why it matters) without writing it; the
    channel-wise form here is the plainest one: the scalar decay of the gated delta
    rule becomes a diagonal matrix on the key side.
    S_{t-1} Diag(a)(I - b k k^T) is expanded as S' - b (S' k) k^T with S' = S_{t-1} Diag(a).

    S  [b][Hv][dv][dk] float64   q, k [b][Hk][dk]   v [b][Hv][dv]
    g  [b][Hv][dk] (log decay per key channel)   beta [b][Hv]
    Returns (S_t, o_t) with o_t [b][Hv][dv].
    """
    Hv = S.shape[1]
    kh = group_of_head(Hv, k.shape[1])
    kk = k[:, kh, :]
    qq = q[:, kh, :]
    b = beta[:, :, None, None]
    Sd = S * np.exp(g)[:, :, None, :]                   # S_{t-1} Diag(a)
    Sk = np.einsum("bhvk,bhk->bhv", Sd, kk)
    S_new = Sd - b * Sk[:, :, :, None] * kk[:, :, None, :] + b * v[:, :, :, None] * kk[:, :, None, :]
    o = np.einsum("bhvk,bhk->bhv", S_new, qq)
    return S_new, o


def kda_delta(S, k, v, g, beta):
    """The delta record of one per-channel-gated token: u_t = b_t (v_t - S_{t-1} (a_t * k_t)),
    so that S_t = S_{t-1} Diag(a_t) + u_t k_t^T (shapes as kda_step)."""
    Hv = S.shape[1]
    kk = k[:, group_of_head(Hv, k.shape[1]), :]
    Sk = np.einsum("bhvk,bhk->bhv", S, np.exp(g) * kk)
    return beta[:, :, None] * (v - Sk)
