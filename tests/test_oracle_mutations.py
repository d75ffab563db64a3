"""The pins must catch plausible oracle mistakes.

Each case plants one mistake in a copy of an oracle recurrence (on the CPU),
installs it where the pins look it up, and checks that at least one pin of
tests/test_oracle_pins.py fails.
"""

import numpy as np
import pytest

import oracle.layer as layer_mod
import tests.test_oracle_pins as pins
from oracle.recurrence import group_of_head


def m2_output_before_update(S, x, dt, A, Bm, Cm):
    grp = group_of_head(S.shape[1], Bm.shape[1])
    a = np.exp(dt * A[None, :])
    y = np.einsum("bhpn,bhn->bhp", S, Cm[:, grp, :])
    S_new = a[:, :, None, None] * S + (dt[:, :, None] * x)[:, :, :, None] * Bm[:, grp, None, :]
    return S_new, y


def m2_no_decay(S, x, dt, A, Bm, Cm):
    grp = group_of_head(S.shape[1], Bm.shape[1])
    S_new = S + (dt[:, :, None] * x)[:, :, :, None] * Bm[:, grp, None, :]
    return S_new, np.einsum("bhpn,bhn->bhp", S_new, Cm[:, grp, :])


def m2_decay_on_update(S, x, dt, A, Bm, Cm):
    grp = group_of_head(S.shape[1], Bm.shape[1])
    a = np.exp(dt * A[None, :])
    S_new = a[:, :, None, None] * (S + (dt[:, :, None] * x)[:, :, :, None] * Bm[:, grp, None, :])
    return S_new, np.einsum("bhpn,bhn->bhp", S_new, Cm[:, grp, :])


def m2_swapped_bc(S, x, dt, A, Bm, Cm):
    grp = group_of_head(S.shape[1], Bm.shape[1])
    a = np.exp(dt * A[None, :])
    S_new = a[:, :, None, None] * S + (dt[:, :, None] * x)[:, :, :, None] * Cm[:, grp, None, :]
    return S_new, np.einsum("bhpn,bhn->bhp", S_new, Bm[:, grp, :])


def m2_wrong_group(S, x, dt, A, Bm, Cm):
    H, G = S.shape[1], Bm.shape[1]
    grp = np.arange(H) % G
    a = np.exp(dt * A[None, :])
    S_new = a[:, :, None, None] * S + (dt[:, :, None] * x)[:, :, :, None] * Bm[:, grp, None, :]
    return S_new, np.einsum("bhpn,bhn->bhp", S_new, Cm[:, grp, :])


def m2_v_without_dt(S, x, dt, A, Bm, Cm):
    grp = group_of_head(S.shape[1], Bm.shape[1])
    a = np.exp(dt * A[None, :])
    S_new = a[:, :, None, None] * S + x[:, :, :, None] * Bm[:, grp, None, :]
    return S_new, np.einsum("bhpn,bhn->bhp", S_new, Cm[:, grp, :])


def _gdn(variant):
    def step(S, q, k, v, g, beta):
        kh = group_of_head(S.shape[1], k.shape[1])
        a = np.exp(g)[:, :, None, None]
        b = beta[:, :, None, None]
        kk, qq = k[:, kh, :], q[:, kh, :]
        Sk = np.einsum("bhvk,bhk->bhv", S, kk)
        outer_vk = v[:, :, :, None] * kk[:, :, None, :]
        if variant == "plus_erase":
            S_new = a * (S + b * Sk[..., None] * kk[:, :, None, :]) + b * outer_vk
        elif variant == "left_projection":
            kS = np.einsum("bhk,bhkv->bhv", kk, S)          # k^T S instead of S k
            S_new = a * (S - b * kk[:, :, :, None] * kS[:, :, None, :]) + b * outer_vk
        elif variant == "erase_without_beta":
            S_new = a * (S - Sk[..., None] * kk[:, :, None, :]) + b * outer_vk
        elif variant == "decay_on_write":
            S_new = a * (S - b * Sk[..., None] * kk[:, :, None, :] + b * outer_vk)
        o = np.einsum("bhvk,bhk->bhv", S_new, qq)
        return S_new, o
    return step


M2_PINS = ["test_mamba2_dyadic_hand_values", "test_mamba2_geometric_series",
           "test_mamba2_unit_decay_is_prefix_sum", "test_mamba2_group_mapping",
           "test_mamba2_unrolled_identity", "test_mamba2_chunkwise_verify_matches_oracle",
           "test_commit_advances_by_accepted_prefix"]
GDN_PINS = ["test_gdn_dyadic_hand_values", "test_gdn_zero_beta_is_pure_decay",
            "test_gdn_delta_rule_writes_value_at_key", "test_gdn_general_step_along_and_across_key",
            "test_gdn_from_zero_state", "test_gdn_delta_form",
            "test_gdn_chunkwise_verify_with_triangular_solve"]


def _some_pin_fails(names) -> bool:
    for name in names:
        try:
            getattr(pins, name)()
        except (AssertionError, np.linalg.LinAlgError):
            return True
    return False


@pytest.mark.parametrize("bad", [m2_output_before_update, m2_no_decay, m2_decay_on_update,
                                 m2_swapped_bc, m2_wrong_group, m2_v_without_dt])
def test_mamba2_mistake_is_caught(monkeypatch, bad):
    monkeypatch.setattr(pins, "mamba2_step", bad)
    monkeypatch.setattr(layer_mod, "mamba2_step", bad)
    assert _some_pin_fails(M2_PINS)


@pytest.mark.parametrize("variant", ["plus_erase", "left_projection", "erase_without_beta", "decay_on_write"])
def test_gdn_mistake_is_caught(monkeypatch, variant):
    bad = _gdn(variant)
    monkeypatch.setattr(pins, "gdn_step", bad)
    monkeypatch.setattr(layer_mod, "gdn_step", bad)
    assert _some_pin_fails(GDN_PINS)


# --- read-copy branch of OracleLayer ------------------------------------------

import tests.test_oracle_readcopy_pins as rc_pins  # noqa: E402
from oracle.layer import OracleLayer, _wide  # noqa: E402


class _DecayOffByOne(OracleLayer):
    """Mistake: the copy error is decayed by the records before this token only
    (the current token's decay left out of the sum)."""

    def decode(self, inp):
        tok = _wide(inp)
        S_prev_ckpt = self.ckpt.copy()
        before = self.logdecay.copy()
        self.S, y, ld = self._token(self.S, tok)
        self.logdecay += ld
        grp = (np.arange(self.shape.n_heads) * self.shape.n_groups) // self.shape.n_heads
        err = np.einsum("bhpn,bhn->bhp", self.read_copy - S_prev_ckpt, tok["C"][:, grp, :])
        self.last_read_out = y + np.exp(before)[:, :, None] * err
        for i, r in enumerate(self.rings):
            if r.decode():
                self.ckpt[i] = self.S[i]
                self.logdecay[i] = 0.0
                self.last_read_out[i] = y[i]
                self._refresh_read_copy(i)
        return y


class _StaleCopy(OracleLayer):
    """Mistake: a fold re-quantises the copy from the checkpoint as it was before the fold."""

    def _refresh_read_copy(self, i):
        if self.read_mode is None:
            return
        old = getattr(self, "_ckpt_before", None)
        if old is None:
            return super()._refresh_read_copy(i)
        keep = self.ckpt[i].copy()
        self.ckpt[i] = old[i]
        super()._refresh_read_copy(i)
        self.ckpt[i] = keep

    def decode(self, inp):
        self._ckpt_before = self.ckpt.copy()
        return super().decode(inp)

    def commit(self, accepted):
        self._ckpt_before = self.ckpt.copy()
        return super().commit(accepted)


RC_PINS = ["test_fp8_read_copy_dyadic_hand_values"]


def _rc_pin_fails() -> bool:
    cases = [lambda: rc_pins.test_fp8_read_copy_dyadic_hand_values()]
    for mode in ("fp8", "nvfp4"):
        cases.append(lambda m=mode: rc_pins.test_read_copy_output_equals_recurrence_restarted_from_the_copy(m))
        cases.append(lambda m=mode: rc_pins.test_read_copy_output_after_commits_equals_restarted_recurrence(m))
    failed = 0
    for c in cases:
        try:
            c()
        except AssertionError:
            failed += 1
    return failed > 0


@pytest.mark.parametrize("bad", [_DecayOffByOne, _StaleCopy])
def test_read_copy_mistake_is_caught(monkeypatch, bad):
    monkeypatch.setattr(rc_pins, "OracleLayer", bad)
    assert _rc_pin_fails()


def test_read_copy_pins_pass_unmutated():
    assert not _rc_pin_fails()


def _bad_delta(S, k, v, g, beta):
    """Mistake: the delta record without the decay on the erased value."""
    kh = group_of_head(S.shape[1], k.shape[1])
    Sk = np.einsum("bhvk,bhk->bhv", S, k[:, kh, :])
    return beta[:, :, None] * (v - Sk)


def test_gdn_delta_mistake_is_caught(monkeypatch):
    import oracle.recurrence as rec
    monkeypatch.setattr(rec, "gdn_delta", _bad_delta)
    monkeypatch.setattr(layer_mod, "gdn_delta", _bad_delta)
    names = ["test_gdn_delta_reproduces_the_state_and_vanishes_without_write",
             "test_oracle_layer_records_draft_deltas_along_the_draft_chain"]
    failed = 0
    for n in names:
        try:
            getattr(pins, n)()
        except AssertionError:
            failed += 1
    assert failed > 0


# --- tree verify and path commit ------------------------------------------------

import tests.test_oracle_tree_pins as tree_pins  # noqa: E402


class _TreeAsChain(OracleLayer):
    """Mistake: the parents are ignored and the drafts verified as a chain."""

    def verify_tree(self, drafts, T, parents):
        Y = self.verify(drafts, T)
        self._tree = [int(p) for p in parents]
        return Y


class _PathAsPrefix(OracleLayer):
    """Mistake: a path commit advances the state by the first len(path) drafts."""

    def commit_path(self, paths):
        tok, T = self._drafts
        for i, path in enumerate(paths):
            for node in range(len(path)):
                S_new, _, ld = self._token(self.S[i:i + 1], {k: v[i:i + 1, node] for k, v in tok.items()})
                self.S[i] = S_new[0]
                self.logdecay[i] += ld[0]
        for i, r in enumerate(self.rings):
            if r.commit(len(paths[i])):
                self.ckpt[i] = self.S[i]
                self.logdecay[i] = 0.0
        self._drafts = None
        self._tree = None


def _tree_pin_fails() -> bool:
    cases = []
    for par in tree_pins.TREES:
        cases.append(lambda p=par: tree_pins.test_mamba2_tree_verify_is_the_ancestor_masked_chunkwise_form(p))
        cases.append(lambda p=par: tree_pins.test_gdn_tree_verify_is_the_ancestor_masked_triangular_solve(p))
    for par, path in [([-1, -1, 0, 1], [1, 3]), ([-1, 0, 0, 2], [0, 2, 3])]:
        cases.append(lambda p=par, q=path: tree_pins.test_commit_path_equals_plain_decode_along_the_path(p, q))
    failed = 0
    for c in cases:
        try:
            c()
        except AssertionError:
            failed += 1
    return failed > 0


@pytest.mark.parametrize("bad", [_TreeAsChain, _PathAsPrefix])
def test_tree_mistake_is_caught(monkeypatch, bad):
    monkeypatch.setattr(tree_pins, "OracleLayer", bad)
    assert _tree_pin_fails()


def test_tree_pins_pass_unmutated():
    assert not _tree_pin_fails()


def _kda(variant):
    def step(S, q, k, v, g, beta):
        kh = group_of_head(S.shape[1], k.shape[1])
        kk, qq = k[:, kh, :], q[:, kh, :]
        b = beta[:, :, None, None]
        a = np.exp(g)
        if variant == "erase_before_decay":      # S (I - b k k^T) Diag(a): the order swapped
            Sk = np.einsum("bhvk,bhk->bhv", S, kk)
            S_new = (S - b * Sk[..., None] * kk[:, :, None, :]) * a[:, :, None, :] + b * v[..., None] * kk[:, :, None, :]
        else:                                    # decay on the value side: Diag(a) applied to rows
            Sd = S * a[:, :, :, None] if a.shape[-1] == S.shape[2] else S * a[:, :, None, :]
            Sd = np.swapaxes(np.swapaxes(S, 2, 3) * a[:, :, None, :], 2, 3)
            Sk = np.einsum("bhvk,bhk->bhv", Sd, kk)
            S_new = Sd - b * Sk[..., None] * kk[:, :, None, :] + b * v[..., None] * kk[:, :, None, :]
        return S_new, np.einsum("bhvk,bhk->bhv", S_new, qq)
    return step


@pytest.mark.parametrize("variant", ["erase_before_decay", "decay_on_value_side"])
def test_kda_mistake_is_caught(monkeypatch, variant):
    import oracle.recurrence as rec
    bad = _kda(variant)
    monkeypatch.setattr(rec, "kda_step", bad)
    names = ["test_kda_dyadic_hand_values", "test_kda_with_equal_channels_is_gated_deltanet",
             "test_kda_without_write_is_per_channel_decay", "test_kda_unrolled_identity"]
    failed = 0
    for n in names:
        try:
            getattr(pins, n)()
        except AssertionError:
            failed += 1
    assert failed > 0
