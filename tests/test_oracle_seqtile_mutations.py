"""Mutation test for the sequence-tiled oracle (oracle/seqtile_ref.py): plausible mistakes are
planted in its helpers, one at a time, and each must make at least one of the pins in
tests/test_oracle_seqtile.py fail. This shows the pins constrain every part of the loss and
MLP arithmetic, not only the parts a single check happens to touch."""
import numpy as np
import pytest

import oracle.seqtile_ref as ref
import tests.test_oracle_seqtile as pins


def _all_pins():
    for name in dir(pins):
        if name.startswith("test_"):
            yield name, getattr(pins, name)


# ---- loss mutants -----------------------------------------------------------------------

def _stats_loss_sign(logits, tgt):
    lse, loss = _orig_row_stats(logits, tgt)
    return lse, np.where(tgt >= 0, -loss, 0.0)


def _stats_target_off_by_one(logits, tgt):
    m = logits.max(axis=1)
    lse = m + np.log(np.exp(logits - m[:, None]).sum(axis=1))
    t1 = np.clip(tgt + 1, 0, logits.shape[1] - 1)
    picked = logits[np.arange(len(tgt)), t1]
    return lse, np.where(tgt >= 0, lse - picked, 0.0)


def _stats_ignored_counted(logits, tgt):
    m = logits.max(axis=1)
    lse = m + np.log(np.exp(logits - m[:, None]).sum(axis=1))
    picked = logits[np.arange(len(tgt)), np.maximum(tgt, 0)]
    return lse, lse - picked


def _stats_log2(logits, tgt):
    m = logits.max(axis=1)
    lse = m + np.log2(np.exp(logits - m[:, None]).sum(axis=1))
    valid = tgt >= 0
    picked = np.where(valid, logits[np.arange(len(tgt)), np.where(valid, tgt, 0)], 0.0)
    return lse, np.where(valid, lse - picked, 0.0)


def _dl_no_onehot(logits, lse, tgt, G):
    p = np.exp(logits - lse[:, None])
    return p * np.where(tgt >= 0, G, 0.0)[:, None]


def _dl_sign(logits, lse, tgt, G):
    return -_orig_dlogits(logits, lse, tgt, G)


def _dl_ignores_g(logits, lse, tgt, G):
    return _orig_dlogits(logits, lse, tgt, np.ones_like(G))


def _dl_ignored_rows_kept(logits, lse, tgt, G):
    p = np.exp(logits - lse[:, None])
    rows = np.nonzero(tgt >= 0)[0]
    p[rows, tgt[rows]] -= 1.0
    return p * G[:, None]


# ---- MLP mutants ------------------------------------------------------------------------

def _silu_wrong_derivative(z):
    s = 1.0 / (1.0 + np.exp(-np.clip(z, -700, 700)))
    return z * s, s * (1.0 + z)


def _silu_is_sigmoid(z):
    s = 1.0 / (1.0 + np.exp(-np.clip(z, -700, 700)))
    return s, s * (1.0 - s)


def _mlp_gate_up_swapped(X, Wgu, Wd, dY):
    F = Wd.shape[1]
    Wsw = np.concatenate([Wgu[F:], Wgu[:F]], axis=0)
    return _orig_mlp_rows(X, Wsw, Wd, dY)


def _mlp_dx_gate_path_only(X, Wgu, Wd, dY):
    y, dx, dgu, a = _orig_mlp_rows(X, Wgu, Wd, dY)
    if dY is None:
        return y, dx, dgu, a
    F = Wd.shape[1]
    return y, dgu[:, :F] @ Wgu[:F], dgu, a


def _mlp_du_uses_da(X, Wgu, Wd, dY):
    y, dx, dgu, a = _orig_mlp_rows(X, Wgu, Wd, dY)
    if dY is None:
        return y, dx, dgu, a
    F = Wd.shape[1]
    da = dY @ Wd
    dgu = np.concatenate([dgu[:, :F], da], axis=1)
    return y, dgu @ Wgu, dgu, a


_orig_row_stats = ref._row_stats
_orig_dlogits = ref._dlogits
_orig_mlp_rows = ref._mlp_rows

MUTANTS = [
    ("loss_sign_flipped", "_row_stats", _stats_loss_sign),
    ("target_off_by_one", "_row_stats", _stats_target_off_by_one),
    ("ignored_token_counted", "_row_stats", _stats_ignored_counted),
    ("lse_in_log2", "_row_stats", _stats_log2),
    ("dlogits_without_onehot", "_dlogits", _dl_no_onehot),
    ("dlogits_sign_flipped", "_dlogits", _dl_sign),
    ("dlogits_ignores_upstream_gradient", "_dlogits", _dl_ignores_g),
    ("dlogits_keeps_ignored_rows", "_dlogits", _dl_ignored_rows_kept),
    ("silu_derivative_missing_factor", "_silu_parts", _silu_wrong_derivative),
    ("silu_replaced_by_sigmoid", "_silu_parts", _silu_is_sigmoid),
    ("gate_and_up_swapped", "_mlp_rows", _mlp_gate_up_swapped),
    ("dx_without_up_path", "_mlp_rows", _mlp_dx_gate_path_only),
    ("du_without_silu", "_mlp_rows", _mlp_du_uses_da),
]


@pytest.mark.parametrize("name,attr,mutant", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistakes(monkeypatch, name, attr, mutant):
    monkeypatch.setattr(ref, attr, mutant)
    failed = []
    for pin, fn in _all_pins():
        try:
            with np.errstate(all="ignore"):
                fn()
        except (AssertionError, ValueError, FloatingPointError, IndexError):
            failed.append(pin)
    assert failed, f"planted mistake {name} passed every pin"


def test_unmutated_oracle_passes_every_pin():
    for pin, fn in _all_pins():
        fn()
