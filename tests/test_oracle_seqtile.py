"""Pins for the fp64 sequence-tiled loss oracle (oracle/seqtile_ref.py) against things fixed
by the mathematics, not by the oracle's own formula: finite differences, closed forms, the
two-class (logistic) special case, scipy's logsumexp, and invariants of softmax
cross-entropy. A dropped term, a wrong sign, a transposed operand or a mis-indexed target
fails at least one of them."""
import math

import numpy as np
import pytest

from oracle.seqtile_ref import ce_loss_bwd_ref, ce_loss_ref, ce_rows_ref


def _problem(rng, S, Dm, V, ignore=()):
    h = rng.standard_normal((S, Dm))
    w = rng.standard_normal((V, Dm)) * 0.7
    t = rng.integers(0, V, size=S)
    for i in ignore:
        t[i] = -1
    g = rng.standard_normal(S)
    return h, w, t, g


def test_finite_differences_of_weighted_loss():
    # d/dx sum_i g_i loss_i by central differences, for every entry of h and w
    rng = np.random.default_rng(11)
    S, Dm, V = 5, 4, 7
    h, w, t, g = _problem(rng, S, Dm, V, ignore=(3,))
    _, _, dh, dw = ce_loss_bwd_ref(h, w, t, g)

    def f(hh, ww):
        return float(np.dot(g, ce_loss_ref(hh, ww, t)[0]))

    eps = 1e-6
    num_dh = np.zeros_like(h)
    for idx in np.ndindex(*h.shape):
        hp, hm = h.copy(), h.copy()
        hp[idx] += eps
        hm[idx] -= eps
        num_dh[idx] = (f(hp, w) - f(hm, w)) / (2 * eps)
    num_dw = np.zeros_like(w)
    for idx in np.ndindex(*w.shape):
        wp, wm = w.copy(), w.copy()
        wp[idx] += eps
        wm[idx] -= eps
        num_dw[idx] = (f(h, wp) - f(h, wm)) / (2 * eps)
    assert np.abs(num_dh - dh).max() <= 1e-6 * max(1.0, np.abs(dh).max())
    assert np.abs(num_dw - dw).max() <= 1e-6 * max(1.0, np.abs(dw).max())
    assert np.all(dh[3] == 0.0)  # the ignored token takes no gradient


def test_zero_readout_closed_form():
    # w = 0: every logit is 0, so lse = loss = ln V; dlogits = g (1/V - onehot)
    rng = np.random.default_rng(2)
    S, Dm, V = 9, 6, 13
    h, _, t, g = _problem(rng, S, Dm, V, ignore=(0,))
    w = np.zeros((V, Dm))
    loss, lse, dh, dw = ce_loss_bwd_ref(h, w, t, g)
    assert np.allclose(lse, math.log(V), rtol=0, atol=1e-15)
    assert loss[0] == 0.0 and np.allclose(loss[1:], math.log(V), rtol=0, atol=1e-15)
    assert np.all(dh == 0.0)
    want = np.zeros((V, Dm))
    for i in range(1, S):
        want += g[i] * (1.0 / V) * h[i]
        want[t[i]] -= g[i] * h[i]
    assert np.allclose(dw, want, rtol=0, atol=1e-13)


def test_scaled_identity_closed_form():
    # Dm = V, w = a I, h_i = e_{c_i}: row i's logits are a at c_i and 0 elsewhere, so
    # lse = ln(e^a + V - 1), loss = lse - a when the target is c_i, lse otherwise
    V, a = 6, 2.5
    c = np.array([0, 3, 5, 3, 1])
    h = np.eye(V)[c]
    w = a * np.eye(V)
    t = np.array([0, 2, 5, 3, 4])
    loss, lse = ce_loss_ref(h, w, t)
    L = math.log(math.exp(a) + V - 1)
    assert np.allclose(lse, L, rtol=0, atol=1e-14)
    want = np.where(t == c, L - a, L)
    assert np.allclose(loss, want, rtol=0, atol=1e-14)


def test_two_classes_is_logistic_loss():
    # V = 2: loss = log(1 + exp(l_other - l_target)) (the textbook logistic loss), and its
    # derivative wrt l_target is -sigmoid(l_other - l_target)
    rng = np.random.default_rng(5)
    S, Dm = 40, 3
    h, w, t, g = _problem(rng, S, Dm, 2)
    loss, _, dh, _ = ce_loss_bwd_ref(h, w, t, g)
    lg = h @ w.T
    z = lg[np.arange(S), 1 - t] - lg[np.arange(S), t]
    assert np.allclose(loss, np.log1p(np.exp(z)), rtol=1e-13, atol=1e-15)
    sig = 1.0 / (1.0 + np.exp(-z))
    # dlogits: +g sig on the other class, -g sig on the target
    want_dh = (g * sig)[:, None] * (w[1 - t] - w[t])
    assert np.allclose(dh, want_dh, rtol=1e-12, atol=1e-14)


def test_lse_matches_scipy_logsumexp():
    special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(7)
    h, w, t, _ = _problem(rng, 33, 16, 300)
    h *= 4.0  # logits of a few tens: the max shift matters
    _, lse = ce_loss_ref(h, w, t, block=8)
    assert np.allclose(lse, special.logsumexp(h @ w.T, axis=1), rtol=1e-14, atol=1e-12)


def test_common_shift_of_vocabulary_rows():
    # adding the same vector c to every w_j shifts row i's logits by the constant <h_i, c>:
    # the loss and the gradient of h stay, lse moves by <h_i, c>
    rng = np.random.default_rng(9)
    h, w, t, g = _problem(rng, 12, 5, 17, ignore=(4,))
    c = rng.standard_normal(5)
    l0, s0, dh0, _ = ce_loss_bwd_ref(h, w, t, g)
    l1, s1, dh1, _ = ce_loss_bwd_ref(h, w + c, t, g)
    assert np.allclose(l0, l1, rtol=0, atol=1e-12)
    assert np.allclose(s1 - s0, h @ c, rtol=0, atol=1e-12)
    # dh = sum_j dlogits_ij (w_j + c) = dh0 + c * sum_j dlogits_ij = dh0
    assert np.allclose(dh0, dh1, rtol=0, atol=1e-12)


def test_vocabulary_sum_of_dw_vanishes_and_ignored_rows_drop_out():
    rng = np.random.default_rng(13)
    S, Dm, V = 30, 8, 50
    ign = (2, 7, 29)
    h, w, t, g = _problem(rng, S, Dm, V, ignore=ign)
    _, _, dh, dw = ce_loss_bwd_ref(h, w, t, g, block=7)
    # each valid row of dlogits sums to g_i (1 - 1) = 0, so the rows of dw sum to 0
    assert np.abs(dw.sum(axis=0)).max() <= 1e-12 * np.abs(dw).max()
    keep = np.array([i for i in range(S) if i not in ign])
    _, _, dh_k, dw_k = ce_loss_bwd_ref(h[keep], w, t[keep], g[keep])
    assert np.allclose(dw, dw_k, rtol=0, atol=1e-12)
    assert np.allclose(dh[keep], dh_k, rtol=0, atol=1e-12)
    assert np.all(dh[list(ign)] == 0.0)


def test_blocking_and_sampled_rows_agree_with_whole_problem():
    rng = np.random.default_rng(17)
    h, w, t, g = _problem(rng, 70, 8, 40, ignore=(10,))
    a = ce_loss_bwd_ref(h, w, t, g, block=1)
    b = ce_loss_bwd_ref(h, w, t, g, block=1000)
    for x, y in zip(a, b):
        assert np.allclose(x, y, rtol=0, atol=1e-12)
    rows = np.array([0, 10, 33, 69])
    loss, lse, dh = ce_rows_ref(h, w, t, g, rows)
    assert np.allclose(loss, b[0][rows], rtol=0, atol=1e-13)
    assert np.allclose(lse, b[1][rows], rtol=0, atol=1e-13)
    assert np.allclose(dh, b[2][rows], rtol=0, atol=1e-13)
    # with g zero off the sampled rows, their share of dw is all of dw
    gs = np.zeros_like(g)
    gs[rows] = g[rows]
    vr = [0, 5, 17, 39]
    _, _, _, dw_full = ce_loss_bwd_ref(h, w, t, gs)
    _, _, _, dw_part = ce_rows_ref(h, w, t, gs, rows, vocab_rows=vr)
    assert np.allclose(dw_part, dw_full[vr], rtol=0, atol=1e-13)


# ---- gated (SwiGLU) MLP ---------------------------------------------------------------------

from oracle.seqtile_ref import mlp_bwd_ref, mlp_ref, mlp_rows_ref  # noqa: E402


def _mlp_problem(rng, S, Dm, F):
    x = rng.standard_normal((S, Dm))
    w_gu = rng.standard_normal((2 * F, Dm)) * 0.6
    w_d = rng.standard_normal((Dm, F)) * 0.6
    dy = rng.standard_normal((S, Dm))
    return x, w_gu, w_d, dy


def test_mlp_finite_differences():
    rng = np.random.default_rng(21)
    S, Dm, F = 3, 4, 5
    x, w_gu, w_d, dy = _mlp_problem(rng, S, Dm, F)
    _, dx, dw_gu, dw_d = mlp_bwd_ref(x, w_gu, w_d, dy)

    def f(xx, gg, dd):
        return float(np.sum(dy * mlp_ref(xx, gg, dd)))

    eps = 1e-6
    for arr, grad, which in ((x, dx, 0), (w_gu, dw_gu, 1), (w_d, dw_d, 2)):
        num = np.zeros_like(arr)
        for idx in np.ndindex(*arr.shape):
            p, m = arr.copy(), arr.copy()
            p[idx] += eps
            m[idx] -= eps
            args_p = [x, w_gu, w_d]
            args_m = [x, w_gu, w_d]
            args_p[which], args_m[which] = p, m
            num[idx] = (f(*args_p) - f(*args_m)) / (2 * eps)
        assert np.abs(num - grad).max() <= 1e-6 * max(1.0, np.abs(grad).max()), which


def test_mlp_matches_torch_autograd():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(23)
    x, w_gu, w_d, dy = _mlp_problem(rng, 17, 12, 9)
    y, dx, dw_gu, dw_d = mlp_bwd_ref(x, w_gu, w_d, dy, block=5)
    X = torch.tensor(x, requires_grad=True)
    G = torch.tensor(w_gu, requires_grad=True)
    D = torch.tensor(w_d, requires_grad=True)
    F = w_d.shape[1]
    h = X @ G.T
    Y = (torch.nn.functional.silu(h[:, :F]) * h[:, F:]) @ D.T
    Y.backward(torch.tensor(dy))
    assert np.allclose(y, Y.detach().numpy(), rtol=1e-12, atol=1e-12)
    assert np.allclose(dx, X.grad.numpy(), rtol=1e-12, atol=1e-12)
    assert np.allclose(dw_gu, G.grad.numpy(), rtol=1e-12, atol=1e-12)
    assert np.allclose(dw_d, D.grad.numpy(), rtol=1e-12, atol=1e-12)


def test_mlp_closed_forms():
    # gate weights zero: g = 0, silu(0) = 0, so y = 0; silu'(0) = 1/2, so dg = da*u/2, du = 0
    rng = np.random.default_rng(25)
    S, Dm, F = 6, 5, 4
    x, w_gu, w_d, dy = _mlp_problem(rng, S, Dm, F)
    w_gu[:F] = 0.0
    y, dx, dw_gu, dw_d = mlp_bwd_ref(x, w_gu, w_d, dy)
    assert np.all(y == 0.0) and np.all(dw_d == 0.0)
    u = x @ w_gu[F:].T
    da = dy @ w_d
    assert np.allclose(dw_gu[:F], (0.5 * da * u).T @ x, rtol=0, atol=1e-12)
    assert np.all(dw_gu[F:] == 0.0)
    # huge positive gate: silu(g) -> g, so y -> ((x Wg^T) * (x Wu^T)) Wd^T
    x2, w2, d2, _ = _mlp_problem(rng, 4, 3, 2)
    w2[:2] = np.abs(w2[:2]) * 1e3
    x2 = np.abs(x2)
    g = x2 @ w2[:2].T
    want = (g * (x2 @ w2[2:].T)) @ d2.T
    assert np.allclose(mlp_ref(x2, w2, d2), want, rtol=1e-12, atol=0)


def test_silu_matches_logistic_and_is_stable():
    special = pytest.importorskip("scipy.special")
    from oracle.seqtile_ref import _silu_parts
    z = np.linspace(-800.0, 800.0, 4001)
    s, ds = _silu_parts(z)
    assert np.all(np.isfinite(s)) and np.all(np.isfinite(ds))
    assert np.allclose(s, z * special.expit(z), rtol=1e-14, atol=1e-300)
    h = 1e-6
    zz = np.linspace(-20, 20, 81)
    num = (_silu_parts(zz + h)[0] - _silu_parts(zz - h)[0]) / (2 * h)
    assert np.allclose(_silu_parts(zz)[1], num, rtol=1e-7, atol=1e-9)


def test_mlp_rows_and_blocking_agree_with_whole_problem():
    rng = np.random.default_rng(27)
    x, w_gu, w_d, dy = _mlp_problem(rng, 40, 6, 5)
    a = mlp_bwd_ref(x, w_gu, w_d, dy, block=3)
    b = mlp_bwd_ref(x, w_gu, w_d, dy, block=100)
    for p, q in zip(a, b):
        assert np.allclose(p, q, rtol=0, atol=1e-12)
    rows = [0, 7, 39]
    y, dx = mlp_rows_ref(x, w_gu, w_d, dy, rows)
    assert np.allclose(y, b[0][rows], rtol=0, atol=1e-13)
    assert np.allclose(dx, b[1][rows], rtol=0, atol=1e-13)
    dys = np.zeros_like(dy)
    dys[rows] = dy[rows]
    _, _, dwg_full, dwd_full = mlp_bwd_ref(x, w_gu, w_d, dys)
    gr, dr = [0, 3, 9], [1, 4]
    _, _, dwg, dwd = mlp_rows_ref(x, w_gu, w_d, dys, rows, gu_rows=gr, d_rows=dr)
    assert np.allclose(dwg, dwg_full[gr], rtol=0, atol=1e-12)
    assert np.allclose(dwd, dwd_full[dr], rtol=0, atol=1e-12)


# ---- hand-worked examples (tests/golden/, derivations in each file's "_about") --------------

import json  # noqa: E402
import os  # noqa: E402

_GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_loss_hand_worked_example():
    e = json.load(open(os.path.join(_GOLDEN, "ce_hand_example_s2_v2.json")))
    loss, lse, dh, dw = ce_loss_bwd_ref(np.array(e["h"]), np.array(e["w"]),
                                        np.array(e["target"]), np.array(e["g"]))
    assert np.allclose(loss, e["loss"], rtol=0, atol=1e-14)
    assert np.allclose(lse, e["lse"], rtol=0, atol=1e-14)
    assert np.allclose(dh, e["dh"], rtol=0, atol=1e-14)
    assert np.allclose(dw, e["dw"], rtol=0, atol=1e-14)


def test_mlp_hand_worked_example():
    e = json.load(open(os.path.join(_GOLDEN, "mlp_hand_example_d1_f1.json")))
    y, dx, dw_gu, dw_d = mlp_bwd_ref(np.array(e["x"]), np.array(e["w_gu"]), np.array(e["w_d"]),
                                     np.array(e["dy"]))
    assert np.allclose(y, e["y"], rtol=0, atol=1e-13)
    assert np.allclose(dx, e["dx"], rtol=0, atol=1e-13)
    assert np.allclose(dw_gu, e["dw_gu"], rtol=0, atol=1e-13)
    assert np.allclose(dw_d, e["dw_d"], rtol=0, atol=1e-13)
