"""Pins for the fp64 oracle (CPU only, no GPU).

The oracle is checked against things other than itself: a hand-worked example, central finite
differences of its own forward, closed forms (Q = 0 gives prefix means), invariants (rows of P
sum to 1, constant V, the first causal row, GQA = MHA with repeated K/V heads), a scalar
brute-force restatement, torch's fp64 scaled_dot_product_attention as a library special case,
and the exactness of the trunked / head-chunked schedule. A mutation test plants plausible
mistakes in the oracle and checks that the pins catch each one.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle.attn_ref as ref
from workloads import random_small

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _np(t):
    return t.detach().cpu().numpy().astype(np.float64)


# ---------------------------------------------------------------------------------------
# checkers (each returns normally on success, raises AssertionError on a mismatch)
# ---------------------------------------------------------------------------------------

def check_hand_example():
    g = json.load(open(os.path.join(GOLDEN, "hand_example_s2_d1.json")))
    q = np.array(g["q"]).reshape(1, 2, 1, 1)
    k = np.array(g["k"]).reshape(1, 2, 1, 1)
    v = np.array(g["v"]).reshape(1, 2, 1, 1)
    do = np.array(g["dout"]).reshape(1, 2, 1, 1)
    o, lse, dq, dk, dv = ref.attn_bwd_ref(q, k, v, do, causal=True)
    np.testing.assert_allclose(o.ravel(), g["o"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse.ravel(), g["lse"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dq.ravel(), g["dq"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk.ravel(), g["dk"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv.ravel(), g["dv"], rtol=0, atol=1e-12)
    o2, lse2 = ref.attn_fwd_ref(q, k, v, causal=True)
    np.testing.assert_allclose(o2.ravel(), g["o"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse2.ravel(), g["lse"], rtol=0, atol=1e-12)


def check_finite_differences(causal, B=1, S=6, Hq=4, Hkv=2, D=3, seed=11):
    """<dO, dO/dx> by central differences of the oracle's own forward vs its analytic
    gradients, for every element of q, k and v (fp64, step 1e-6)."""
    q, k, v, do = (_np(t) for t in random_small(B, S, Hq, Hkv, D, seed))
    _, _, dq, dk, dv = ref.attn_bwd_ref(q, k, v, do, causal=causal)

    def loss(qq, kk, vv):
        o, _ = ref.attn_fwd_ref(qq, kk, vv, causal=causal)
        return float(np.sum(o * do))

    eps = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp = x.copy(); xp[idx] += eps
            xm = x.copy(); xm[idx] -= eps
            args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        err = np.abs(num - g).max() / max(1e-12, np.abs(g).max())
        assert err <= 1e-6, f"finite differences disagree for d{name}: rel err {err:.2e}"


def check_identity_v_rows(causal, S=7, D=8, Hq=2, Hkv=1, seed=5):
    """V = unit rows e_j (D >= S) makes O_i = P_i, the i-th row of P. Rows sum to 1, are
    non-negative, vanish above the diagonal when causal, and equal the brute-force
    exp(s_ij) / sum_j exp(s_ij) written with scalar math.exp."""
    q, k, _, _ = (_np(t) for t in random_small(1, S, Hq, Hkv, D, seed))
    v = np.zeros((1, S, Hkv, D))
    for j in range(S):
        v[0, j, :, j] = 1.0
    o, lse = ref.attn_fwd_ref(q, k, v, causal=causal)
    sc = 1.0 / math.sqrt(D)
    for h in range(Hq):
        P = o[0, :, h, :S]
        np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-13)
        assert (P >= 0).all()
        if causal:
            assert np.all(P[np.triu_indices(S, 1)] == 0.0)
        for i in range(S):
            js = range(i + 1) if causal else range(S)
            w = [math.exp(sc * sum(q[0, i, h, d] * k[0, j, h // (Hq // Hkv), d]
                                   for d in range(D))) for j in js]
            tot = sum(w)
            for j, wj in zip(js, w):
                assert abs(P[i, j] - wj / tot) <= 1e-13
            assert abs(lse[0, h, i] - math.log(tot)) <= 1e-12


def check_constant_v_and_first_row(seed=3):
    q, k, v, _ = (_np(t) for t in random_small(2, 9, 4, 2, 5, seed))
    c = np.array([0.5, -1.25, 3.0, 0.0, 2.0])
    vc = np.broadcast_to(c, v.shape).copy()
    o, _ = ref.attn_fwd_ref(q, k, vc, causal=True)
    np.testing.assert_allclose(o, np.broadcast_to(c, o.shape), rtol=0, atol=1e-13)
    o, lse = ref.attn_fwd_ref(q, k, v, causal=True)
    for h in range(4):
        np.testing.assert_allclose(o[:, 0, h, :], v[:, 0, h // 2, :], rtol=0, atol=1e-15)
        np.testing.assert_allclose(lse[:, h, 0],
                                   np.sum(q[:, 0, h, :] * k[:, 0, h // 2, :], axis=1)
                                   / math.sqrt(5), rtol=0, atol=1e-13)


def check_q_zero_closed_form(S=11, Hq=4, Hkv=2, D=6, seed=8):
    """Q = 0: every visible score is 0, so P is uniform over j <= i. Then
    O_i = mean(V_0..V_i), LSE_i = ln(i+1), dV_j = sum_{h in grp} sum_{i>=j} dO_i/(i+1),
    dK = 0, and dQ_i = scale/(i+1) * sum_{j<=i} <dO_i, v_j - O_i> k_j."""
    _, k, v, do = (_np(t) for t in random_small(1, S, Hq, Hkv, D, seed))
    q = np.zeros((1, S, Hq, D))
    o, lse, dq, dk, dv = ref.attn_bwd_ref(q, k, v, do, causal=True)
    G = Hq // Hkv
    sc = 1.0 / math.sqrt(D)
    for h in range(Hq):
        kh = h // G
        pm = np.cumsum(v[0, :, kh, :], axis=0) / np.arange(1, S + 1)[:, None]
        np.testing.assert_allclose(o[0, :, h, :], pm, rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[0, h, :], np.log(np.arange(1, S + 1)), rtol=0,
                                   atol=1e-13)
        for i in range(S):
            want = np.zeros(D)
            for j in range(i + 1):
                want += np.dot(do[0, i, h, :], v[0, j, kh, :] - pm[i]) * k[0, j, kh, :]
            np.testing.assert_allclose(dq[0, i, h, :], sc * want / (i + 1), rtol=0,
                                       atol=1e-12)
    np.testing.assert_allclose(dk, 0.0, rtol=0, atol=0)
    for kh in range(Hkv):
        for j in range(S):
            want = sum(do[0, i, h, :] / (i + 1)
                       for h in range(kh * G, (kh + 1) * G) for i in range(j, S))
            np.testing.assert_allclose(dv[0, j, kh, :], want, rtol=0, atol=1e-12)


def check_gqa_equals_repeated_mha(causal, seed=21):
    q, k, v, do = (_np(t) for t in random_small(2, 10, 6, 2, 4, seed))
    G = 3
    kr, vr = np.repeat(k, G, axis=2), np.repeat(v, G, axis=2)
    a = ref.attn_bwd_ref(q, k, v, do, causal=causal)
    m = ref.attn_bwd_ref(q, kr, vr, do, causal=causal)
    for x, y in zip(a[:3], m[:3]):
        np.testing.assert_allclose(x, y, rtol=0, atol=1e-13)
    dk_sum = m[3].reshape(2, 10, 2, G, 4).sum(axis=3)
    dv_sum = m[4].reshape(2, 10, 2, G, 4).sum(axis=3)
    np.testing.assert_allclose(a[3], dk_sum, rtol=0, atol=1e-12)
    np.testing.assert_allclose(a[4], dv_sum, rtol=0, atol=1e-12)


def check_torch_sdpa(causal, B=2, S=33, Hq=8, Hkv=2, D=16, seed=9):
    """Library special case: torch's fp64 CPU scaled_dot_product_attention with the KV heads
    expanded by repeat_interleave, differentiated by autograd."""
    q, k, v, do = random_small(B, S, Hq, Hkv, D, seed)
    G = Hq // Hkv
    qt = q.transpose(1, 2).clone().requires_grad_(True)
    kt = k.transpose(1, 2).clone().requires_grad_(True)
    vt = v.transpose(1, 2).clone().requires_grad_(True)
    ot = torch.nn.functional.scaled_dot_product_attention(
        qt, kt.repeat_interleave(G, dim=1), vt.repeat_interleave(G, dim=1), is_causal=causal)
    ot.backward(do.transpose(1, 2))
    o, lse, dq, dk, dv = ref.attn_bwd_ref(_np(q), _np(k), _np(v), _np(do), causal=causal)
    np.testing.assert_allclose(o, _np(ot.transpose(1, 2)), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dq, _np(qt.grad.transpose(1, 2)), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, _np(kt.grad.transpose(1, 2)), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, _np(vt.grad.transpose(1, 2)), rtol=0, atol=1e-12)


def _brute_force(q, k, v, do, causal):
    """Scalar restatement with Python loops: tiny inputs only."""
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    sc = 1.0 / math.sqrt(D)
    o = np.zeros(q.shape); lse = np.zeros((B, Hq, S))
    dq = np.zeros(q.shape); dk = np.zeros(k.shape); dv = np.zeros(v.shape)
    for b in range(B):
        for h in range(Hq):
            c = h // G
            for i in range(S):
                js = list(range(i + 1)) if causal else list(range(S))
                s = [sc * sum(q[b, i, h, d] * k[b, j, c, d] for d in range(D)) for j in js]
                mx = max(s)
                w = [math.exp(x - mx) for x in s]
                tot = sum(w)
                p = [x / tot for x in w]
                lse[b, h, i] = mx + math.log(tot)
                for d in range(D):
                    o[b, i, h, d] = sum(p[t] * v[b, j, c, d] for t, j in enumerate(js))
                Di = sum(do[b, i, h, d] * o[b, i, h, d] for d in range(D))
                for t, j in enumerate(js):
                    dp = sum(do[b, i, h, d] * v[b, j, c, d] for d in range(D))
                    ds = p[t] * (dp - Di)
                    for d in range(D):
                        dq[b, i, h, d] += sc * ds * k[b, j, c, d]
                        dk[b, j, c, d] += sc * ds * q[b, i, h, d]
                        dv[b, j, c, d] += p[t] * do[b, i, h, d]
    return o, lse, dq, dk, dv


def check_brute_force(causal, seed=4):
    q, k, v, do = (_np(t) for t in random_small(2, 5, 4, 2, 3, seed))
    got = ref.attn_bwd_ref(q, k, v, do, causal=causal, row_block=2)
    want = _brute_force(q, k, v, do, causal)
    for x, y in zip(got, want):
        np.testing.assert_allclose(x, y, rtol=0, atol=1e-12)


def check_trunked_equals_plain(S, hc, T, causal=True, seed=13):
    q, k, v, do = (_np(t) for t in random_small(2, S, 8, 4, 8, seed))
    plain = ref.attn_bwd_ref(q, k, v, do, causal=causal, row_block=7)
    tr = ref.attn_bwd_trunked_ref(q, k, v, do, hc, T, causal=causal)
    for x, y in zip(plain, tr):
        np.testing.assert_allclose(x, y, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------------------
# tests
# ---------------------------------------------------------------------------------------

def test_hand_example():
    check_hand_example()


@pytest.mark.parametrize("causal", [True, False])
def test_finite_differences(causal):
    check_finite_differences(causal)


@pytest.mark.parametrize("causal", [True, False])
def test_identity_v_exposes_softmax_rows(causal):
    check_identity_v_rows(causal)


def test_constant_v_and_first_causal_row():
    check_constant_v_and_first_row()


def test_q_zero_closed_form():
    check_q_zero_closed_form()


@pytest.mark.parametrize("causal", [True, False])
def test_gqa_equals_repeated_mha(causal):
    check_gqa_equals_repeated_mha(causal)


@pytest.mark.parametrize("causal", [True, False])
def test_torch_sdpa_special_case(causal):
    check_torch_sdpa(causal)


@pytest.mark.parametrize("causal", [True, False])
def test_brute_force(causal):
    check_brute_force(causal)


@pytest.mark.parametrize("S,hc,T", [(40, 8, 40), (40, 4, 16), (40, 2, 8), (37, 8, 16),
                                    (37, 4, 37), (33, 2, 5)])
@pytest.mark.parametrize("causal", [True, False])
def test_trunk_and_head_chunk_invariance(S, hc, T, causal):
    """FPDT's trunk-by-trunk statistics merge and UPipe's head-group loop leave the result
    unchanged (to fp64 rounding), including a ragged last trunk."""
    check_trunked_equals_plain(S, hc, T, causal)


@pytest.mark.parametrize("causal", [True, False])
def test_sampled_rows_and_key_window_match_full(causal):
    q, k, v, do = random_small(1, 70, 4, 2, 8, 17)
    o, lse, dq, dk, dv = ref.attn_bwd_ref(q, k, v, do, causal=causal)
    for h in (0, 3):
        rows, ro, rl, rdq = ref.attn_rows_ref(q, k, v, do, 0, h, [69, 0, 33, 1, 64],
                                              causal=causal, row_block=2)
        np.testing.assert_allclose(ro, o[0, rows, h], rtol=0, atol=1e-13)
        np.testing.assert_allclose(rl, lse[0, h, rows], rtol=0, atol=1e-13)
        np.testing.assert_allclose(rdq, dq[0, rows, h], rtol=0, atol=1e-13)
    for kvh in (0, 1):
        wk, wv = ref.attn_dkdv_window_ref(q, k, v, do, 0, kvh, 50, 62, causal=causal,
                                          row_block=9)
        np.testing.assert_allclose(wk, dk[0, 50:62, kvh], rtol=0, atol=1e-13)
        np.testing.assert_allclose(wv, dv[0, 50:62, kvh], rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("key_lo,key_hi,want_rows", [(0, None, True), (23, 41, True),
                                                     (23, 41, False), (60, 70, False)])
def test_group_slice_matches_full(causal, key_lo, key_hi, want_rows):
    """attn_group_ref (PyTorch fp64 CPU, for the full-size checks) equals the slice of the
    pinned numpy oracle: every row of the group's q-heads, every key of the window, with
    row blocks that do not divide S."""
    q, k, v, do = random_small(2, 70, 6, 2, 8, 19)
    o, lse, dq, dk, dv = ref.attn_bwd_ref(q, k, v, do, causal=causal)
    G = 3
    for b, kvh in ((0, 1), (1, 0)):
        rows, go, gl, gdq, gdk, gdv = ref.attn_group_ref(
            q, k, v, do, b, kvh, causal=causal, key_lo=key_lo, key_hi=key_hi,
            want_rows=want_rows, row_block=9)
        hi = 70 if key_hi is None else key_hi
        np.testing.assert_allclose(gdk, dk[b, key_lo:hi, kvh], rtol=0, atol=1e-13)
        np.testing.assert_allclose(gdv, dv[b, key_lo:hi, kvh], rtol=0, atol=1e-13)
        if not want_rows:
            assert rows.size == 0
            continue
        assert rows[0] == (key_lo if causal else 0) and rows[-1] == 69
        hs = slice(kvh * G, (kvh + 1) * G)
        np.testing.assert_allclose(go, o[b, rows, hs], rtol=0, atol=1e-13)
        np.testing.assert_allclose(gl, lse[b, hs][:, rows], rtol=0, atol=1e-13)
        np.testing.assert_allclose(gdq, dq[b, rows, hs], rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("row_lo,key_lo,key_hi,want_dq", [(0, 0, None, True), (0, 23, 41, False),
                                                          (17, 23, 41, False), (23, 60, 70, True),
                                                          (0, 0, 70, False)])
def test_backward_from_row_statistics_matches_full(causal, row_lo, key_lo, key_hi, want_dq):
    """Splitting the backward into per-row statistics (LSE_i, D_i: the expensive forward half)
    and the dK/dV/dQ pass from them gives the slices of the pinned numpy oracle."""
    if not causal:
        row_lo = 0
    q, k, v, do = random_small(2, 70, 6, 2, 8, 29)
    o, lse, dq, dk, dv = ref.attn_bwd_ref(q, k, v, do, causal=causal)
    G = 3
    for b, kvh in ((0, 1), (1, 0)):
        hs = list(range(kvh * G, (kvh + 1) * G))
        st = [ref.attn_row_stats_ref(q, k, v, do, b, h, row_lo, 70, causal=causal, row_block=11)
              for h in hs]
        sl = np.stack([x[0] for x in st])
        sd = np.stack([x[1] for x in st])
        np.testing.assert_allclose(sl, lse[b][hs, row_lo:], rtol=0, atol=1e-13)
        want_d = np.einsum("ihd,ihd->hi", _np(do)[b][row_lo:, hs], o[b][row_lo:, hs])
        np.testing.assert_allclose(sd, want_d, rtol=0, atol=1e-12)
        gdk, gdv, gdq = ref.attn_group_from_stats_ref(q, k, v, do, b, kvh, sl, sd, row_lo,
                                                      key_lo=key_lo, key_hi=key_hi,
                                                      causal=causal, want_dq=want_dq,
                                                      row_block=9)
        hi = 70 if key_hi is None else key_hi
        np.testing.assert_allclose(gdk, dk[b, key_lo:hi, kvh], rtol=0, atol=1e-12)
        np.testing.assert_allclose(gdv, dv[b, key_lo:hi, kvh], rtol=0, atol=1e-12)
        if want_dq:
            np.testing.assert_allclose(gdq, dq[b][row_lo:, hs], rtol=0, atol=1e-12)
        else:
            assert gdq is None


def test_group_slice_closed_form_and_sdpa():
    """Two pins independent of the numpy oracle: with Q = 0 every causal row is the prefix
    mean of V, LSE_i = ln(i+1), dK = 0 and dV_j = sum_{i>=j} dO_i/(i+1) summed over the
    group; on random inputs it equals torch's fp64 scaled_dot_product_attention + autograd."""
    q, k, v, do = random_small(1, 40, 4, 2, 8, 23)
    z = torch.zeros_like(q)
    rows, go, gl, gdq, gdk, gdv = ref.attn_group_ref(z, k, v, do, 0, 1, row_block=7)
    vv = _np(v)[0, :, 1]
    dd = _np(do)[0, :, 2:4]
    n = np.arange(1, 41, dtype=np.float64)
    prefix = np.cumsum(vv, axis=0) / n[:, None]
    np.testing.assert_allclose(go[:, 0], prefix, rtol=0, atol=1e-12)
    np.testing.assert_allclose(go[:, 1], prefix, rtol=0, atol=1e-12)
    np.testing.assert_allclose(gl, np.log(n)[None, :].repeat(2, 0), rtol=0, atol=1e-12)
    np.testing.assert_allclose(gdk, 0.0, atol=1e-12)
    w = (dd / n[:, None, None]).sum(axis=1)
    want_dv = np.cumsum(w[::-1], axis=0)[::-1]
    np.testing.assert_allclose(gdv, want_dv, rtol=0, atol=1e-12)
    qt = q.transpose(1, 2).clone().requires_grad_(True)
    kt = k.transpose(1, 2).clone().requires_grad_(True)
    vt = v.transpose(1, 2).clone().requires_grad_(True)
    ot = torch.nn.functional.scaled_dot_product_attention(
        qt, kt.repeat_interleave(2, dim=1), vt.repeat_interleave(2, dim=1), is_causal=True)
    ot.backward(do.transpose(1, 2))
    rows, go, gl, gdq, gdk, gdv = ref.attn_group_ref(q, k, v, do, 0, 1, row_block=16)
    np.testing.assert_allclose(go, _np(ot.transpose(1, 2))[0, :, 2:4], rtol=0, atol=1e-12)
    np.testing.assert_allclose(gdq, _np(qt.grad.transpose(1, 2))[0, :, 2:4], rtol=0, atol=1e-12)
    np.testing.assert_allclose(gdk, _np(kt.grad.transpose(1, 2))[0, :, 1], rtol=0, atol=1e-12)
    np.testing.assert_allclose(gdv, _np(vt.grad.transpose(1, 2))[0, :, 1], rtol=0, atol=1e-12)


def test_torch_inputs_upcast_exactly():
    q, k, v, do = random_small(1, 16, 2, 1, 8, 1, dtype=torch.bfloat16)
    a = ref.attn_fwd_ref(q, k, v)
    b = ref.attn_fwd_ref(q.double().numpy(), k.double().numpy(), v.double().numpy())
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


# ---------------------------------------------------------------------------------------
# mutation test: plausible mistakes planted in the oracle must each fail some pin
# ---------------------------------------------------------------------------------------

def _all_pins():
    yield "hand", check_hand_example
    yield "fd", lambda: check_finite_differences(True, S=4, Hq=2, Hkv=1, D=2)
    yield "idv", lambda: check_identity_v_rows(True)
    yield "constv", check_constant_v_and_first_row
    yield "qzero", check_q_zero_closed_form
    yield "gqa", lambda: check_gqa_equals_repeated_mha(True)
    yield "sdpa", lambda: check_torch_sdpa(True, B=1, S=9, Hq=4, Hkv=2, D=4)
    yield "brute", lambda: check_brute_force(True)


def _mut_mask_off_by_one(qrows, keys, scale, row_pos, causal):
    s = scale * (qrows @ keys.T)
    if causal:
        j = np.arange(keys.shape[0])[None, :]
        s = np.where(j <= row_pos[:, None] + 1, s, -np.inf)
    return s


def _mut_transposed_scores(qrows, keys, scale, row_pos, causal):
    s = scale * (qrows @ keys.T)
    if s.shape[0] == s.shape[1]:
        s = s.T.copy()
    if causal:
        j = np.arange(keys.shape[0])[None, :]
        s = np.where(j <= row_pos[:, None], s, -np.inf)
    return s


def _mut_lse_no_max(s):
    mx = s.max(axis=1, keepdims=True)
    e = np.exp(s - mx)
    l = e.sum(axis=1, keepdims=True)
    return e / l, np.log(l)[:, 0]


def _mut_softmax_unnormalised(s):
    mx = s.max(axis=1, keepdims=True)
    e = np.exp(s - mx)
    l = e.sum(axis=1, keepdims=True)
    return e / l.mean(), (mx + np.log(l))[:, 0]


@pytest.mark.parametrize("name,attr,mutant", [
    ("mask_off_by_one", "_scores", _mut_mask_off_by_one),
    ("transposed_scores", "_scores", _mut_transposed_scores),
    ("scale_1_over_D", "_scale", lambda D, scale: 1.0 / D),
    ("scale_missing", "_scale", lambda D, scale: 1.0),
    ("lse_without_max", "_softmax_rows", _mut_lse_no_max),
    ("softmax_not_normalised", "_softmax_rows", _mut_softmax_unnormalised),
])
def test_pins_catch_planted_mistakes(monkeypatch, name, attr, mutant):
    monkeypatch.setattr(ref, attr, mutant)
    failed = []
    for pin, fn in _all_pins():
        try:
            with np.errstate(all="ignore"):
                fn()
        except (AssertionError, ValueError, FloatingPointError):
            failed.append(pin)
    assert failed, f"planted mistake {name} passed every pin"
