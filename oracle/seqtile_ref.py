"""fp64 CPU oracle for the sequence-tiled per-token computations: the language-model readout
(hidden state times the vocabulary matrix) followed by token-level cross-entropy, and the
gated (SwiGLU) MLP.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports, calls or links this module:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg use it.
It shares no code with the CUDA path; both take their inputs from ``workloads``.

What it computes. The pages name sequence tiling as the step that chunks the per-token
("element-wise along the sequence") computations, the loss among them, so that no buffer
with the whole sequence along one dimension is ever created ["Road to 5 million sequence
length" talk notes, the Arctic sequence-tiling passage; "Road to 5 Million Tokens" summary,
§2 item 5, "Sequence Tiling"]. Tiling does not change the result: every token's loss
depends on that token alone. So the oracle is the plain, untiled definition:

    logits[i, j] = <h_i, w_j>                          (i < S tokens, j < V vocabulary rows)
    lse[i]       = log sum_j exp(logits[i, j])         (natural log)
    loss[i]      = lse[i] - logits[i, target[i]]       (0 where target[i] < 0: ignored token)

and, for an upstream gradient g[i] = d(total)/d(loss[i]),

    dlogits[i, j] = g[i] * (softmax(logits[i])_j - [j == target[i]])   (row 0 if ignored)
    dh[i]         = sum_j dlogits[i, j] * w_j
    dw[j]         = sum_i dlogits[i, j] * h_i

Readings where the pages are silent: the loss is next-token cross-entropy over the logits of
a linear readout (the buffer the pages call huge is the S x V logits); a negative target
marks a token that takes no loss and no gradient (padding); lse and loss are returned per
token, and the caller's reduction (mean, sum) enters only through g.

Layouts: h [S, Dm], w [V, Dm], target [S] integers, loss / lse / g [S], dh [S, Dm],
dw [V, Dm]. Arithmetic is numpy float64 on exactly upcast inputs; the logits are formed
``block`` rows at a time only to bound memory (each row is independent, so the blocking
cannot change any value).

The MLP (the other per-token computation the same passages name) is the gated form of the
Llama-family models whose shapes the workloads use:

    g = x Wg^T,  u = x Wu^T  (Wg, Wu [F, Dm], stacked as w_gu = [Wg; Wu], [2F, Dm])
    a = silu(g) * u,  silu(z) = z / (1 + exp(-z))
    y = a Wd^T  (Wd [Dm, F])

and, for dy = d(total)/dy,

    da = dy Wd;  dg = da * u * silu'(g),  silu'(z) = s (1 + z (1 - s)),  s = 1/(1 + exp(-z))
    du = da * silu(g);  dx = dg Wg + du Wu
    dWd = dy^T a;  dWg = dg^T x;  dWu = du^T x  (returned stacked as dw_gu = [dWg; dWu])

Readings: the pages name "the MLPs" without a form; SwiGLU is read as the MLP of the modelled
architecture, with no biases. Every token's y and dx depend on that token alone.

Parity status: every public function here is pinned by tests/test_oracle_seqtile.py (finite
differences, closed forms, a logistic-loss special case, scipy's logsumexp, torch's fp64
autograd of the MLP, invariants).
"""
from __future__ import annotations

import numpy as np

__all__ = ["ce_loss_ref", "ce_loss_bwd_ref", "ce_rows_ref", "mlp_ref", "mlp_bwd_ref",
           "mlp_rows_ref"]


def _f64(x):
    """Exact upcast to a float64 numpy array (bf16 -> fp32 -> fp64 are exact)."""
    if hasattr(x, "detach"):
        t = x.detach()
        if t.is_floating_point() and t.element_size() < 4:
            t = t.float()
        return t.cpu().numpy().astype(np.float64, copy=False)
    return np.asarray(x, dtype=np.float64)


def _i64(x):
    if hasattr(x, "detach"):
        return x.detach().cpu().numpy().astype(np.int64, copy=False)
    return np.asarray(x, dtype=np.int64)


def _row_stats(logits, tgt):
    """lse and loss of a block of logit rows (max-shifted log-sum-exp, natural log)."""
    m = logits.max(axis=1)
    lse = m + np.log(np.exp(logits - m[:, None]).sum(axis=1))
    valid = tgt >= 0
    picked = np.where(valid, logits[np.arange(len(tgt)), np.where(valid, tgt, 0)], 0.0)
    loss = np.where(valid, lse - picked, 0.0)
    return lse, loss


def _dlogits(logits, lse, tgt, G):
    """g (softmax - onehot(target)) for a block of logit rows; rows of ignored tokens are 0."""
    p = np.exp(logits - lse[:, None])          # softmax rows
    valid = tgt >= 0
    rows = np.nonzero(valid)[0]
    p[rows, tgt[rows]] -= 1.0
    p *= np.where(valid, G, 0.0)[:, None]
    return p


def ce_loss_ref(h, w, target, block: int = 512):
    """Forward: per-token (loss, lse), each float64 [S]."""
    H, W, t = _f64(h), _f64(w), _i64(target)
    S = H.shape[0]
    lse = np.empty(S)
    loss = np.empty(S)
    for r0 in range(0, S, block):
        r1 = min(S, r0 + block)
        lse[r0:r1], loss[r0:r1] = _row_stats(H[r0:r1] @ W.T, t[r0:r1])
    return loss, lse


def ce_loss_bwd_ref(h, w, target, g, block: int = 512):
    """Forward and backward: (loss, lse, dh, dw), float64, dh [S, Dm], dw [V, Dm]."""
    H, W, t, G = _f64(h), _f64(w), _i64(target), _f64(g)
    S = H.shape[0]
    lse = np.empty(S)
    loss = np.empty(S)
    dh = np.empty_like(H)
    dw = np.zeros_like(W)
    for r0 in range(0, S, block):
        r1 = min(S, r0 + block)
        logits = H[r0:r1] @ W.T
        tb = t[r0:r1]
        lse[r0:r1], loss[r0:r1] = _row_stats(logits, tb)
        p = _dlogits(logits, lse[r0:r1], tb, G[r0:r1])
        dh[r0:r1] = p @ W
        dw += p.T @ H[r0:r1]
    return loss, lse, dh, dw


def ce_rows_ref(h, w, target, g, rows, vocab_rows=None):
    """loss, lse and dh at the given token rows only (each row needs only its own logits):
    the check used where the whole problem is too large for the CPU. With ``vocab_rows``, also
    the sampled tokens' share of dw at those vocabulary rows, sum_{i in rows} dlogits[i, j] h_i
    - the whole of dw[j] when g is zero at every other token."""
    rows = np.asarray(rows, dtype=np.int64)
    if hasattr(h, "detach"):
        import torch
        idx = torch.as_tensor(rows, device=h.device)
        H = _f64(h[idx])
        t = _i64(target[idx])
        G = _f64(g[idx])
    else:
        H, t, G = _f64(h)[rows], _i64(target)[rows], _f64(g)[rows]
    W = _f64(w)
    logits = H @ W.T
    lse, loss = _row_stats(logits, t)
    p = _dlogits(logits, lse, t, G)
    if vocab_rows is None:
        return loss, lse, p @ W
    vr = np.asarray(vocab_rows, dtype=np.int64)
    return loss, lse, p @ W, p[:, vr].T @ H


# ---- gated (SwiGLU) MLP ---------------------------------------------------------------------

def _silu_parts(z):
    """silu(z) and its derivative, with the logistic s = 1/(1 + e^-z) formed stably."""
    s = np.empty_like(z)
    pos = z >= 0
    s[pos] = 1.0 / (1.0 + np.exp(-z[pos]))
    ez = np.exp(z[~pos])
    s[~pos] = ez / (1.0 + ez)
    return z * s, s * (1.0 + z * (1.0 - s))


def _mlp_rows(X, Wgu, Wd, dY):
    F = Wd.shape[1]
    gu = X @ Wgu.T
    g, u = gu[:, :F], gu[:, F:]
    sg, dsg = _silu_parts(g)
    a = sg * u
    y = a @ Wd.T
    if dY is None:
        return y, None, None, None
    da = dY @ Wd
    dgu = np.concatenate([da * u * dsg, da * sg], axis=1)
    dx = dgu @ Wgu
    return y, dx, dgu, a


def mlp_ref(x, w_gu, w_d, block: int = 512):
    """Forward: y [S, Dm] float64."""
    X, Wgu, Wd = _f64(x), _f64(w_gu), _f64(w_d)
    y = np.empty((X.shape[0], Wd.shape[0]))
    for r0 in range(0, X.shape[0], block):
        y[r0:r0 + block] = _mlp_rows(X[r0:r0 + block], Wgu, Wd, None)[0]
    return y


def mlp_bwd_ref(x, w_gu, w_d, dy, block: int = 512):
    """Forward and backward: (y, dx, dw_gu [2F, Dm], dw_d [Dm, F]), float64."""
    X, Wgu, Wd, dY = _f64(x), _f64(w_gu), _f64(w_d), _f64(dy)
    S = X.shape[0]
    y = np.empty((S, Wd.shape[0]))
    dx = np.empty_like(X)
    dw_gu = np.zeros_like(Wgu)
    dw_d = np.zeros_like(Wd)
    for r0 in range(0, S, block):
        r1 = min(S, r0 + block)
        yb, dxb, dgu, a = _mlp_rows(X[r0:r1], Wgu, Wd, dY[r0:r1])
        y[r0:r1], dx[r0:r1] = yb, dxb
        dw_gu += dgu.T @ X[r0:r1]
        dw_d += dY[r0:r1].T @ a
    return y, dx, dw_gu, dw_d


def mlp_rows_ref(x, w_gu, w_d, dy, rows, gu_rows=None, d_rows=None):
    """y and dx at the given token rows only, and, when gu_rows / d_rows are given, those
    tokens' share of dw_gu (at rows gu_rows) and of dw_d (at rows d_rows) - the whole of them
    when dy is zero at every other token."""
    rows = np.asarray(rows, dtype=np.int64)
    if hasattr(x, "detach"):
        import torch
        idx = torch.as_tensor(rows, device=x.device)
        X, dY = _f64(x[idx]), _f64(dy[idx])
    else:
        X, dY = _f64(x)[rows], _f64(dy)[rows]
    Wgu, Wd = _f64(w_gu), _f64(w_d)
    y, dx, dgu, a = _mlp_rows(X, Wgu, Wd, dY)
    out = [y, dx]
    if gu_rows is not None:
        out.append(dgu[:, np.asarray(gu_rows)].T @ X)
    if d_rows is not None:
        out.append(dY[:, np.asarray(d_rows)].T @ a)
    return tuple(out)
