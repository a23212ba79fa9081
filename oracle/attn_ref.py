"""fp64 CPU oracle for exact causal (GQA) self-attention, forward and backward.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports, calls or links this module:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg use it.
It shares no code with the CUDA path; both take their inputs from ``workloads``.

What it computes (the plain definition; the head-chunked, trunked method reaches exactly this
result, only with less memory):
  * exact attention, every query attending every earlier-or-equal key
    ["Road to 5 Million Tokens" summary, "The Bottlenecks": quadratic pairwise interactions;
     "Training Ultra Long Context LM with FPDT", Technical Deep Dive: a query token attends
     to the keys/values that precede it or are simultaneous];
  * softmax with the running-maximum statistic the FPDT Technical Deep Dive names; here the
    maximum is taken over the full row at once (no online merge), which is the definition;
  * the backward pass is the analytic gradient of that function; P is recomputed from the
    saved statistic the way FlashAttention-style backward passes recompute it
    ["Training Ultra Long Context LM with FPDT", Background: the attention backward pass].

Readings where the pages are silent (all from the workload definitions, not the pages):
  scale = 1/sqrt(D); causal visibility j <= i with S_q = S_k; GQA maps q-head h to kv-head
  floor(h / (Hq/Hkv)); LSE uses the natural log and is returned as [B, Hq, S].

Layouts: q, dout, o, dq are token-major [B, S, Hq, D]; k, v, dk, dv are [B, S, Hkv, D].
All arithmetic is float64: numpy, except attn_group_ref, which evaluates the same formulas
with PyTorch's CPU fp64 operations so that whole slices at S >= 128K use every host core.
Inputs of any float dtype are upcast exactly.

Parity status: every public function here is pinned by tests/test_oracle.py (finite
differences, closed forms, invariants, brute force, a library special case).
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "attn_fwd_ref",
    "attn_bwd_ref",
    "attn_rows_ref",
    "attn_dkdv_window_ref",
    "attn_group_ref",
    "attn_row_stats_ref",
    "attn_group_from_stats_ref",
    "attn_fwd_trunked_ref",
    "attn_bwd_trunked_ref",
]


def _f64(x):
    """Exact upcast to a float64 numpy array (bf16/fp16 -> fp32 -> fp64 are exact)."""
    if hasattr(x, "detach"):  # a torch tensor, on any device
        t = x.detach()
        if t.is_floating_point() and t.element_size() < 4:
            t = t.float()
        return t.cpu().numpy().astype(np.float64, copy=False)
    return np.asarray(x, dtype=np.float64)


def _take(x, b, rows, h):
    """x[b, rows, h, :] for a numpy array or a torch tensor (rows: int array)."""
    if hasattr(x, "detach"):
        import torch
        return x[b, torch.as_tensor(rows, device=x.device), h, :]
    return np.asarray(x)[b, rows, h, :]


def _shapes(q, k):
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    return B, S, Hq, Hkv, D, Hq // Hkv


def _scale(D, scale):
    return 1.0 / math.sqrt(D) if scale is None else float(scale)


def _scores(qrows, keys, scale, row_pos, causal):
    """s_ij = scale * <q_i, k_j>, with keys j > i set to -inf when causal.
    qrows [n, D] at absolute positions row_pos [n]; keys [m, D] at positions 0..m-1."""
    s = scale * (qrows @ keys.T)
    if causal:
        j = np.arange(keys.shape[0])[None, :]
        s = np.where(j <= row_pos[:, None], s, -np.inf)
    return s


def _softmax_rows(s):
    """P = exp(s - max) / sum exp(s - max) over each full row, plus LSE = max + ln(sum)."""
    mx = s.max(axis=1, keepdims=True)
    e = np.exp(s - mx)
    l = e.sum(axis=1, keepdims=True)
    return e / l, (mx + np.log(l))[:, 0]


def attn_fwd_ref(q, k, v, causal=True, scale=None, row_block=512):
    """O = softmax(scale * Q K^T + causal mask) V per (b, h); LSE per row.

    Returns (o [B,S,Hq,D], lse [B,Hq,S]) in float64."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, S, Hq, Hkv, D, G = _shapes(q, k)
    sc = _scale(D, scale)
    o = np.empty((B, S, Hq, D))
    lse = np.empty((B, Hq, S))
    for b in range(B):
        for h in range(Hq):
            kh = h // G
            K, V = k[b, :, kh, :], v[b, :, kh, :]
            for i0 in range(0, S, row_block):
                i1 = min(S, i0 + row_block)
                m = i1 if causal else S  # keys beyond the block's last row are all masked
                s = _scores(q[b, i0:i1, h, :], K[:m], sc, np.arange(i0, i1), causal)
                P, l = _softmax_rows(s)
                o[b, i0:i1, h, :] = P @ V[:m]
                lse[b, h, i0:i1] = l
    return o, lse


def attn_bwd_ref(q, k, v, dout, causal=True, scale=None, row_block=512):
    """Analytic gradients of O = softmax(scale*QK^T + mask) V, given dO.

    With P recomputed per row block:
        D_i   = <dO_i, O_i>
        dP_ij = <dO_i, v_j>
        dS_ij = P_ij (dP_ij - D_i)
        dQ_i  = scale * sum_j dS_ij k_j
        dK_j  = scale * sum_{h in group} sum_i dS_ij q_i
        dV_j  = sum_{h in group} sum_i P_ij dO_i
    Returns (o, lse, dq, dk, dv) in float64 (o, lse as in attn_fwd_ref)."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, S, Hq, Hkv, D, G = _shapes(q, k)
    sc = _scale(D, scale)
    o = np.empty((B, S, Hq, D))
    lse = np.empty((B, Hq, S))
    dq = np.empty((B, S, Hq, D))
    dk = np.zeros((B, S, Hkv, D))
    dv = np.zeros((B, S, Hkv, D))
    for b in range(B):
        for h in range(Hq):
            kh = h // G
            K, V = k[b, :, kh, :], v[b, :, kh, :]
            for i0 in range(0, S, row_block):
                i1 = min(S, i0 + row_block)
                m = i1 if causal else S
                Qb, dOb = q[b, i0:i1, h, :], do[b, i0:i1, h, :]
                s = _scores(Qb, K[:m], sc, np.arange(i0, i1), causal)
                P, l = _softmax_rows(s)
                Ob = P @ V[:m]
                o[b, i0:i1, h, :] = Ob
                lse[b, h, i0:i1] = l
                Di = np.sum(dOb * Ob, axis=1, keepdims=True)
                dP = dOb @ V[:m].T
                dS = P * (dP - Di)
                dq[b, i0:i1, h, :] = sc * (dS @ K[:m])
                dk[b, :m, kh, :] += sc * (dS.T @ Qb)
                dv[b, :m, kh, :] += P.T @ dOb
    return o, lse, dq, dk, dv


def attn_rows_ref(q, k, v, dout, b, h, rows, causal=True, scale=None, row_block=64):
    """O_i, LSE_i and dQ_i for the query rows ``rows`` of (batch b, q-head h) only.

    Each row is the same definition as attn_bwd_ref restricted to that row (its softmax
    still runs over the row's full key range); its cost is O(i * D), which makes spot checks
    at S >= 128K affordable. Rows are processed in sorted blocks so K and V stream through
    BLAS once per block. Returns (rows_sorted, o [n,D], lse [n], dq [n,D])."""
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    kh = h // (Hq // Hkv)
    sc = _scale(D, scale)
    rows = np.asarray(sorted(set(int(r) for r in rows)), dtype=np.int64)
    m_all = int(rows[-1]) + 1 if causal else S
    K = _f64(k[b, :m_all, kh, :])
    V = _f64(v[b, :m_all, kh, :])
    o = np.empty((len(rows), D))
    lse = np.empty(len(rows))
    dq = np.empty((len(rows), D))
    for n0 in range(0, len(rows), row_block):
        r = rows[n0:n0 + row_block]
        m = int(r[-1]) + 1 if causal else S
        Qb = _f64(_take(q, b, r, h))
        dOb = _f64(_take(dout, b, r, h))
        s = _scores(Qb, K[:m], sc, r, causal)
        P, l = _softmax_rows(s)
        Ob = P @ V[:m]
        Di = np.sum(dOb * Ob, axis=1, keepdims=True)
        dS = P * (dOb @ V[:m].T - Di)
        o[n0:n0 + len(r)] = Ob
        lse[n0:n0 + len(r)] = l
        dq[n0:n0 + len(r)] = sc * (dS @ K[:m])
    return rows, o, lse, dq


def attn_dkdv_window_ref(q, k, v, dout, b, kvh, j0, j1, causal=True, scale=None,
                         row_block=256):
    """dK_j and dV_j for key rows j in [j0, j1) of (batch b, kv-head kvh).

    Sums over the G q-heads of the group and over every query row that sees key j
    (rows i >= j0 when causal); each such row's softmax is taken over its full key range,
    so the window's result equals the corresponding slice of attn_bwd_ref."""
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    sc = _scale(D, scale)
    dk = np.zeros((j1 - j0, D))
    dv = np.zeros((j1 - j0, D))
    i_start = j0 if causal else 0
    K = _f64(k[b, :, kvh, :])
    V = _f64(v[b, :, kvh, :])
    for h in range(kvh * G, (kvh + 1) * G):
        for i0 in range(i_start, S, row_block):
            i1 = min(S, i0 + row_block)
            m = max(i1, j1) if causal else S  # window keys past row i are masked to 0
            Qb = _f64(q[b, i0:i1, h, :])
            dOb = _f64(dout[b, i0:i1, h, :])
            s = _scores(Qb, K[:m], sc, np.arange(i0, i1), causal)
            P, _ = _softmax_rows(s)
            Ob = P @ V[:m]
            Di = np.sum(dOb * Ob, axis=1, keepdims=True)
            Pw = P[:, j0:j1]
            dSw = Pw * (dOb @ V[j0:j1].T - Di)
            dk += sc * (dSw.T @ Qb)
            dv += Pw.T @ dOb
    return dk, dv


def attn_group_ref(q, k, v, dout, b, kvh, causal=True, scale=None, key_lo=0, key_hi=None,
                   want_rows=True, row_block=512):
    """One (batch b, kv-head kvh) slice of the definition, for the full-size checks.

    For every q-head h of the kv-head's group (h in [kvh*G, (kvh+1)*G)):
      * with want_rows: O_i, LSE_i and dQ_i for every query row i in [row_lo, S);
      * dK_j and dV_j for key rows j in [key_lo, key_hi) (default: all keys), summed over the
        group's q-heads and over every query row that sees key j;
    where row_lo = key_lo when causal (earlier rows see none of the window's keys), else 0.
    Each row's softmax is taken over its full key range, so every value equals the matching
    entry of attn_bwd_ref: the same formulas (D_i = <dO_i, O_i>, dS = P (dP - D), dQ, dK,
    dV as there), evaluated with PyTorch's fp64 CPU operations, whose matrix products and
    element-wise passes use every host core. That is what makes a whole slice affordable at
    S = 128K (about 5e13 flops) and a key window at S = 1M.

    Returns (rows [n], o [n, G, D], lse [G, n], dq [n, G, D], dk [m, D], dv [m, D]) as fp64
    numpy arrays, rows = arange(row_lo, S) (empty arrays when want_rows is False)."""
    import torch

    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    sc = _scale(D, scale)
    key_hi = S if key_hi is None else int(key_hi)
    key_lo = int(key_lo)
    row_lo = key_lo if causal else 0
    f64 = torch.float64

    def col(x, h, lo=0):  # rows [lo, S) of head h of a [B, S, H, D] tensor, fp64 on the CPU
        t = torch.as_tensor(x) if not hasattr(x, "detach") else x.detach()
        return t[b, lo:, h, :].to("cpu").to(f64)

    K = col(k, kvh)
    V = col(v, kvh)
    n = S - row_lo if want_rows else 0
    o = torch.zeros((n, G, D), dtype=f64)
    lse = torch.zeros((G, n), dtype=f64)
    dq = torch.zeros((n, G, D), dtype=f64)
    dk = torch.zeros((key_hi - key_lo, D), dtype=f64)
    dv = torch.zeros((key_hi - key_lo, D), dtype=f64)
    for g in range(G):
        h = kvh * G + g
        Q = col(q, h, row_lo)
        dO = col(dout, h, row_lo)
        for i0 in range(row_lo, S, row_block):
            i1 = min(S, i0 + row_block)
            m = i1 if causal else S  # keys past the block's last row are masked for all rows
            Qb, dOb = Q[i0 - row_lo:i1 - row_lo], dO[i0 - row_lo:i1 - row_lo]
            s = torch.mm(Qb, K[:m].T).mul_(sc)
            if causal:  # only columns j >= i0 can lie above a row of this block
                j = torch.arange(i0, m)[None, :]
                i = torch.arange(i0, i1)[:, None]
                s[:, i0:].masked_fill_(j > i, float("-inf"))
            mx = s.max(dim=1, keepdim=True).values
            P = s.sub_(mx).exp_()  # in place: s is not needed again
            l = P.sum(dim=1, keepdim=True)
            P.div_(l)
            Ob = P @ V[:m]
            Di = (dOb * Ob).sum(dim=1, keepdim=True)
            w1 = min(key_hi, m)
            if want_rows:
                dS = torch.mm(dOb, V[:m].T).sub_(Di).mul_(P)
                r = slice(i0 - row_lo, i1 - row_lo)
                o[r, g] = Ob
                lse[g, r] = (mx + torch.log(l))[:, 0]
                dq[r, g] = sc * (dS @ K[:m])
                dSw = dS[:, key_lo:w1]
            else:
                dSw = torch.mm(dOb, V[key_lo:w1].T).sub_(Di).mul_(P[:, key_lo:w1])
            if w1 > key_lo:
                dk[: w1 - key_lo] += sc * (dSw.T @ Qb)
                dv[: w1 - key_lo] += P[:, key_lo:w1].T @ dOb
    rows = np.arange(row_lo, S) if want_rows else np.zeros(0, dtype=np.int64)
    return rows, o.numpy(), lse.numpy(), dq.numpy(), dk.numpy(), dv.numpy()


def attn_row_stats_ref(q, k, v, dout, b, h, row_lo, row_hi, causal=True, scale=None,
                       row_block=512):
    """The two per-row statistics the backward pass needs, for query rows [row_lo, row_hi) of
    (batch b, q-head h): LSE_i = max_j s_ij + ln sum_j exp(s_ij - max) and D_i = <dO_i, O_i>,
    each row's softmax taken over its full key range (the definition, as in attn_bwd_ref),
    with PyTorch's fp64 CPU operations. Returns (lse [n], dvec [n]) as fp64 numpy arrays.

    This is the expensive half of a backward check at S >= 128K: the statistics of every row
    that sees a key window need that row's full score row and O_i."""
    import torch

    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    kvh = h // (Hq // Hkv)
    sc = _scale(D, scale)
    f64 = torch.float64

    def rows_of(x, hh, lo, hi):
        t = torch.as_tensor(x) if not hasattr(x, "detach") else x.detach()
        return t[b, lo:hi, hh, :].to("cpu").to(f64)

    m_all = row_hi if causal else S
    K = rows_of(k, kvh, 0, m_all)
    V = rows_of(v, kvh, 0, m_all)
    Q = rows_of(q, h, row_lo, row_hi)
    dO = rows_of(dout, h, row_lo, row_hi)
    lse = torch.empty(row_hi - row_lo, dtype=f64)
    dvec = torch.empty(row_hi - row_lo, dtype=f64)
    for i0 in range(row_lo, row_hi, row_block):
        i1 = min(row_hi, i0 + row_block)
        m = i1 if causal else S
        r = slice(i0 - row_lo, i1 - row_lo)
        s = torch.mm(Q[r], K[:m].T).mul_(sc)
        if causal:
            j = torch.arange(i0, m)[None, :]
            i = torch.arange(i0, i1)[:, None]
            s[:, i0:].masked_fill_(j > i, float("-inf"))
        mx = s.max(dim=1, keepdim=True).values
        P = s.sub_(mx).exp_()
        l = P.sum(dim=1, keepdim=True)
        P.div_(l)
        lse[r] = (mx + torch.log(l))[:, 0]
        dvec[r] = (dO[r] * (P @ V[:m])).sum(dim=1)
    return lse.numpy(), dvec.numpy()


def attn_group_from_stats_ref(q, k, v, dout, b, kvh, lse, dvec, row_lo, key_lo=0, key_hi=None,
                              causal=True, scale=None, want_dq=False, row_block=512):
    """The backward of one (batch b, kv-head kvh) slice from given row statistics.

    lse, dvec: [G, S - row_lo] fp64, LSE_i and D_i of rows [row_lo, S) of the group's q-heads
    (from attn_row_stats_ref). With P_ij = exp(s_ij - LSE_i) (the probabilities recomputed
    from the saved statistic, as the FPDT talk's Background describes the attention backward)
    and dS_ij = P_ij (dP_ij - D_i), returns
      dK_j = scale sum_h sum_i dS_ij q_i and dV_j = sum_h sum_i P_ij dO_i for keys
      [key_lo, key_hi), and, with want_dq, dQ_i = scale sum_j dS_ij k_j for rows [row_lo, S).
    Causal rows below key_lo see no key of the window, so row_lo <= key_lo suffices (row_lo
    must be 0 when not causal). Returns (dk [m, D], dv [m, D], dq [S - row_lo, G, D] or None)
    as fp64 numpy arrays; PyTorch fp64 CPU operations."""
    import torch

    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    sc = _scale(D, scale)
    key_hi = S if key_hi is None else int(key_hi)
    if row_lo > (key_lo if causal else 0):
        raise ValueError("rows below row_lo would see the key window")
    f64 = torch.float64

    def rows_of(x, hh, lo, hi):
        t = torch.as_tensor(x) if not hasattr(x, "detach") else x.detach()
        return t[b, lo:hi, hh, :].to("cpu").to(f64)

    lse = torch.as_tensor(np.asarray(lse, dtype=np.float64))
    dvec = torch.as_tensor(np.asarray(dvec, dtype=np.float64))
    K = rows_of(k, kvh, 0, S)
    V = rows_of(v, kvh, 0, S)
    dk = torch.zeros((key_hi - key_lo, D), dtype=f64)
    dv = torch.zeros((key_hi - key_lo, D), dtype=f64)
    dq = torch.zeros((S - row_lo, G, D), dtype=f64) if want_dq else None
    # rows that matter: all given rows for dQ; else those that see the window
    first_row = row_lo if want_dq else (key_lo if causal else 0)
    for g in range(G):
        h = kvh * G + g
        Q = rows_of(q, h, row_lo, S)
        dO = rows_of(dout, h, row_lo, S)
        for i0 in range(first_row, S, row_block):
            i1 = min(S, i0 + row_block)
            r = slice(i0 - row_lo, i1 - row_lo)
            # key columns this block needs: every visible key (for dQ) or the window's
            visible = i1 if causal else S
            c0 = 0 if want_dq else key_lo
            c1 = visible if want_dq else min(key_hi, visible)
            if c1 <= c0:
                continue
            s = torch.mm(Q[r], K[c0:c1].T).mul_(sc)
            s.sub_(lse[g, r][:, None])
            if causal:  # columns j >= i0 can lie above a row of this block
                lo = max(c0, i0)
                if lo < c1:
                    j = torch.arange(lo, c1)[None, :]
                    i = torch.arange(i0, i1)[:, None]
                    s[:, lo - c0:].masked_fill_(j > i, float("-inf"))
            P = s.exp_()
            dS = torch.mm(dO[r], V[c0:c1].T).sub_(dvec[g, r][:, None]).mul_(P)
            if want_dq:
                dq[r, g] = sc * (dS @ K[c0:c1])
            w0, w1 = max(key_lo, c0), min(key_hi, c1)
            if w1 > w0:
                dk[w0 - key_lo:w1 - key_lo] += sc * (dS[:, w0 - c0:w1 - c0].T @ Q[r])
                dv[w0 - key_lo:w1 - key_lo] += P[:, w0 - c0:w1 - c0].T @ dO[r]
    return dk.numpy(), dv.numpy(), (dq.numpy() if want_dq else None)


# ----------------------------------------------------------------------------------------
# The head-chunked, trunked formulation. Used only to self-check the merge arithmetic the
# method relies on: it must reproduce attn_fwd_ref / attn_bwd_ref to fp64 rounding.
# ----------------------------------------------------------------------------------------

def _trunks(S, T):
    return [(t0, min(S, t0 + T)) for t0 in range(0, S, T)]


def attn_fwd_trunked_ref(q, k, v, head_chunk, seq_trunk, causal=True, scale=None):
    """UPipe x FPDT forward schedule, written out in fp64.

    For each head group of ``head_chunk`` q-heads ["Road to 5 million sequence length"
    talk, UPipe passage: compute one set of heads at a time, reusing the buffers], for each
    query trunk m, fold the key/value trunks n = 0..m (all n when not causal) into running
    statistics ["Training Ultra Long Context LM with FPDT", Technical Deep Dive: partial
    output plus maximum-logit statistics updated per trunk]:
        m_new = max(m_run, rowmax(s));  a = exp(m_run - m_new)
        l_run = a*l_run + rowsum(exp(s - m_new));  acc = a*acc + exp(s - m_new) V_n
    and finish with O = acc / l_run, LSE = m_run + ln(l_run)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, S, Hq, Hkv, D, G = _shapes(q, k)
    if Hq % head_chunk or head_chunk % G:
        raise ValueError("head_chunk must divide Hq and be a multiple of Hq/Hkv")
    sc = _scale(D, scale)
    o = np.empty((B, S, Hq, D))
    lse = np.empty((B, Hq, S))
    trunks = _trunks(S, seq_trunk)
    for g0 in range(0, Hq, head_chunk):
        for b in range(B):
            for h in range(g0, g0 + head_chunk):
                kh = h // G
                for mi, (q0, q1) in enumerate(trunks):
                    Qm = q[b, q0:q1, h, :]
                    acc = np.zeros((q1 - q0, D))
                    m_run = np.full(q1 - q0, -np.inf)
                    l_run = np.zeros(q1 - q0)
                    for ni, (k0, k1) in enumerate(trunks):
                        if causal and ni > mi:
                            break
                        s = sc * (Qm @ k[b, k0:k1, kh, :].T)
                        if causal and ni == mi:
                            vis = np.arange(k0, k1)[None, :] <= np.arange(q0, q1)[:, None]
                            s = np.where(vis, s, -np.inf)
                        m_new = np.maximum(m_run, s.max(axis=1))
                        a = np.exp(m_run - m_new)
                        p = np.exp(s - m_new[:, None])
                        l_run = a * l_run + p.sum(axis=1)
                        acc = a[:, None] * acc + p @ v[b, k0:k1, kh, :]
                        m_run = m_new
                    o[b, q0:q1, h, :] = acc / l_run[:, None]
                    lse[b, h, q0:q1] = m_run + np.log(l_run)
    return o, lse


def attn_bwd_trunked_ref(q, k, v, dout, head_chunk, seq_trunk, causal=True, scale=None):
    """Backward in the same schedule: per head group, per key/value trunk n (outer), per
    query trunk m >= n (all m when not causal), P recomputed from the forward's LSE:
        P = exp(s - LSE_i), dS = P (dO V_n^T - D_i), D_i = <dO_i, O_i>,
        dV_n += P^T dO_m, dK_n += scale dS^T Q_m, dQ_m += scale dS K_n.
    Returns (o, lse, dq, dk, dv) in float64."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, S, Hq, Hkv, D, G = _shapes(q, k)
    sc = _scale(D, scale)
    o, lse = attn_fwd_trunked_ref(q, k, v, head_chunk, seq_trunk, causal, scale)
    dq = np.zeros((B, S, Hq, D))
    dk = np.zeros((B, S, Hkv, D))
    dv = np.zeros((B, S, Hkv, D))
    trunks = _trunks(S, seq_trunk)
    for g0 in range(0, Hq, head_chunk):
        for b in range(B):
            for h in range(g0, g0 + head_chunk):
                kh = h // G
                Dvec = np.sum(do[b, :, h, :] * o[b, :, h, :], axis=1)
                for ni, (k0, k1) in enumerate(trunks):
                    Kn, Vn = k[b, k0:k1, kh, :], v[b, k0:k1, kh, :]
                    for mi, (q0, q1) in enumerate(trunks):
                        if causal and mi < ni:
                            continue
                        Qm, dOm = q[b, q0:q1, h, :], do[b, q0:q1, h, :]
                        s = sc * (Qm @ Kn.T)
                        if causal and mi == ni:
                            vis = np.arange(k0, k1)[None, :] <= np.arange(q0, q1)[:, None]
                            s = np.where(vis, s, -np.inf)
                        P = np.exp(s - lse[b, h, q0:q1][:, None])
                        dS = P * (dOm @ Vn.T - Dvec[q0:q1][:, None])
                        dv[b, k0:k1, kh, :] += P.T @ dOm
                        dk[b, k0:k1, kh, :] += sc * (dS.T @ Qm)
                        dq[b, q0:q1, h, :] += sc * (dS @ Kn)
    return o, lse, dq, dk, dv
