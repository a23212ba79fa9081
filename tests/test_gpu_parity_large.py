"""Parity at the full sizes of the three long-sequence workloads, in the launch configuration the
benchmark times. The fp64 oracle cannot afford every output of every head here. Its costly
half, the per-row statistics LSE_i and D_i = <dO_i, O_i> of the rows that matter, is stored in
tests/golden/ (written by tests/golden/attn_stats.py, which calls only the oracle, with a
fingerprint of the exact input bytes); each test recomputes the rest. The checks cover:
  * one full (batch 0, kv-head 0) slice at S = 128K: dK, dV of every key and LSE of every row
    of the kv-head's q-heads, at each (head_chunk, trunk) point, so every key tile is checked
    over its whole backward walk, trunk boundaries included;
  * at S = 1M (K/V in pinned host memory) and S = 256K (peaky keys): dK and dV on a 256-key
    window straddling a trunk boundary (S - T at 1M; at 256K the last boundary whose window
    holds one of the x8 key rows), and LSE of every later row;
  * O, LSE and dQ on seeded samples of query rows (always including tile and trunk edges and
    the last row) of several q-heads, each row's softmax taken over its full key range (the
    oracle in full, at test time), and dK, dV on the last keys of another kv-head;
  * properties that hold at any size: everything finite and the workspace ratio.
Needs an sm_103a GPU with the memory of a GB300.
"""
import numpy as np
import pytest
import torch

import context_parallelism_gb300 as up
import oracle
from tests._parity import (GRAD_REL_FRO, LSE_MAX_ABS, O_MAX_ABS, gpu_fwd_bwd, max_abs,
                           pinned_copy, rel_fro, to_np)
from tests.golden import attn_stats
from workloads import WORKLOADS, make_inputs, peaky_rows, sample_rows

pytestmark = pytest.mark.gpu


def _check_sampled(w, inputs, outs, heads, n_rows, kv_heads, window=256, T=None):
    q, k, v, do = inputs
    o, lse, dq, dk, dv = outs
    T = T or w.seq_trunk
    errs = {"o": 0.0, "lse": 0.0}
    dq_num = dq_den = 0.0
    for h in heads:
        rows = sample_rows(w.S, T, n_rows, seed=1000 + h)
        r, ro, rl, rdq = oracle.attn_rows_ref(q, k, v, do, 0, h, rows, causal=w.causal)
        ridx = torch.as_tensor(r, device=o.device)
        go = to_np(o[0, ridx, h])
        gl = to_np(lse[0, h, ridx])
        gdq = to_np(dq[0, ridx, h])
        errs["o"] = max(errs["o"], max_abs(go, ro))
        errs["lse"] = max(errs["lse"], max_abs(gl, rl))
        dq_num += float(np.sum((gdq - rdq) ** 2))
        dq_den += float(np.sum(rdq ** 2))
    errs["dq"] = (dq_num / max(dq_den, 1e-30)) ** 0.5
    dk_num = dk_den = dv_num = dv_den = 0.0
    for kvh in kv_heads:
        j0 = w.S - window
        rdk, rdv = oracle.attn_dkdv_window_ref(q, k, v, do, 0, kvh, j0, w.S, causal=w.causal)
        gdk = to_np(dk[0, j0:, kvh])
        gdv = to_np(dv[0, j0:, kvh])
        dk_num += float(np.sum((gdk - rdk) ** 2)); dk_den += float(np.sum(rdk ** 2))
        dv_num += float(np.sum((gdv - rdv) ** 2)); dv_den += float(np.sum(rdv ** 2))
    errs["dk"] = (dk_num / max(dk_den, 1e-30)) ** 0.5
    errs["dv"] = (dv_num / max(dv_den, 1e-30)) ** 0.5
    assert errs["o"] <= O_MAX_ABS, errs
    assert errs["lse"] <= LSE_MAX_ABS, errs
    for g in ("dq", "dk", "dv"):
        assert errs[g] <= GRAD_REL_FRO, errs
    for t in (o, lse, dq, dk, dv):
        assert bool(torch.isfinite(t).all())
    return errs


def _stored_stats(name, inputs):
    """The oracle's stored row statistics for this workload (tests/golden/attn_stats.py), after
    checking that they were computed from exactly these input bytes."""
    st = attn_stats.load(name)
    fp = attn_stats.fingerprint(*inputs, st["kvh"], st["row_lo"])
    assert fp == st["fingerprint"], (
        f"{name}: the seeded inputs differ from those the stored statistics were computed "
        f"from; rerun python -m tests.golden.attn_stats {name}")
    return st


def _check_stats_and_keys(outs, inputs, st, key_lo, key_hi, label):
    """LSE of every covered row of the kv-head's q-heads against the stored oracle values;
    dK, dV of keys [key_lo, key_hi) against the oracle's backward from those statistics."""
    o, lse, dq, dk, dv = outs
    q, k, v, do = inputs
    kvh, row_lo = st["kvh"], st["row_lo"]
    G = q.shape[2] // k.shape[2]
    errs = {"lse": max_abs(to_np(lse[0, kvh * G:(kvh + 1) * G, row_lo:]), st["lse"])}
    rdk, rdv, _ = oracle.attn_group_from_stats_ref(q, k, v, do, 0, kvh, st["lse"], st["dvec"],
                                                   row_lo, key_lo=key_lo, key_hi=key_hi,
                                                   causal=True, row_block=1024)
    errs["dk"] = rel_fro(to_np(dk[0, key_lo:key_hi, kvh]), rdk)
    errs["dv"] = rel_fro(to_np(dv[0, key_lo:key_hi, kvh]), rdv)
    assert errs["lse"] <= LSE_MAX_ABS, (label, errs)
    assert max(errs["dk"], errs["dv"]) <= GRAD_REL_FRO, (label, errs)
    return errs


def _free():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def test_llama8b_s128k_full_group_slice_and_samples():
    """The whole (batch 0, kv-head 0) slice: dK, dV of all 131072 keys and LSE of all 4 x 131072
    rows of the kv-head's q-heads (the oracle's backward from its stored row statistics, about
    3.5e13 fp64 flops on the host cores), at the benchmark's point and two chunked/trunked
    points; O, LSE and dQ on sampled rows of three q-heads."""
    w = WORKLOADS["llama8b_s128k"]
    inputs = make_inputs(w)
    st = _stored_stats(w.name, inputs)
    G = w.Hq // w.Hkv
    q, k, v, do = inputs
    rdk, rdv, _ = oracle.attn_group_from_stats_ref(q, k, v, do, 0, 0, st["lse"], st["dvec"], 0,
                                                   causal=True, row_block=1024)
    for hc, T in ((8, 131072), (4, 32768), (32, 16384)):
        o, lse, dq, dk, dv = outs = gpu_fwd_bwd(*inputs, True, hc, T)
        errs = {"lse": max_abs(to_np(lse[0, 0:G]), st["lse"]),
                "dk": rel_fro(to_np(dk[0, :, 0]), rdk), "dv": rel_fro(to_np(dv[0, :, 0]), rdv)}
        assert errs["lse"] <= LSE_MAX_ABS, (hc, T, errs)
        assert max(errs["dk"], errs["dv"]) <= GRAD_REL_FRO, (hc, T, errs)
        _check_sampled(w, inputs, outs, heads=[0, 13, 31], n_rows=48, kv_heads=[7], T=T)
        del outs, o, lse, dq, dk, dv
    _free()


def test_llama8b_s1m_host_kv_sampled_and_trunk_window():
    """The 1M-token workload: K/V in pinned host memory, 64K trunks. Besides the sampled rows,
    dK/dV of kv-head 7 on [S - T - 128, S - T + 128), the window straddling the last trunk
    boundary, and LSE of every query row from S - T - 128 on."""
    w = WORKLOADS["llama8b_s1m_hostkv"]
    q, k, v, do = make_inputs(w)
    st = _stored_stats(w.name, (q, k, v, do))
    kh, vh = pinned_copy(k), pinned_copy(v)
    outs = gpu_fwd_bwd(q, kh, vh, do, True, w.head_chunk, w.seq_trunk)
    del kh, vh
    _check_sampled(w, (q, k, v, do), outs, heads=[0, 31], n_rows=32, kv_heads=[7],
                   window=128)
    _, _, (j0, j1) = attn_stats.spec(w.name)
    _check_stats_and_keys(outs, (q, k, v, do), st, j0, j1, "S=1M trunk window")
    del outs
    _free()


def test_gqa32b_s256k_peaky_sampled_and_workspace_ratio():
    """32B-class shape with 1% of K rows scaled x8. dK/dV of kv-head 0 on a 256-key window
    straddling the last trunk boundary whose window holds one of the scaled key rows."""
    w = WORKLOADS["gqa32b_s256k_peaky"]
    inputs = make_inputs(w)
    st = _stored_stats(w.name, inputs)
    _, j0, (k0, k1) = attn_stats.spec(w.name, peaky_rows(w))
    assert j0 == st["row_lo"]
    T = w.seq_trunk
    need = {}
    for hc in (8, 64):
        outs = gpu_fwd_bwd(*inputs, True, hc, T)
        _check_sampled(w, inputs, outs, heads=[0, 37, 63], n_rows=32, kv_heads=[0], T=T)
        _check_stats_and_keys(outs, inputs, st, k0, k1, f"peaky window hc={hc}")
        need[hc] = up.upipe_workspace_bytes(w.B, w.S, w.Hq, w.Hkv, w.D, 1, hc, T,
                                            up.UPIPE_PASS_BOTH, 0)
        del outs
        _free()
    assert need[8] / need[64] <= 8 / 64 + 1e-9
