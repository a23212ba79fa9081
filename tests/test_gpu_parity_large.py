"""Parity at the full sizes of the three long-sequence workloads, in the launch configuration the
benchmark times. The fp64 oracle cannot afford every output here, so the check covers:
  * O, LSE and dQ on seeded samples of query rows (always including tile and trunk edges and
    the last row) of several q-heads, each row's softmax taken over its full key range;
  * dK and dV on the last 256 key rows of two kv-heads (they need only the last 256 query
    rows' statistics), which straddles a 128-row tile edge and ends the last trunk;
  * properties that hold at any size: everything finite, the workspace ratio, and no device
    allocation beyond the caller's workspace.
Needs an sm_103a GPU with the memory of a GB300."""
import numpy as np
import pytest
import torch

import context_parallelism_gb300 as up
import oracle
from tests._parity import (GRAD_REL_FRO, LSE_MAX_ABS, O_MAX_ABS, gpu_fwd_bwd, max_abs,
                           pinned_copy, rel_fro, to_np)
from workloads import WORKLOADS, make_inputs, sample_rows

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


def _free():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def test_llama8b_s128k_sampled():
    w = WORKLOADS["llama8b_s128k"]
    inputs = make_inputs(w)
    for hc, T in ((8, 131072), (4, 32768), (32, 16384)):
        outs = gpu_fwd_bwd(*inputs, True, hc, T)
        _check_sampled(w, inputs, outs, heads=[0, 13, 31], n_rows=48, kv_heads=[0, 7], T=T)
        del outs
    _free()


def test_llama8b_s1m_host_kv_sampled():
    w = WORKLOADS["llama8b_s1m_hostkv"]
    q, k, v, do = make_inputs(w)
    kh, vh = pinned_copy(k), pinned_copy(v)
    outs = gpu_fwd_bwd(q, kh, vh, do, True, w.head_chunk, w.seq_trunk)
    _check_sampled(w, (q, k, v, do), outs, heads=[0, 31], n_rows=32, kv_heads=[7],
                   window=128)
    del outs, kh, vh
    _free()


def test_gqa32b_s256k_peaky_sampled_and_workspace_ratio():
    w = WORKLOADS["gqa32b_s256k_peaky"]
    inputs = make_inputs(w)
    need = {}
    for hc in (8, 64):
        outs = gpu_fwd_bwd(*inputs, True, hc, w.seq_trunk)
        _check_sampled(w, inputs, outs, heads=[0, 37, 63], n_rows=32, kv_heads=[0], T=w.seq_trunk)
        need[hc] = up.upipe_workspace_bytes(w.B, w.S, w.Hq, w.Hkv, w.D, 1, hc, w.seq_trunk,
                                            up.UPIPE_PASS_BOTH, 0)
        del outs
        _free()
    assert need[8] / need[64] <= 8 / 64 + 1e-9
