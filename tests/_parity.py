"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI and compare
it with the fp64 oracle.

Tolerances (from the workload definitions): max |O - O_ref| <= 1e-2 and relative Frobenius
error <= 2e-2 for dQ, dK and dV. LSE is held to max |LSE - LSE_ref| <= 5e-3, a gate derived
from the arithmetic: the kernel sums bf16-rounded probabilities against an fp32 running
maximum, so its LSE error is a few fp32 ulps of ln(l) plus the ex2/lg2 approximation error
(< 1e-5 relative), far inside 5e-3.
"""
import numpy as np
import torch

import context_parallelism_gb300 as up

O_MAX_ABS = 1e-2
LSE_MAX_ABS = 5e-3
GRAD_REL_FRO = 2e-2


def rel_fro(x, ref, floor_rms=0.0):
    """||x - ref||_F / ||ref||_F.

    floor_rms > 0 floors the denominator at that RMS per element. Only a caller whose exact
    gradient vanishes identically passes it (one token: P = 1, so dS = 0 and dQ = dK = 0),
    so that rounding noise of the order of fp32 ulps is not divided by zero; every other
    comparison is a plain relative error."""
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    num = float(np.linalg.norm(x - ref))
    den = max(float(np.linalg.norm(ref)), floor_rms * np.sqrt(max(ref.size, 1)))
    if den == 0.0:
        return 0.0 if num == 0.0 else float("inf")
    return num / den


def max_abs(x, ref):
    return float(np.max(np.abs(np.asarray(x, np.float64) - np.asarray(ref, np.float64))))


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def gpu_fwd_bwd(q, k, v, do, causal, hc, T):
    """Runs upipe_attn_fwd then upipe_attn_bwd (k/v may be pinned host tensors)."""
    o, lse = up.attention_forward(q, k, v, causal=causal, head_chunk=hc, seq_trunk=T)
    up.upipe_sync_status()
    dq, dk, dv = up.attention_backward(q, k, v, o, lse, do, causal=causal, head_chunk=hc,
                                       seq_trunk=T)
    up.upipe_sync_status()
    return o, lse, dq, dk, dv


def check_full(gpu, ref, label="", grad_floor_rms=0.0):
    """Every output against the oracle's. grad_floor_rms: see rel_fro (one-token cases only)."""
    o, lse, dq, dk, dv = gpu
    ro, rlse, rdq, rdk, rdv = ref
    errs = {
        "o_max_abs": max_abs(to_np(o), ro),
        "lse_max_abs": max_abs(to_np(lse), rlse),
        "dq_rel_fro": rel_fro(to_np(dq), rdq, grad_floor_rms),
        "dk_rel_fro": rel_fro(to_np(dk), rdk, grad_floor_rms),
        "dv_rel_fro": rel_fro(to_np(dv), rdv, grad_floor_rms),
    }
    bad = [k for k, lim in (("o_max_abs", O_MAX_ABS), ("lse_max_abs", LSE_MAX_ABS),
                            ("dq_rel_fro", GRAD_REL_FRO), ("dk_rel_fro", GRAD_REL_FRO),
                            ("dv_rel_fro", GRAD_REL_FRO)) if not errs[k] <= lim]
    assert not bad, f"{label}: {errs}"
    return errs


def pinned_copy(t):
    h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    h.copy_(t)
    return h
