"""The forward entry point that allocates nothing, checked against the ordinary forward.

Some callers cannot call cudaMalloc: code running under an allocator or memory pool that owns
every device byte, code that forbids allocation after start-up, or plugins handed only their
inputs and outputs. upipe_attn_fwd_noalloc serves them by keeping the forward's scratch in a
static device array inside the library. Here it is called through the C ABI twice in a row, on
different inputs and shapes (the second call reuses the array the first one left behind), and
each result must match upipe_attn_fwd with a caller-supplied workspace within the parity
tolerances; neither call may allocate device memory. This file is collected last on purpose.
"""
import pytest
import torch

import context_parallelism_gb300 as up
from tests._parity import LSE_MAX_ABS, O_MAX_ABS
from workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

CALLS = [  # S, head_chunk, seq_trunk, seed: several trunks first, then one ragged trunk
    (1536, 8, 512, 51),
    (1000, 4, 1000, 52),
]


def test_noalloc_forward_matches_workspace_forward_on_two_calls():
    for i, (S, hc, T, seed) in enumerate(CALLS):
        w = WORKLOADS["llama8b_s8k"].with_(S=S, seed=seed)
        q, k, v, _ = (t.cuda() for t in make_inputs(w, "cpu"))
        o_ref, lse_ref = up.attention_forward(q, k, v, causal=True, head_chunk=hc, seq_trunk=T)
        up.upipe_sync_status()
        o = torch.full_like(q, float("nan"))
        lse = torch.full((1, w.Hq, S), float("nan"), device="cuda")
        torch.cuda.synchronize()
        alloc0 = torch.cuda.memory_allocated()
        free0, _ = torch.cuda.mem_get_info()
        up.upipe_attn_fwd_noalloc(q, k, v, o, lse, 1, S, w.Hq, w.Hkv, w.D, 1, hc, T,
                                  check_status=1 if i else 0)
        torch.cuda.synchronize()
        # no allocation through torch, and (after the first call's set-up) none on the device
        assert torch.cuda.memory_allocated() <= alloc0
        if i:
            assert torch.cuda.mem_get_info()[0] >= free0
        err_o = (o.float() - o_ref.float()).abs().max().item()
        err_l = (lse - lse_ref).abs().max().item()
        assert err_o <= O_MAX_ABS, (i, err_o)
        assert err_l <= LSE_MAX_ABS, (i, err_l)
    # a timeout would have been recorded in the entry point's status word: none was
    up.upipe_attn_fwd_noalloc(q, k, v, o, lse, 1, S, w.Hq, w.Hkv, w.D, 1, hc, T, check_status=1)
    torch.cuda.synchronize()


def test_noalloc_rejects_problems_beyond_its_scratch():
    w = WORKLOADS["llama8b_s8k"].with_(S=16384, seed=53)
    q = torch.zeros((1, w.S, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, w.S, w.Hkv, w.D), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((1, w.Hq, w.S), device="cuda")
    n0 = up.upipe_launch_count()
    with pytest.raises(up.UpipeError) as ei:
        up.upipe_attn_fwd_noalloc(q, k, k, o, lse, 1, w.S, w.Hq, w.Hkv, w.D, 1, 32, w.S)
    assert ei.value.status == up.UPIPE_ERR_WORKSPACE_TOO_SMALL
    assert "32 MiB" in str(ei.value)
    assert up.upipe_launch_count() == n0
