"""The forward entry point that allocates nothing, checked against the ordinary forward.

Some callers cannot call cudaMalloc: code running under an allocator or memory pool that owns
every device byte, code that forbids allocation after start-up, or plugins handed only their
inputs and outputs. upipe_attn_fwd_noalloc serves them by keeping the forward's scratch in a
static device array inside the library. It runs the same kernels on the same arena layout as
upipe_attn_fwd with a caller-supplied workspace, so its o and lse must be bitwise equal to that
call's. Each case below calls it through the C ABI twice in a row on different inputs (the
second call reuses the array the first one left behind); neither call may allocate device
memory. The cases cover several trunks, one ragged trunk, a non-causal mask with a ragged last
trunk, the D = 64 kernel and a batch of two. This file is collected last on purpose.
"""
import pytest
import torch

import context_parallelism_gb300 as up
from workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

# (workload, B, S, head_chunk, seq_trunk, causal)
CASES = {
    "several_trunks": ("llama8b_s8k", 1, 1536, 8, 512, 1),
    "one_ragged_trunk": ("llama8b_s8k", 1, 1000, 4, 1000, 1),
    "non_causal_ragged_trunks": ("llama8b_s8k", 1, 1000, 8, 256, 0),
    "d64": ("mha_s512_d64", 1, 512, 2, 256, 1),
    "batch_two": ("llama8b_s8k", 2, 640, 8, 256, 1),
}


def _inputs(name, B, S, seed):
    w = WORKLOADS[name].with_(B=B, S=S, seed=seed)
    q, k, v, _ = (t.cuda() for t in make_inputs(w, "cpu"))
    return w, q, k, v


@pytest.mark.parametrize("case", list(CASES))
def test_noalloc_forward_bitwise_equals_workspace_forward_on_two_calls(case):
    name, B, S, hc, T, causal = CASES[case]
    for call, seed in enumerate((61, 62)):
        w, q, k, v = _inputs(name, B, S, seed)
        o_ref, lse_ref = up.attention_forward(q, k, v, causal=bool(causal), head_chunk=hc,
                                              seq_trunk=T)
        up.upipe_sync_status()
        o = torch.full_like(q, float("nan"))
        lse = torch.full((B, w.Hq, S), float("nan"), device="cuda")
        torch.cuda.synchronize()
        alloc0 = torch.cuda.memory_allocated()
        free0, _ = torch.cuda.mem_get_info()
        up.upipe_attn_fwd_noalloc(q, k, v, o, lse, B, S, w.Hq, w.Hkv, w.D, causal, hc, T,
                                  check_status=call)
        torch.cuda.synchronize()
        assert up.upipe_last_error_message() == ""
        # no allocation through torch, and (after the first call's set-up) none on the device
        assert torch.cuda.memory_allocated() <= alloc0
        if call:
            assert torch.cuda.mem_get_info()[0] >= free0
        assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16)), (case, call)
        assert torch.equal(lse.view(torch.int32), lse_ref.view(torch.int32)), (case, call)
    # a bounded wait that expired would have been recorded in the status word: none was
    up.upipe_attn_fwd_noalloc(q, k, v, o, lse, B, S, w.Hq, w.Hkv, w.D, causal, hc, T,
                              check_status=1)
    torch.cuda.synchronize()


def test_noalloc_leaves_the_current_device_unchanged():
    w, q, k, v = _inputs("mha_s512_d64", 1, 512, 63)
    o = torch.empty_like(q)
    lse = torch.empty((1, w.Hq, 512), device="cuda")
    torch.cuda.set_device(0)
    up.upipe_attn_fwd_noalloc(q, k, v, o, lse, 1, 512, w.Hq, w.Hkv, w.D, 1, 4, 512)
    torch.cuda.synchronize()
    assert torch.cuda.current_device() == 0


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
