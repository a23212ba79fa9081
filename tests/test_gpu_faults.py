"""Failure handling of the host staging, without faulting the GPU: a staging copy made to fail
on the host (the test hook upipe_debug_fail_copy_after) must surface as UPIPE_ERR_CUDA from the
call that would have issued it, leave nothing hung (the stream synchronises), and leave the
library usable: the next call gives bitwise the result of a clean run. Needs an sm_103a GPU."""
import pytest
import torch

import context_parallelism_gb300 as up
from workloads import LOSS_WORKLOADS, MLP_WORKLOADS, WORKLOADS, make_inputs, \
    make_loss_inputs, make_mlp_inputs

pytestmark = pytest.mark.gpu


def _pinned(t):
    out = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    out.copy_(t)
    return out


def _expect_injected(fn):
    with pytest.raises(up.UpipeError) as e:
        fn()
    assert e.value.status == up.UPIPE_ERR_CUDA and "injected" in str(e.value)
    up.upipe_sync_status()  # everything already enqueued completes; no device error


@pytest.mark.parametrize("n", [1, 3])
def test_attention_host_kv_copy_failure_then_recovery(n):
    w = WORKLOADS["llama8b_s8k"].with_(S=1024, seed=61)
    q, k, v, do = make_inputs(w, "cpu")
    qg, dog = q.cuda(), do.cuda()
    kh, vh = _pinned(k), _pinned(v)
    o_ref, lse_ref = up.attention_forward(qg, kh, vh, head_chunk=8, seq_trunk=256)
    up.upipe_debug_fail_copy_after(n)
    _expect_injected(lambda: up.attention_forward(qg, kh, vh, head_chunk=8, seq_trunk=256))
    o, lse = up.attention_forward(qg, kh, vh, head_chunk=8, seq_trunk=256)
    up.upipe_sync_status()
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
    # the backward's dK/dV copy-out path too
    ref = up.attention_backward(qg, kh, vh, o, lse, dog, head_chunk=8, seq_trunk=256,
                                dkdv_on_host=True)
    up.upipe_sync_status()
    up.upipe_debug_fail_copy_after(n + 4)
    _expect_injected(lambda: up.attention_backward(qg, kh, vh, o, lse, dog, head_chunk=8,
                                                   seq_trunk=256, dkdv_on_host=True))
    dq, dk, dv = up.attention_backward(qg, kh, vh, o, lse, dog, head_chunk=8, seq_trunk=256,
                                       dkdv_on_host=True)
    up.upipe_sync_status()
    assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])
    assert (dq.float() - ref[0].float()).abs().max() <= 1e-2  # dQ sums reorder


@pytest.mark.parametrize("n", [1, 2, 5])
def test_tiled_paths_copy_failure_then_recovery(n):
    mw = MLP_WORKLOADS["mlp_small"].with_(S=1000, seed=63)
    x, w_gu, w_d, dy = make_mlp_inputs(mw, "cpu")
    wg, wd = w_gu.cuda(), w_d.cuda()
    xh, dyh = _pinned(x), _pinned(dy)
    ref = up.mlp_backward(xh, wg, wd, dyh, seq_tile=256, dx_on_host=True)
    up.upipe_sync_status()
    up.upipe_debug_fail_copy_after(n)
    _expect_injected(lambda: up.mlp_backward(xh, wg, wd, dyh, seq_tile=256, dx_on_host=True))
    got = up.mlp_backward(xh, wg, wd, dyh, seq_tile=256, dx_on_host=True)
    up.upipe_sync_status()
    assert all(torch.equal(a, b) for a, b in zip(got, ref))

    lw = LOSS_WORKLOADS["readout_small"].with_(seed=65)
    h, w, t, g = make_loss_inputs(lw, "cpu")
    hh, wg2, tg, gg = _pinned(h), w.cuda(), t.cuda(), g.cuda()
    loss, lse = up.ce_loss_forward(hh, wg2, tg, seq_tile=256)
    ref = up.ce_loss_backward(hh, wg2, tg, lse, gg, seq_tile=256, dh_on_host=True)
    up.upipe_sync_status()
    up.upipe_debug_fail_copy_after(n)
    _expect_injected(lambda: up.ce_loss_backward(hh, wg2, tg, lse, gg, seq_tile=256,
                                                 dh_on_host=True))
    got = up.ce_loss_backward(hh, wg2, tg, lse, gg, seq_tile=256, dh_on_host=True)
    up.upipe_sync_status()
    assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])


def test_disarmed_hook_changes_nothing():
    up.upipe_debug_fail_copy_after(0)
    mw = MLP_WORKLOADS["mlp_small"].with_(S=300, seed=67)
    x, w_gu, w_d, _ = make_mlp_inputs(mw, "cpu")
    y1 = up.mlp_forward(_pinned(x), w_gu.cuda(), w_d.cuda(), seq_tile=128)
    y2 = up.mlp_forward(x.cuda(), w_gu.cuda(), w_d.cuda(), seq_tile=128)
    up.upipe_sync_status()
    assert torch.equal(y1, y2)
