"""upipe_shutdown releases every per-device object the library created lazily (the attention
copy streams, the tiled calls' staging streams, events, the status word); the next call
creates them again and computes the same results. Named to run after the other GPU tests.
Needs an sm_103a GPU."""
import pytest
import torch

import context_parallelism_gb300 as up
from workloads import MLP_WORKLOADS, WORKLOADS, make_inputs, make_mlp_inputs

pytestmark = pytest.mark.gpu


def _pinned(t):
    out = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    out.copy_(t)
    return out


def test_shutdown_then_reuse():
    mw = MLP_WORKLOADS["mlp_small"].with_(S=500, seed=91)
    x, w_gu, w_d, _ = make_mlp_inputs(mw, "cpu")
    xh, wg, wd = _pinned(x), w_gu.cuda(), w_d.cuda()
    w = WORKLOADS["llama8b_s8k"].with_(S=512, seed=93)
    q, k, v, _ = make_inputs(w, "cpu")
    qg, kh, vh = q.cuda(), _pinned(k), _pinned(v)

    def run():
        y = up.mlp_forward(xh, wg, wd, seq_tile=128, y_on_host=True)
        o, lse = up.attention_forward(qg, kh, vh, head_chunk=8, seq_trunk=256)
        up.upipe_sync_status()
        return y, o, lse

    first = run()
    torch.cuda.synchronize()
    up.upipe_shutdown()
    second = run()
    up.upipe_shutdown()
    third = run()
    for a, b, c in zip(first, second, third):
        assert torch.equal(a.cpu(), b.cpu()) and torch.equal(a.cpu(), c.cpu())
