"""Workspace bounds: every call is given a workspace of exactly the declared size, cut out of a
larger buffer whose guard bands before and after it hold a canary byte pattern. After the call
the guards must be unchanged: no kernel or staging copy writes outside the bytes the library
declared (the caller-owned arena is the library's only scratch). Needs an sm_103a GPU."""
import pytest
import torch

import context_parallelism_gb300 as up
from workloads import LOSS_WORKLOADS, MLP_WORKLOADS, WORKLOADS, make_inputs, \
    make_loss_inputs, make_mlp_inputs

pytestmark = pytest.mark.gpu

GUARD = 1 << 20  # bytes on each side, a multiple of 256 so the workspace stays aligned
CANARY = 0xA5


class Guarded:
    def __init__(self, nbytes):
        self.n = nbytes
        self.buf = torch.full((nbytes + 2 * GUARD,), CANARY, dtype=torch.uint8, device="cuda")
        self.ws = self.buf[GUARD:GUARD + nbytes]

    def check(self):
        torch.cuda.synchronize()
        lo, hi = self.buf[:GUARD], self.buf[GUARD + self.n:]
        assert int((lo != CANARY).sum()) == 0, "write before the workspace"
        assert int((hi != CANARY).sum()) == 0, "write past the end of the workspace"


def _pinned(t):
    out = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    out.copy_(t)
    return out


@pytest.mark.parametrize("S,hc,T,kv_host,act_host", [
    (1000, 4, 256, False, False),   # several trunks, ragged
    (1000, 8, 1000, False, False),  # one trunk
    (777, 4, 256, True, False),     # host K/V slots
    (640, 4, 256, True, True),      # everything on the host
])
def test_attention_stays_inside_its_workspace(S, hc, T, kv_host, act_host):
    w = WORKLOADS["llama8b_s8k"].with_(S=S, Hq=8, Hkv=2, seed=71 + S)
    q, k, v, do = make_inputs(w, "cpu")
    B, Hq, Hkv, D = w.B, w.Hq, w.Hkv, w.D
    dev = (lambda t: _pinned(t)) if act_host else (lambda t: t.cuda())
    kvd = (lambda t: _pinned(t)) if kv_host else (lambda t: t.cuda())
    qi, doi, ki, vi = dev(q), dev(do), kvd(k), kvd(v)
    mask = (up.UPIPE_HOST_KV if kv_host else 0) | (up.UPIPE_HOST_ACT if act_host else 0)
    for pass_ in (up.UPIPE_PASS_FWD, up.UPIPE_PASS_BWD):
        g = Guarded(up.upipe_workspace_bytes(B, S, Hq, Hkv, D, 1, hc, T, pass_, mask))
        if pass_ == up.UPIPE_PASS_FWD:
            o, lse = up.attention_forward(qi, ki, vi, head_chunk=hc, seq_trunk=T,
                                          workspace=g.ws, o_on_host=act_host)
        else:
            up.attention_backward(qi, ki, vi, o, lse, doi, head_chunk=hc, seq_trunk=T,
                                  workspace=g.ws, dkdv_on_host=kv_host, dq_on_host=act_host)
        up.upipe_sync_status()
        g.check()


@pytest.mark.parametrize("S,T,host", [(1000, 256, False), (1000, 256, True), (100, 128, True)])
def test_tiled_paths_stay_inside_their_workspace(S, T, host):
    lw = LOSS_WORKLOADS["readout_small"].with_(S=S, seed=73 + S)
    h, w, t, gl = make_loss_inputs(lw, "cpu")
    hi = _pinned(h) if host else h.cuda()
    wg, tg, gg = w.cuda(), t.cuda(), gl.cuda()
    mask = up.UPIPE_HOST_ACT if host else 0
    g = Guarded(up.upipe_ce_workspace_bytes(S, lw.Dm, lw.V, T, up.UPIPE_PASS_FWD, mask))
    loss, lse = up.ce_loss_forward(hi, wg, tg, seq_tile=T, workspace=g.ws)
    up.upipe_sync_status()
    g.check()
    g = Guarded(up.upipe_ce_workspace_bytes(S, lw.Dm, lw.V, T, up.UPIPE_PASS_BWD, mask))
    up.ce_loss_backward(hi, wg, tg, lse, gg, seq_tile=T, workspace=g.ws, dh_on_host=host)
    up.upipe_sync_status()
    g.check()

    mw = MLP_WORKLOADS["mlp_small"].with_(S=S, seed=75 + S)
    x, w_gu, w_d, dy = make_mlp_inputs(mw, "cpu")
    xi = _pinned(x) if host else x.cuda()
    dyi = _pinned(dy) if host else dy.cuda()
    wgu, wdd = w_gu.cuda(), w_d.cuda()
    g = Guarded(up.upipe_mlp_workspace_bytes(S, mw.Dm, mw.F, T, up.UPIPE_PASS_FWD, mask))
    up.mlp_forward(xi, wgu, wdd, seq_tile=T, workspace=g.ws, y_on_host=host)
    up.upipe_sync_status()
    g.check()
    g = Guarded(up.upipe_mlp_workspace_bytes(S, mw.Dm, mw.F, T, up.UPIPE_PASS_BWD, mask))
    up.mlp_backward(xi, wgu, wdd, dyi, seq_tile=T, workspace=g.ws, dx_on_host=host)
    up.upipe_sync_status()
    g.check()
