"""Parity of the sequence-tiled gated MLP (upipe_mlp_fwd / upipe_mlp_bwd, through the C ABI)
with the fp64 oracle. Needs an sm_103a GPU.

Tolerances, from the arithmetic: the GEMMs sum exact bf16 products in fp32; between them the
path rounds a = silu(g) u (forward) and g, u, dg, du (backward) to bf16, 2^-9 relative per
element, and y and dx to bf16 on output. Every output is therefore within a few 2^-9 of the
exact value in the relative Frobenius norm: held to 1e-2 (y, dx, dw_gu, dw_d).
"""
import numpy as np
import pytest
import torch

import context_parallelism_gb300 as up
import oracle
from tests._parity import rel_fro, to_np
from workloads import MLP_WORKLOADS, make_mlp_inputs

pytestmark = pytest.mark.gpu

REL_FRO = 1e-2


def _run(x, w_gu, w_d, dy, T):
    xg, wg, wd, dyg = x.cuda(), w_gu.cuda(), w_d.cuda(), dy.cuda()
    y = up.mlp_forward(xg, wg, wd, seq_tile=T)
    dx, dw_gu, dw_d = up.mlp_backward(xg, wg, wd, dyg, seq_tile=T)
    up.upipe_sync_status()
    return y, dx, dw_gu, dw_d


CASES = [
    # S, Dm, F, seq_tile
    (1000, 256, 384, 256),   # 4 token tiles (last ragged), F = 3 x 128
    (1000, 256, 384, 1024),  # one ragged token tile
    (300, 64, 128, 128),     # Dm = one k block, F = one gate/up tile
    (1, 64, 256, 128),       # a single token
    (2048, 512, 1024, 512),  # several full tiles each way
]


@pytest.mark.parametrize("S,Dm,F,T", CASES)
def test_mlp_parity(S, Dm, F, T):
    mw = MLP_WORKLOADS["mlp_small"].with_(S=S, Dm=Dm, F=F, seq_tile=T, seed=40 + S + F)
    x, w_gu, w_d, dy = make_mlp_inputs(mw, "cpu")
    ry, rdx, rdg, rdd = oracle.mlp_bwd_ref(x, w_gu, w_d, dy)
    y, dx, dw_gu, dw_d = _run(x, w_gu, w_d, dy, T)
    tag = f"S={S} Dm={Dm} F={F} T={T}"
    assert rel_fro(to_np(y), ry) <= REL_FRO, tag
    assert rel_fro(to_np(dx), rdx) <= REL_FRO, tag
    assert rel_fro(to_np(dw_gu), rdg) <= REL_FRO, tag
    assert rel_fro(to_np(dw_d), rdd) <= REL_FRO, tag


def test_mlp_tiling_does_not_change_per_token_results():
    mw = MLP_WORKLOADS["mlp_small"].with_(S=1024, seed=45)
    x, w_gu, w_d, dy = make_mlp_inputs(mw, "cpu")
    a = _run(x, w_gu, w_d, dy, 128)
    b = _run(x, w_gu, w_d, dy, 1024)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    assert rel_fro(to_np(a[2]), to_np(b[2])) <= 1e-5
    assert rel_fro(to_np(a[3]), to_np(b[3])) <= 1e-5


def test_mlp_rejects_bad_shapes():
    x = torch.zeros((256, 64), dtype=torch.bfloat16, device="cuda")
    w_gu = torch.zeros((2 * 96, 64), dtype=torch.bfloat16, device="cuda")  # F % 128 != 0
    w_d = torch.zeros((64, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(up.UpipeError) as e:
        up.mlp_forward(x, w_gu, w_d, seq_tile=128)
    assert e.value.status == up.UPIPE_ERR_UNSUPPORTED


def _pinned(t):
    out = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    out.copy_(t)
    return out


@pytest.mark.parametrize("S,T,which", [(1000, 256, "all"), (600, 128, "x"), (300, 128, "dy"),
                                       (100, 128, "outputs")])
def test_mlp_host_activations_equal_device(S, T, which):
    """Any of x, dy (inputs) and y, dx (outputs) in pinned host memory, staged tile by tile,
    give bitwise the device-resident results."""
    mw = MLP_WORKLOADS["mlp_small"].with_(S=S, seed=50 + S)
    x, w_gu, w_d, dy = make_mlp_inputs(mw, "cpu")
    ref = _run(x, w_gu, w_d, dy, T)
    wg, wd = w_gu.cuda(), w_d.cuda()
    xi = _pinned(x) if which in ("all", "x") else x.cuda()
    dyi = _pinned(dy) if which in ("all", "dy") else dy.cuda()
    out_host = which in ("all", "outputs")
    y = up.mlp_forward(xi, wg, wd, seq_tile=T, y_on_host=out_host)
    dx, dw_gu, dw_d = up.mlp_backward(xi, wg, wd, dyi, seq_tile=T, dx_on_host=out_host)
    up.upipe_sync_status()
    assert y.is_cuda != out_host and dx.is_cuda != out_host
    assert torch.equal(y.cpu(), ref[0].cpu()) and torch.equal(dx.cpu(), ref[1].cpu())
    assert torch.equal(dw_gu, ref[2]) and torch.equal(dw_d, ref[3])


def test_mlp_host_activations_need_the_staging_workspace():
    mw = MLP_WORKLOADS["mlp_small"].with_(S=512)
    x, w_gu, w_d, _ = make_mlp_inputs(mw, "cpu")
    dev_ws = up.upipe_mlp_workspace_bytes(512, mw.Dm, mw.F, 256, up.UPIPE_PASS_FWD)
    ws = torch.empty(dev_ws, dtype=torch.uint8, device="cuda")
    with pytest.raises(up.UpipeError) as e:
        up.mlp_forward(_pinned(x), w_gu.cuda(), w_d.cuda(), seq_tile=256, workspace=ws)
    assert e.value.status == up.UPIPE_ERR_WORKSPACE_TOO_SMALL


@pytest.mark.slow
def test_mlp_full_size_sampled():
    """The measured configuration (S = 128K, Dm 4096, F 14336, tiles of 8192) in the launch
    sequence the benchmark times. y and dx at sampled tokens are checked exactly against the
    oracle (each needs only its own token). The weight gradients need every token; they are
    checked exactly with an upstream gradient that is zero except at the sampled tokens."""
    mw = MLP_WORKLOADS["llama8b_mlp_s128k"]
    x, w_gu, w_d, dy = make_mlp_inputs(mw)
    rows = [0, 1, 8191, 8192, 65537, 100000, mw.S - 1]
    y = up.mlp_forward(x, w_gu, w_d, seq_tile=mw.seq_tile)
    dx, dw_gu, dw_d = up.mlp_backward(x, w_gu, w_d, dy, seq_tile=mw.seq_tile)
    up.upipe_sync_status()
    Wgu = w_gu.float().cpu().numpy().astype(np.float64)
    Wd = w_d.float().cpu().numpy().astype(np.float64)
    ry, rdx = oracle.mlp_rows_ref(x, Wgu, Wd, dy, rows)
    assert rel_fro(to_np(y[rows]), ry) <= REL_FRO
    assert rel_fro(to_np(dx[rows]), rdx) <= REL_FRO
    assert torch.isfinite(dw_gu).all() and torch.isfinite(dw_d).all()

    dys = torch.zeros_like(dy)
    dys[rows] = dy[rows]
    dx2, dw_gu2, dw_d2 = up.mlp_backward(x, w_gu, w_d, dys, seq_tile=mw.seq_tile)
    up.upipe_sync_status()
    gen = torch.Generator().manual_seed(7)
    gr = sorted(set(torch.randint(0, 2 * mw.F, (1024,), generator=gen).tolist()) | {0, mw.F,
                                                                                  2 * mw.F - 1})
    dr = sorted(set(torch.randint(0, mw.Dm, (512,), generator=gen).tolist()) | {0, mw.Dm - 1})
    _, rdx2, rdg, rdd = oracle.mlp_rows_ref(x, Wgu, Wd, dys, rows, gu_rows=gr, d_rows=dr)
    assert rel_fro(to_np(dx2[rows]), rdx2) <= REL_FRO
    others = torch.ones(mw.S, dtype=torch.bool, device=dx2.device)
    others[rows] = False
    assert int(torch.count_nonzero(dx2[others])) == 0
    assert rel_fro(to_np(dw_gu2[gr]), rdg) <= REL_FRO
    assert rel_fro(to_np(dw_d2[dr]), rdd) <= REL_FRO
