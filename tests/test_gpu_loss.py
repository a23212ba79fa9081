"""Parity of the sequence-tiled readout + cross-entropy loss (upipe_ce_fwd / upipe_ce_bwd,
through the C ABI) with the fp64 oracle. Needs an sm_103a GPU.

Tolerances, from the arithmetic: the logits are exact bf16 products summed in fp32 on the
tensor cores and the softmax uses ex2.approx (relative error < 2^-22), so loss and lse are
within a few 1e-6 of the exact values at these magnitudes (|lse| ~ 10): they are held to
max abs 1e-3. The backward rounds dlogits to bf16 (relative 2^-9 per element) before its two
GEMMs and dh to bf16 on output, so dh and dw carry a relative error of a few 2^-9 in the
Frobenius norm: held to 1e-2.
"""
import numpy as np
import pytest
import torch

import context_parallelism_gb300 as up
import oracle
from tests._parity import max_abs, rel_fro, to_np
from workloads import LOSS_WORKLOADS, make_loss_inputs

pytestmark = pytest.mark.gpu

LOSS_MAX_ABS = 1e-3
GRAD_REL_FRO = 1e-2


def _random_g(S, seed):
    gen = torch.Generator().manual_seed(seed)
    return (torch.randn(S, generator=gen) / S).float()


def _run(h, w, t, g, seq_tile):
    hg, wg, tg, gg = h.cuda(), w.cuda(), t.cuda(), g.cuda()
    loss, lse = up.ce_loss_forward(hg, wg, tg, seq_tile=seq_tile)
    dh, dw = up.ce_loss_backward(hg, wg, tg, lse, gg, seq_tile=seq_tile)
    up.upipe_sync_status()
    return loss, lse, dh, dw


CASES = [
    # S, Dm, V, seq_tile
    (1000, 256, 1088, 256),   # 4 tiles of tokens (last ragged), 5 vocabulary tiles (last 64)
    (1000, 256, 1088, 1024),  # one ragged tile of tokens
    (300, 64, 320, 128),      # Dm = one k block, ragged tokens and vocabulary
    (128, 128, 64, 128),      # one tile, a vocabulary narrower than a column tile
    (1, 64, 256, 128),        # a single token
    (2048, 512, 2048, 512),   # several full tiles each way
]


@pytest.mark.parametrize("S,Dm,V,T", CASES)
def test_loss_parity(S, Dm, V, T):
    lw = LOSS_WORKLOADS["readout_small"].with_(S=S, Dm=Dm, V=V, seq_tile=T, seed=30 + S + V)
    h, w, t, _ = make_loss_inputs(lw, "cpu")
    g = _random_g(S, lw.seed)
    rl, rs, rdh, rdw = oracle.ce_loss_bwd_ref(h, w, t, g)
    loss, lse, dh, dw = _run(h, w, t, g, T)
    tag = f"S={S} Dm={Dm} V={V} T={T}"
    assert max_abs(to_np(loss), rl) <= LOSS_MAX_ABS, tag
    assert max_abs(to_np(lse), rs) <= LOSS_MAX_ABS, tag
    assert rel_fro(to_np(dh), rdh) <= GRAD_REL_FRO, tag
    assert rel_fro(to_np(dw), rdw) <= GRAD_REL_FRO, tag
    ign = (t < 0).nonzero().flatten()
    assert torch.all(loss.cpu()[ign] == 0) and torch.all(dh.cpu()[ign] == 0), tag


def test_loss_small_workload_mean_reduction():
    lw = LOSS_WORKLOADS["readout_small"]
    h, w, t, g = make_loss_inputs(lw, "cpu")
    rl, rs, rdh, rdw = oracle.ce_loss_bwd_ref(h, w, t, g)
    loss, lse, dh, dw = _run(h, w, t, g, lw.seq_tile)
    assert max_abs(to_np(loss), rl) <= LOSS_MAX_ABS
    assert abs(float((loss.double() * g.cuda().double()).sum()) - float(np.dot(rl, to_np(g)))) <= 1e-4
    assert rel_fro(to_np(dh), rdh) <= GRAD_REL_FRO
    assert rel_fro(to_np(dw), rdw) <= GRAD_REL_FRO


def test_tiling_does_not_change_the_result():
    lw = LOSS_WORKLOADS["readout_small"].with_(S=1024, V=1024, seed=41)
    h, w, t, _ = make_loss_inputs(lw, "cpu")
    g = _random_g(lw.S, 41)
    a = _run(h, w, t, g, 128)
    b = _run(h, w, t, g, 1024)
    # every token's loss and dh come from its own row alone: identical bits
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    # dw sums over the tiles in another order
    assert rel_fro(to_np(a[3]), to_np(b[3])) <= 1e-5


def test_target_outside_vocabulary_is_nan():
    lw = LOSS_WORKLOADS["readout_small"].with_(S=256, V=320, Dm=64, seed=43)
    h, w, t, _ = make_loss_inputs(lw, "cpu")
    t[5] = lw.V  # out of range
    t[6] = -1
    loss, lse, _, _ = _run(h, w, t, _random_g(lw.S, 43), 128)
    loss = loss.cpu()
    assert torch.isnan(loss[5]) and loss[6] == 0
    keep = torch.ones(lw.S, dtype=torch.bool)
    keep[5] = False
    assert torch.isfinite(loss[keep]).all() and torch.isfinite(lse.cpu()).all()


def test_loss_rejects_bad_shapes_and_small_workspace():
    h = torch.zeros((256, 96), dtype=torch.bfloat16, device="cuda")  # Dm % 64 != 0
    w = torch.zeros((128, 96), dtype=torch.bfloat16, device="cuda")
    t = torch.zeros(256, dtype=torch.int64, device="cuda")
    with pytest.raises(up.UpipeError) as e:
        up.ce_loss_forward(h, w, t, seq_tile=128)
    assert e.value.status == up.UPIPE_ERR_UNSUPPORTED
    h = torch.zeros((256, 64), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((128, 64), dtype=torch.bfloat16, device="cuda")
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(up.UpipeError) as e:
        up.ce_loss_forward(h, w, t, seq_tile=128, workspace=small)
    assert e.value.status == up.UPIPE_ERR_WORKSPACE_TOO_SMALL


@pytest.mark.parametrize("S,T", [(1000, 256), (384, 128), (100, 128)])
def test_host_activations_equal_device(S, T):
    """h in pinned host memory (staged tile by tile) and dh returned to pinned host memory
    give bitwise the results of device-resident h and dh: the staging moves bytes only."""
    lw = LOSS_WORKLOADS["readout_small"].with_(S=S, seed=47 + S)
    h, w, t, _ = make_loss_inputs(lw, "cpu")
    g = _random_g(S, lw.seed)
    ref = _run(h, w, t, g, T)
    wg, tg, gg = w.cuda(), t.cuda(), g.cuda()
    hh = torch.empty(h.shape, dtype=h.dtype, pin_memory=True)
    hh.copy_(h)
    loss, lse = up.ce_loss_forward(hh, wg, tg, seq_tile=T)
    dh, dw = up.ce_loss_backward(hh, wg, tg, lse, gg, seq_tile=T, dh_on_host=True)
    up.upipe_sync_status()
    assert not dh.is_cuda and dh.is_pinned()
    assert torch.equal(loss, ref[0]) and torch.equal(lse, ref[1])
    assert torch.equal(dh, ref[2].cpu()) and torch.equal(dw, ref[3])


@pytest.mark.parametrize("S,Dm,V,T,host", [(1000, 256, 1088, 256, False),
                                           (300, 64, 320, 128, False),
                                           (1000, 256, 1088, 256, True),
                                           (1, 64, 256, 128, False)])
def test_fused_forward_backward_equals_two_calls(S, Dm, V, T, host):
    """upipe_ce_fwd_bwd keeps the forward's fp32 logits instead of recomputing them: loss, lse,
    dh and dw are bitwise those of the two calls (and so within tolerance of the oracle)."""
    lw = LOSS_WORKLOADS["readout_small"].with_(S=S, Dm=Dm, V=V, seed=81 + S + V)
    h, w, t, _ = make_loss_inputs(lw, "cpu")
    g = _random_g(S, lw.seed)
    ref = _run(h, w, t, g, T)
    hi = h.cuda()
    if host:
        hi = torch.empty(h.shape, dtype=h.dtype, pin_memory=True)
        hi.copy_(h)
    got = up.ce_loss_fused(hi, w.cuda(), t.cuda(), g.cuda(), seq_tile=T, dh_on_host=host)
    up.upipe_sync_status()
    for a, b in zip(got, ref):
        assert torch.equal(a.cpu(), b.cpu())
    rl, rs, rdh, rdw = oracle.ce_loss_bwd_ref(h, w, t, g)
    assert max_abs(to_np(got[0]), rl) <= LOSS_MAX_ABS
    assert rel_fro(to_np(got[2]), rdh) <= GRAD_REL_FRO and rel_fro(to_np(got[3]), rdw) <= GRAD_REL_FRO


def test_fused_at_width_4096_and_full_vocabulary():
    """The measured shape's width and vocabulary over two 8192-token tiles: bitwise the two
    calls, and sampled tokens against the oracle."""
    lw = LOSS_WORKLOADS["llama8b_readout_s128k"].with_(S=16384)
    h, w, t, g = make_loss_inputs(lw)
    loss, lse = up.ce_loss_forward(h, w, t, seq_tile=8192)
    dh, dw = up.ce_loss_backward(h, w, t, lse, g, seq_tile=8192)
    got = up.ce_loss_fused(h, w, t, g, seq_tile=8192)
    up.upipe_sync_status()
    assert torch.equal(got[0], loss) and torch.equal(got[1], lse)
    assert torch.equal(got[2], dh) and torch.equal(got[3], dw)
    rows = [0, 8191, 8192, 16383]
    rl, rs, rdh = oracle.ce_rows_ref(h, w, t, g, rows)
    assert max_abs(to_np(got[0][rows]), rl) <= LOSS_MAX_ABS
    assert rel_fro(to_np(got[2][rows]), rdh) <= GRAD_REL_FRO


@pytest.mark.slow
def test_loss_full_size_sampled():
    """The measured configuration (S = 128K tokens, Dm 4096, V 128256, tiles of 8192) in the
    launch sequence the benchmark times. Each token's loss, lse and dh need only its own row
    of logits, so the oracle checks sampled tokens exactly. dw needs every token; it is
    checked (a) exactly, with an upstream gradient that is zero except at the sampled tokens
    (dw is then the sum of their rank-one terms), and (b) with the mean gradient, through the
    property that its rows sum to zero over the vocabulary."""
    lw = LOSS_WORKLOADS["llama8b_readout_s128k"]
    h, w, t, g = make_loss_inputs(lw)
    rows = [0, 1, 4095, 8191, 8192, 65537, 100000, lw.S - 1]
    t[rows[2]] = -1  # one ignored token among the samples
    loss, lse = up.ce_loss_forward(h, w, t, seq_tile=lw.seq_tile)
    dh, dw = up.ce_loss_backward(h, w, t, lse, g, seq_tile=lw.seq_tile)
    up.upipe_sync_status()
    W64 = w.float().cpu().numpy().astype(np.float64)  # exact upcast, reused by every check
    rl, rs, rdh = oracle.ce_rows_ref(h, W64, t, g, rows)
    assert max_abs(to_np(loss[rows]), rl) <= LOSS_MAX_ABS
    assert max_abs(to_np(lse[rows]), rs) <= LOSS_MAX_ABS
    assert rel_fro(to_np(dh[rows]), rdh) <= GRAD_REL_FRO
    col_sum = to_np(dw.sum(dim=0))
    assert np.linalg.norm(col_sum) <= 1e-2 * float(dw.double().norm())

    # sparse upstream gradient: dw = sum over the sampled tokens of g_i dlogits_i (x) h_i
    gs = torch.zeros_like(g)
    gen = torch.Generator().manual_seed(5)
    vals = torch.randn(len(rows), generator=gen).float()
    gs[rows] = vals.to(gs.device)
    dh2, dw2 = up.ce_loss_backward(h, w, t, lse, gs, seq_tile=lw.seq_tile)
    up.upipe_sync_status()
    tr = t[rows].cpu().tolist()
    gen_v = torch.Generator().manual_seed(6)
    vrows = sorted(set(torch.randint(0, lw.V, (2048,), generator=gen_v).tolist())
                   | {x for x in tr if x >= 0} | {0, lw.V - 1})
    _, _, rdh2, rdw2 = oracle.ce_rows_ref(h, W64, t, gs, rows, vocab_rows=vrows)
    assert rel_fro(to_np(dh2[rows]), rdh2) <= GRAD_REL_FRO
    others = torch.ones(lw.S, dtype=torch.bool, device=dh2.device)
    others[rows] = False
    assert int(torch.count_nonzero(dh2[others])) == 0
    assert rel_fro(to_np(dw2[vrows]), rdw2) <= GRAD_REL_FRO
