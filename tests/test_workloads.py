"""The seeded input recipes (workloads/__init__.py) do what the design notes say: the same seed
gives the same bytes, the draws have the stated distributions and structure, and the recipes
hold no method arithmetic (inputs only). CPU only."""
import math

import torch

from workloads import (LOSS_WORKLOADS, MLP_WORKLOADS, WORKLOADS, make_inputs, make_loss_inputs,
                       make_mlp_inputs, peaky_rows)


def test_attention_recipe_is_seeded_bf16_normal():
    w = WORKLOADS["llama8b_s8k"].with_(S=2048)
    a = make_inputs(w, "cpu")
    b = make_inputs(w, "cpu")
    for x, y in zip(a, b):
        assert x.dtype == torch.bfloat16 and torch.equal(x, y)
    q = a[0].float()
    assert abs(q.mean().item()) < 0.01 and abs(q.std().item() - 1.0) < 0.01
    assert tuple(a[0].shape) == (w.B, w.S, w.Hq, w.D) and tuple(a[1].shape) == (w.B, w.S, w.Hkv, w.D)


def test_peaky_recipe_scales_one_percent_of_key_rows_by_eight():
    w = WORKLOADS["gqa32b_s256k_peaky"].with_(S=4096, gen_device="cpu")
    q, k, v, do = make_inputs(w, "cpu")
    plain = make_inputs(w.with_(peaky_frac=0.0), "cpu")[1]
    rows = peaky_rows(w, "cpu")
    assert len(rows) == math.floor(0.01 * w.S) == len(set(rows.tolist()))
    assert torch.equal(k[:, rows].float(), plain[:, rows].float() * 8)
    keep = torch.ones(w.S, dtype=torch.bool)
    keep[rows] = False
    assert torch.equal(k[:, keep], plain[:, keep])


def test_loss_recipe():
    lw = LOSS_WORKLOADS["readout_small"].with_(S=8192, V=2048, Dm=512)
    h, w, t, g = make_loss_inputs(lw, "cpu")
    h2, w2, t2, g2 = make_loss_inputs(lw, "cpu")
    assert torch.equal(h, h2) and torch.equal(w, w2) and torch.equal(t, t2) and torch.equal(g, g2)
    assert h.dtype == w.dtype == torch.bfloat16 and t.dtype == torch.int64
    assert abs(h.float().std().item() - 1.0) < 0.01
    assert abs(w.float().std().item() - lw.w_std / math.sqrt(lw.Dm)) < 0.002
    ignored = (t < 0).float().mean().item()
    assert abs(ignored - lw.ignore_frac) < 0.01
    assert int(t.max()) < lw.V and set(t[t < 0].tolist()) <= {-1}
    n = int((t >= 0).sum())
    assert torch.all(g == 1.0 / n)  # the mean over counted tokens


def test_mlp_recipe():
    mw = MLP_WORKLOADS["mlp_small"].with_(S=4096, Dm=256, F=512)
    x, w_gu, w_d, dy = make_mlp_inputs(mw, "cpu")
    again = make_mlp_inputs(mw, "cpu")
    assert all(torch.equal(a, b) for a, b in zip((x, w_gu, w_d, dy), again))
    assert tuple(w_gu.shape) == (2 * mw.F, mw.Dm) and tuple(w_d.shape) == (mw.Dm, mw.F)
    assert abs(w_gu.float().std().item() - 1 / math.sqrt(mw.Dm)) < 0.002
    assert abs(w_d.float().std().item() - 1 / math.sqrt(mw.F)) < 0.002
    assert abs(dy.float().std().item() - 1.0) < 0.02


def test_flop_conventions():
    w = WORKLOADS["llama8b_s128k"]
    assert w.flops_fwd() == 4 * w.B * w.Hq * w.D * w.S * w.S / 2
    assert w.flops_bwd() == 2.5 * w.flops_fwd()
    assert w.with_(causal=False).flops_fwd() == 2 * w.flops_fwd()
    lw = LOSS_WORKLOADS["llama8b_readout_s128k"]
    assert lw.flops_fwd() == 2 * lw.S * lw.V * lw.Dm and lw.flops_bwd() == 3 * lw.flops_fwd()
    mw = MLP_WORKLOADS["llama8b_mlp_s128k"]
    assert mw.flops_fwd() == 6 * mw.S * mw.Dm * mw.F and mw.flops_bwd() == 16 * mw.S * mw.Dm * mw.F
