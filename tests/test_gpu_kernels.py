"""GPU checks of the building blocks under the attention kernels (needs an sm_103a GPU):
the tensor-core tile path in every operand layout the kernels use, the bounded device wait,
and the layout gathers."""
import pytest
import torch

import context_parallelism_gb300 as up

pytestmark = pytest.mark.gpu


def _logical(a, b, N, K, a_mn, b_mn):
    A = (a[:K, :].t() if a_mn else a[:, :K]).float()
    Bm = (b[:K, :N].t() if b_mn else b[:N, :K]).float()
    return A @ Bm.t()


LAYOUTS = [  # (a_mn, b_mn, a_manual): the combinations the forward and backward kernels issue
    (0, 0, 0),  # S = Q K^T, S^T = K Q^T, dP^T = V dO^T
    (0, 1, 0),  # O += P V, dV += P^T dO, dK += dS^T Q (A from TMA here)
    (0, 1, 1),  # the same with A written by the kernels' own swizzled stores (P, P^T, dS^T)
    (0, 0, 1),
    (1, 1, 0),  # dQ = dS K (A = dS^T tile read MN-major)
    (1, 0, 0),
    (0, 1, 2),  # A from tensor memory (P kept in TMEM), B MN-major
    (0, 0, 2),
]


@pytest.mark.parametrize("N,K", [(128, 128), (64, 64), (128, 64), (64, 128)])
@pytest.mark.parametrize("a_mn,b_mn,a_manual", LAYOUTS)
def test_umma_tile(N, K, a_mn, b_mn, a_manual):
    g = torch.Generator(device="cuda").manual_seed(1000 + N + K + 10 * a_mn + 100 * b_mn)
    a = torch.randn((128, 128), generator=g, device="cuda").to(torch.bfloat16)
    b = torch.randn((128, 128), generator=g, device="cuda").to(torch.bfloat16)
    c = torch.full((128, N), float("nan"), device="cuda")
    up.upipe_selftest_umma(a, b, c, N, K, a_mn, b_mn, a_manual)
    up.upipe_sync_status()
    want = _logical(a, b, N, K, a_mn, b_mn)
    if not torch.allclose(c, want, rtol=1e-4, atol=1e-3):
        diag = []
        if a_mn or b_mn:  # report whether the swapped offsets would have matched
            c2 = torch.full((128, N), float("nan"), device="cuda")
            up.upipe_selftest_umma(a, b, c2, N, K, a_mn, b_mn, a_manual, lbo=1024, sbo=16384)
            up.upipe_sync_status()
            diag.append(f"swapped lbo/sbo matches: {torch.allclose(c2, want, rtol=1e-4, atol=1e-3)}")
        err = (c - want).abs().max().item()
        pytest.fail(f"tile mismatch max err {err}; " + "; ".join(diag))


def test_bounded_wait_reports_timeout_and_context_survives():
    up.upipe_sync_status()
    up.upipe_selftest_wait_timeout(20000)  # 20 ms on a barrier nothing completes
    with pytest.raises(up.UpipeError) as ei:
        up.upipe_sync_status()
    assert ei.value.status == up.UPIPE_ERR_TIMEOUT
    up.upipe_sync_status()  # cleared
    # the context is still usable: a small attention call runs and is finite
    q = torch.randn((1, 256, 4, 64), device="cuda").to(torch.bfloat16)
    o, lse = up.attention_forward(q, q, q, causal=True)
    up.upipe_sync_status()
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


@pytest.mark.parametrize("B,S,H,D,h0,hn", [(2, 333, 8, 128, 2, 3), (1, 128, 4, 64, 0, 4),
                                           (3, 77, 32, 128, 24, 8)])
def test_layout_gather_scatter_bitwise(B, S, H, D, h0, hn):
    src = torch.randn((B, S, H, D), device="cuda").to(torch.bfloat16)
    dst = torch.empty((B, hn, S, D), device="cuda", dtype=torch.bfloat16)
    up.upipe_seq_to_head_major(src, dst, B, S, H, D, h0, hn)
    torch.cuda.synchronize()
    assert torch.equal(dst, src[:, :, h0:h0 + hn].permute(0, 2, 1, 3))
    back = torch.zeros_like(src)
    up.upipe_head_to_seq_major(dst, back, B, S, H, D, h0, hn)
    torch.cuda.synchronize()
    assert torch.equal(back[:, :, h0:h0 + hn], src[:, :, h0:h0 + hn])
    assert torch.count_nonzero(back[:, :, :h0]) == 0
    assert torch.count_nonzero(back[:, :, h0 + hn:]) == 0
