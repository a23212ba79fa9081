"""Element-by-element parity of the CUDA forward and backward (through the C ABI) with the fp64
oracle, on inputs small enough for the oracle to run in full: the two small workloads, ragged
sequence lengths, several trunks, non-causal attention, GQA ratios, and K/V staged from
pinned host memory. Needs an sm_103a GPU."""
import pytest
import torch

import context_parallelism_gb300 as up
import oracle
from tests._parity import (GRAD_REL_FRO, LSE_MAX_ABS, O_MAX_ABS, check_full, gpu_fwd_bwd,
                           max_abs, pinned_copy, rel_fro, to_np)
from workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


def _oracle(q, k, v, do, causal):
    o, lse, dq, dk, dv = oracle.attn_bwd_ref(q, k, v, do, causal=causal)
    return o, lse, dq, dk, dv


@pytest.mark.parametrize("name", ["mha_s512_d64", "llama8b_s8k"])
def test_small_workloads_full(name):
    w = WORKLOADS[name]
    q, k, v, do = make_inputs(w)  # CPU, seeded
    ref = _oracle(q, k, v, do, w.causal)
    qg, kg, vg, dog = (t.cuda() for t in (q, k, v, do))
    gpu = gpu_fwd_bwd(qg, kg, vg, dog, w.causal, w.head_chunk, w.seq_trunk)
    check_full(gpu, ref, name)


CASES = [
    # B, S, Hq, Hkv, D, causal, head_chunk, seq_trunk, kv_on_host
    (2, 1000, 8, 2, 128, True, 4, 256, False),   # ragged S, 4 trunks (last ragged), 2 groups
    (2, 1000, 8, 2, 128, True, 8, 1000, False),  # ragged S, one trunk, one group
    (1, 1000, 8, 2, 128, False, 4, 384, False),  # non-causal, ragged trunks
    (2, 777, 4, 4, 64, True, 2, 256, False),     # D = 64, MHA, ragged
    (1, 1000, 8, 2, 128, True, 4, 256, True),    # K/V in pinned host memory, double buffer
    (1, 640, 8, 1, 128, True, 8, 128, True),     # G = 8, many small host trunks
    (1, 129, 4, 2, 64, True, 2, 128, False),     # one full tile + 1-row tail
    (1, 1, 2, 1, 128, True, 2, 1, False),        # a single token
    (3, 300, 6, 3, 128, False, 6, 300, False),   # odd head counts, non-causal
    (1, 900, 8, 2, 128, False, 4, 256, True),    # host K/V, non-causal: every trunk pair
    (2, 700, 4, 2, 64, True, 2, 256, True),      # host K/V, D = 64, batch 2, ragged
]


@pytest.mark.parametrize("B,S,Hq,Hkv,D,causal,hc,T,kv_host", CASES)
def test_parity_cases(B, S, Hq, Hkv, D, causal, hc, T, kv_host):
    w = WORKLOADS["llama8b_s8k"].with_(B=B, S=S, Hq=Hq, Hkv=Hkv, D=D, causal=causal,
                                       seed=7 + S + Hq)
    q, k, v, do = make_inputs(w, "cpu")
    ref = _oracle(q, k, v, do, causal)
    qg, dog = q.cuda(), do.cuda()
    if kv_host:
        kg, vg = pinned_copy(k), pinned_copy(v)
    else:
        kg, vg = k.cuda(), v.cuda()
    gpu = gpu_fwd_bwd(qg, kg, vg, dog, causal, hc, T)
    # one token: the exact dQ and dK vanish identically, so their error is held to an
    # absolute RMS of 1e-3 instead of a relative one
    check_full(gpu, ref, f"{B}x{S}x{Hq}/{Hkv}x{D} causal={causal} hc={hc} T={T} host={kv_host}",
               grad_floor_rms=1e-3 if S == 1 else 0.0)


def test_head_chunk_does_not_change_forward_bits():
    """Grouping heads changes memory, not the per-head computation: O and LSE are bitwise
    identical for every head_chunk at a fixed trunk length."""
    w = WORKLOADS["llama8b_s8k"].with_(S=2048, seed=31)
    q, k, v, _ = (t.cuda() for t in make_inputs(w, "cpu"))
    outs = []
    for hc in (4, 8, 16, 32):
        o, lse = up.attention_forward(q, k, v, causal=True, head_chunk=hc, seq_trunk=2048)
        up.upipe_sync_status()
        outs.append((o, lse))
    for o, lse in outs[1:]:
        assert torch.equal(o, outs[0][0])
        assert torch.equal(lse, outs[0][1])


def test_trunk_length_sweep_matches_oracle():
    """Q trunk m folding KV trunks 0..m over several launches gives the untrunked result."""
    w = WORKLOADS["llama8b_s8k"].with_(S=2048, seed=32)
    q, k, v, do = make_inputs(w, "cpu")
    ref = _oracle(q, k, v, do, True)
    qg, kg, vg, dog = (t.cuda() for t in (q, k, v, do))
    for T in (256, 512, 1024, 2048):
        gpu = gpu_fwd_bwd(qg, kg, vg, dog, True, 8, T)
        check_full(gpu, ref, f"T={T}")


def test_host_kv_equals_device_kv_forward():
    """Staging K/V trunks from pinned host memory changes where bytes come from, not the
    arithmetic: the forward is bitwise identical to the device-resident run."""
    w = WORKLOADS["llama8b_s8k"].with_(S=1536, seed=33)
    q, k, v, _ = make_inputs(w, "cpu")
    qg = q.cuda()
    o1, l1 = up.attention_forward(qg, k.cuda(), v.cuda(), causal=True, head_chunk=8, seq_trunk=512)
    o2, l2 = up.attention_forward(qg, pinned_copy(k), pinned_copy(v), causal=True, head_chunk=8,
                                  seq_trunk=512)
    up.upipe_sync_status()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("B,D,T", [(1, 128, 512), (2, 64, 384)])
def test_host_dkdv_equals_device_dkdv(B, D, T):
    """With K/V and dK/dV all in pinned host memory, each trunk's dK/dV is copied out of a
    device slot as the next trunk computes. dK/dV accumulate in the same order as in the
    device run, so they are bitwise identical; dQ (reduced with atomics) is checked against
    the oracle."""
    w = WORKLOADS["llama8b_s8k"].with_(B=B, S=1400, D=D, Hq=8, Hkv=2, seed=37)
    q, k, v, do = make_inputs(w, "cpu")
    qg, dog = q.cuda(), do.cuda()
    o, lse = up.attention_forward(qg, k.cuda(), v.cuda(), causal=True, head_chunk=4, seq_trunk=T)
    _, dk1, dv1 = up.attention_backward(qg, k.cuda(), v.cuda(), o, lse, dog, causal=True,
                                        head_chunk=4, seq_trunk=T)
    dq2, dk2, dv2 = up.attention_backward(qg, pinned_copy(k), pinned_copy(v), o, lse, dog,
                                          causal=True, head_chunk=4, seq_trunk=T,
                                          dkdv_on_host=True)
    up.upipe_sync_status()
    assert not dk2.is_cuda and dk2.is_pinned()
    assert torch.equal(dk1.cpu(), dk2) and torch.equal(dv1.cpu(), dv2)
    ref = oracle.attn_bwd_ref(*(t.double().numpy() for t in (q, k, v, do)), causal=True)
    check_full((o, lse, dq2, dk2, dv2), ref, "host dk/dv")


def test_host_dkdv_needs_host_kv_and_matching_placement():
    w = WORKLOADS["mha_s512_d64"]
    q, k, v, do = (t.cuda() for t in make_inputs(w, "cpu"))
    o, lse = up.attention_forward(q, k, v)
    up.upipe_sync_status()
    B, S, H, D = q.shape
    dq = torch.empty_like(q)
    hk = torch.empty((B, S, H, D), dtype=q.dtype, pin_memory=True)
    dv_dev = torch.empty_like(k)
    ws = torch.empty(up.upipe_workspace_bytes(B, S, H, H, D, 1, H, S, up.UPIPE_PASS_BWD, 1),
                     dtype=torch.uint8, device="cuda")
    n0 = up.upipe_launch_count()
    for kk, vv, dk_, dv_ in ((k, v, hk, dv_dev),          # mixed dk/dv placement
                             (k, v, hk, hk.clone().pin_memory()),  # host dk/dv, device k/v
                             (pinned_copy(k.cpu()), pinned_copy(v.cpu()), hk, dv_dev)):
        with pytest.raises(up.UpipeError) as ei:
            up.upipe_attn_bwd(q, kk, vv, o, lse, do, dq, dk_, dv_, B, S, H, H, D, 1, H, S, ws,
                              None)
        assert ei.value.status == up.UPIPE_ERR_INVALID_ARG
    assert up.upipe_launch_count() == n0


@pytest.mark.parametrize("D,host_kv", [(128, False), (128, True), (64, False)])
def test_prefill_forward_without_lse(D, host_kv):
    """A prefill (inference) forward passes no lse buffer: the same kernels run, only o is
    written. o matches the fp64 oracle within the forward tolerance, and is bitwise the o of
    the training forward (several trunks, ragged tail)."""
    w = WORKLOADS["llama8b_s8k"].with_(S=1100, D=D, Hq=8, Hkv=2, seed=38)
    q, k, v, _ = make_inputs(w, "cpu")
    qg = q.cuda()
    kk, vv = (pinned_copy(k), pinned_copy(v)) if host_kv else (k.cuda(), v.cuda())
    o1, _ = up.attention_forward(qg, kk, vv, causal=True, head_chunk=4, seq_trunk=256)
    o2, l2 = up.attention_forward(qg, kk, vv, causal=True, head_chunk=4, seq_trunk=256,
                                  with_lse=False)
    up.upipe_sync_status()
    assert l2 is None
    ro, _ = oracle.attn_fwd_ref(q, k, v, causal=True)
    err = max_abs(to_np(o2), ro)
    assert err <= O_MAX_ABS, err
    assert torch.equal(o1, o2)


def test_rising_scores_force_rescales():
    """The last head-dim channel carries a ramp: q's is 2 and key j's is 0.28*j, so every
    score rises by about 0.05 per key (on top of the random part). The row maximum then climbs
    by ~9 log2 units per 128-key tile, so the forward's running maximum moves in nearly every
    tile, also between the two 64-column halves (the exact power-of-two rescale of O, the row
    sum and the first half's P), while each row's softmax stays ~20 keys wide."""
    w = WORKLOADS["llama8b_s8k"].with_(S=1536, Hq=8, Hkv=2, seed=39)
    q, k, v, do = make_inputs(w, "cpu")
    q[..., -1] = 2.0
    k[..., -1] = (0.28 * torch.arange(w.S, dtype=torch.float32)).view(1, w.S, 1).to(torch.bfloat16)
    ref = _oracle(q, k, v, do, True)
    o, lse, dq, dk, dv = gpu_fwd_bwd(q.cuda(), k.cuda(), v.cuda(), do.cuda(), True, 4, 512)
    # dQ's ramp channel is sum_j dS_ij * 0.28 j with sum_j dS_ij = 0: rounding dS to bf16 for
    # the dQ MMA (as any bf16 attention backward does) leaves ~3 % there even with everything
    # else exact, so that one channel is left out of the dQ check.
    dq_ref = ref[2][..., :-1]
    check_full((o, lse, dq[..., :-1], dk, dv), (ref[0], ref[1], dq_ref, ref[3], ref[4]),
               "rising scores")


@pytest.mark.parametrize("D", [128, 64])
def test_constant_values_come_back_exactly_with_peaky_keys(D):
    """With V the same vector at every position of a kv-head, every softmax row averages that
    vector: O = V exactly, whatever the weights (the oracle's constant-V pin). The kernel
    divides the P.V product by the sum of the same bf16-rounded weights it multiplied, so it
    returns V bit for bit here, also on rows carried by one of the x8 keys, where the dominant
    weight is far from a power of two."""
    w = WORKLOADS["gqa32b_s256k_peaky"].with_(S=1000, Hq=8, Hkv=2, D=D, seed=43)
    q, k, v, _ = make_inputs(w, "cpu")
    v = v[:, :1].expand_as(v).contiguous()
    o, _ = up.attention_forward(q.cuda(), k.cuda(), v.cuda(), causal=True, head_chunk=4,
                                seq_trunk=1000)
    up.upipe_sync_status()
    want = v.repeat_interleave(w.Hq // w.Hkv, dim=2)
    assert torch.equal(o.cpu(), want)


@pytest.mark.parametrize("q_host,o_host,kv_host", [(True, False, False), (False, True, False),
                                                     (True, True, True)])
def test_host_q_and_o_forward(q_host, o_host, kv_host):
    """q read from and o written to pinned host memory, one head group at a time on the copy
    stream (the next group's Q staged and the previous group's O copied out while a group
    computes): o and lse match the fp64 oracle, and (the same kernels) are bitwise those of
    the device-resident run.
    Three head groups exercise both staging buffers and their reuse."""
    w = WORKLOADS["llama8b_s8k"].with_(S=1100, Hq=12, Hkv=3, seed=40)
    q, k, v, _ = make_inputs(w, "cpu")
    o1, l1 = up.attention_forward(q.cuda(), k.cuda(), v.cuda(), causal=True, head_chunk=4,
                                  seq_trunk=256)
    qq = pinned_copy(q) if q_host else q.cuda()
    kk, vv = (pinned_copy(k), pinned_copy(v)) if kv_host else (k.cuda(), v.cuda())
    o2, l2 = up.attention_forward(qq, kk, vv, causal=True, head_chunk=4, seq_trunk=256,
                                  o_on_host=o_host)
    up.upipe_sync_status()
    assert (not o2.is_cuda) == o_host
    ro, rl = oracle.attn_fwd_ref(q, k, v, causal=True)
    err_o, err_l = max_abs(to_np(o2), ro), max_abs(to_np(l2), rl)
    assert err_o <= O_MAX_ABS and err_l <= LSE_MAX_ABS, (err_o, err_l)
    assert torch.equal(o1.cpu(), o2.cpu()) and torch.equal(l1, l2)


@pytest.mark.parametrize("host", [("q", "o", "dout", "dq"), ("o",), ("dout", "dq"), ("q",)])
def test_host_activations_backward(host):
    """q, o, dout read from and dq written to pinned host memory, head group by head group:
    dK and dV accumulate in the same order as the device-resident run (bitwise equal); dQ,
    reduced with atomics, is checked against the oracle. Three head groups and host K/V with
    host dK/dV in the full case exercise every staging buffer and the shared copy stream."""
    w = WORKLOADS["llama8b_s8k"].with_(S=900, Hq=12, Hkv=3, seed=41)
    q, k, v, do = make_inputs(w, "cpu")
    full = len(host) == 4
    kg, vg = (pinned_copy(k), pinned_copy(v)) if full else (k.cuda(), v.cuda())
    o, lse = up.attention_forward(q.cuda(), k.cuda(), v.cuda(), causal=True, head_chunk=4,
                                  seq_trunk=256)
    _, dk1, dv1 = up.attention_backward(q.cuda(), k.cuda(), v.cuda(), o, lse, do.cuda(),
                                        causal=True, head_chunk=4, seq_trunk=256)
    qq = pinned_copy(q) if "q" in host else q.cuda()
    oo = pinned_copy(o.cpu()) if "o" in host else o
    dd = pinned_copy(do) if "dout" in host else do.cuda()
    dq2, dk2, dv2 = up.attention_backward(qq, kg, vg, oo, lse, dd, causal=True, head_chunk=4,
                                          seq_trunk=256, dkdv_on_host=full,
                                          dq_on_host="dq" in host)
    up.upipe_sync_status()
    assert (not dq2.is_cuda) == ("dq" in host)
    assert torch.equal(dk1.cpu(), dk2.cpu()) and torch.equal(dv1.cpu(), dv2.cpu())
    # O and LSE come from the ordinary forward (checked elsewhere); the gradients are this
    # call's output
    ref = _oracle(q, k, v, do, True)
    for name, got, want in (("dq", dq2, ref[2]), ("dk", dk2, ref[3]), ("dv", dv2, ref[4])):
        err = rel_fro(to_np(got), want)
        assert err <= GRAD_REL_FRO, (host, name, err)


def test_forward_is_deterministic():
    w = WORKLOADS["llama8b_s8k"].with_(S=1024, seed=34)
    q, k, v, _ = (t.cuda() for t in make_inputs(w, "cpu"))
    a = up.attention_forward(q, k, v, head_chunk=8, seq_trunk=512)
    b = up.attention_forward(q, k, v, head_chunk=8, seq_trunk=512)
    up.upipe_sync_status()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_pageable_host_kv_rejected_without_launch():
    w = WORKLOADS["mha_s512_d64"]
    q, k, v, _ = make_inputs(w, "cpu")
    n0 = up.upipe_launch_count()
    with pytest.raises(up.UpipeError) as ei:
        up.attention_forward(q.cuda(), k, v)  # pageable CPU tensors
    assert ei.value.status == up.UPIPE_ERR_INVALID_ARG
    assert up.upipe_launch_count() == n0


def test_workspace_too_small_rejected():
    w = WORKLOADS["mha_s512_d64"]
    q, k, v, _ = (t.cuda() for t in make_inputs(w, "cpu"))
    need = up.upipe_workspace_bytes(1, 512, 4, 4, 64, 1, 4, 512, up.UPIPE_PASS_FWD, 0)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((1, 4, 512), device="cuda")
    with pytest.raises(up.UpipeError) as ei:
        up.upipe_attn_fwd(q, k, v, o, lse, 1, 512, 4, 4, 64, 1, 4, 512, ws, need - 256)
    assert ei.value.status == up.UPIPE_ERR_WORKSPACE_TOO_SMALL


def test_no_device_allocation_per_call():
    """The caller's workspace is the only device memory a call uses: torch's allocator and the
    device's free memory are unchanged across calls after the first."""
    w = WORKLOADS["llama8b_s8k"].with_(S=1024, seed=35)
    q, k, v, do = (t.cuda() for t in make_inputs(w, "cpu"))
    gpu_fwd_bwd(q, k, v, do, True, 8, 512)  # first call creates the per-device state
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    o = torch.empty_like(q)
    lse = torch.empty((1, 32, 1024), device="cuda")
    need = up.upipe_workspace_bytes(1, 1024, 32, 8, 128, 1, 8, 512, up.UPIPE_PASS_FWD, 0)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        up.upipe_attn_fwd(q, k, v, o, lse, 1, 1024, 32, 8, 128, 1, 8, 512, ws)
    up.upipe_sync_status()
    free2, _ = torch.cuda.mem_get_info()
    assert free2 == free1
    assert free0 - free1 <= o.nbytes + lse.nbytes + ws.nbytes + (64 << 20)
