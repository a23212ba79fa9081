"""Host-side checks of the C ABI that need no GPU: the library loads, exports every function the
header declares, sizes workspaces by the documented formula, and rejects bad arguments before
touching the device."""
import ctypes
import os
import re

import pytest

import context_parallelism_gb300 as up
from workloads import WORKLOADS, WORKLOAD_ORDER

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "upipe.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(upipe_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("upipe_attn_fwd", "upipe_attn_bwd", "upipe_workspace_bytes",
                 "upipe_seq_to_head_major", "upipe_head_to_seq_major", "upipe_sync_status"):
        assert must in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(up.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in upipe.h but not exported"
    assert set(declared_functions()) == set(up.SIGNATURES), "binding and header disagree"


def _expected_ws(B, S, Hq, Hkv, D, hc, T, kv_host, act_host=False, causal=True):
    """The workspace arena as documented: every segment 256-byte aligned."""
    al = lambda x: (x + 255) // 256 * 256  # noqa: E731
    G = Hq // Hkv
    kc = hc // G
    T = min(T, S)
    S_pad = (S + 127) // 128 * 128
    ntr = (S + T - 1) // T
    qw = B * hc * S * D * 2
    kv = 4 * al(B * kc * T * D * 2) if kv_host else 2 * al(B * kc * S * D * 2)
    fwd = al(qw) + kv + (3 * al(qw) if act_host else 0)  # host q/o: Q buffer 2, 2 O stagings
    if kv_host and ntr > 1:  # running state of every query trunk, kept between launches
        fwd += al(B * hc * S_pad * D * 4) + al(B * hc * S_pad * 8)
    # host K/V: the backward also holds two dK and two dV trunk slots (used when dk/dv are
    # pinned host memory as well)
    dkdv = 4 * al(B * kc * T * D * 2) if kv_host else 0
    bwd = 2 * al(qw) + kv + dkdv + al(B * hc * S_pad * D * 4) + 2 * al(B * hc * S_pad * 4)
    rows = (T + 127) // 128 * 128 if kv_host else S_pad
    if causal and D == 128 and G > 1 and rows // 128 * B <= (512 if kv_host else 128):
        bwd += al(G * B * kc * rows * 2 * D * 4)  # split backward: G fp32 dK/dV shares
    if act_host:  # host q/o/dout/dq: Q and dO buffer 2, 2 head-major O copies, 2 dQ stagings
        bwd += 6 * al(qw)
    return fwd, bwd


@pytest.mark.parametrize("name", WORKLOAD_ORDER)
def test_workspace_matches_formula(name):
    w = WORKLOADS[name]
    fwd, bwd = _expected_ws(w.B, w.S, w.Hq, w.Hkv, w.D, w.head_chunk, w.seq_trunk, w.kv_on_host)
    args = (w.B, w.S, w.Hq, w.Hkv, w.D, 1, w.head_chunk, w.seq_trunk)
    assert up.upipe_workspace_bytes(*args, up.UPIPE_PASS_FWD, w.kv_on_host) == fwd
    assert up.upipe_workspace_bytes(*args, up.UPIPE_PASS_BWD, w.kv_on_host) == bwd
    assert up.upipe_workspace_bytes(*args, up.UPIPE_PASS_BOTH, w.kv_on_host) == max(fwd, bwd)


@pytest.mark.parametrize("name", WORKLOAD_ORDER)
@pytest.mark.parametrize("pass_", [0, 1])
def test_workspace_scales_with_head_chunk(name, pass_):
    """Chunked / unchunked workspace = head_chunk / Hq at the same trunk: the 32B-class
    workload with 8 of 64 heads per group is the 87.5% cut the UPipe abstract reports."""
    w = WORKLOADS[name]
    G = w.Hq // w.Hkv
    full = up.upipe_workspace_bytes(w.B, w.S, w.Hq, w.Hkv, w.D, 1, w.Hq, w.seq_trunk, pass_,
                                    w.kv_on_host)
    for hc in range(G, w.Hq + 1, G):
        if w.Hq % hc:
            continue
        part = up.upipe_workspace_bytes(w.B, w.S, w.Hq, w.Hkv, w.D, 1, hc, w.seq_trunk, pass_,
                                        w.kv_on_host)
        assert part * w.Hq <= full * hc + 256 * 16 * w.Hq
        assert abs(part / full - hc / w.Hq) < 1e-6
    if name == "gqa32b_s256k_peaky":
        part = up.upipe_workspace_bytes(w.B, w.S, w.Hq, w.Hkv, w.D, 1, 8, w.seq_trunk, pass_, 0)
        full = up.upipe_workspace_bytes(w.B, w.S, w.Hq, w.Hkv, w.D, 1, 64, w.seq_trunk, pass_, 0)
        assert part / full == pytest.approx(0.125, abs=1e-9)


@pytest.mark.parametrize("args", [
    (0, 512, 4, 4, 64, 1, 4, 512),      # B = 0
    (1, 0, 4, 4, 64, 1, 4, 512),        # S = 0
    (1, 512, 6, 4, 64, 1, 6, 512),      # Hq % Hkv
    (1, 512, 32, 8, 128, 1, 6, 512),    # head_chunk does not divide Hq
    (1, 512, 32, 8, 128, 1, 2, 512),    # head_chunk not a multiple of Hq/Hkv
    (1, 1024, 4, 4, 64, 1, 4, 300),     # seq_trunk < S and not a multiple of 128
    (1, 512, 4, 4, 64, 2, 4, 512),      # causal not 0/1
])
def test_workspace_zero_for_invalid(args):
    assert up.upipe_workspace_bytes(*args, 0, 0) == 0


FAKE = 1 << 20  # an aligned non-null address; validation must fail before it is dereferenced


@pytest.mark.parametrize("args,status", [
    ((1, 512, 6, 4, 64, 1, 6, 512), up.UPIPE_ERR_INVALID_ARG),
    ((1, 512, 32, 8, 128, 1, 2, 512), up.UPIPE_ERR_INVALID_ARG),
    ((1, 1024, 4, 4, 64, 1, 4, 300), up.UPIPE_ERR_INVALID_ARG),
    ((1, 512, 4, 4, 96, 1, 4, 512), up.UPIPE_ERR_UNSUPPORTED),
    ((1, 512, 4, 4, 256, 1, 4, 512), up.UPIPE_ERR_UNSUPPORTED),
])
def test_attention_calls_validate_before_device_access(args, status):
    B, S, Hq, Hkv, D, causal, hc, T = args
    st = up._lib.upipe_attn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, B, S, Hq, Hkv, D, causal, hc, T,
                                FAKE, 1 << 40, None)
    assert st == status, up.upipe_last_error_message()
    assert up.upipe_last_error_message()
    st = up._lib.upipe_attn_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, B, S, Hq,
                                Hkv, D, causal, hc, T, FAKE, 1 << 40, None)
    assert st == status


def test_null_and_misaligned_pointers_rejected():
    st = up._lib.upipe_attn_fwd(None, FAKE, FAKE, FAKE, FAKE, 1, 512, 4, 4, 64, 1, 4, 512, FAKE,
                                1 << 30, None)
    assert st == up.UPIPE_ERR_INVALID_ARG
    st = up._lib.upipe_attn_fwd(FAKE + 2, FAKE, FAKE, FAKE, FAKE, 1, 512, 4, 4, 64, 1, 4, 512,
                                FAKE, 1 << 30, None)
    assert st == up.UPIPE_ERR_INVALID_ARG
    st = up._lib.upipe_attn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 512, 4, 4, 64, 1, 4, 512,
                                FAKE + 16, 1 << 30, None)
    assert st == up.UPIPE_ERR_INVALID_ARG  # workspace must be 256-byte aligned
    st = up._lib.upipe_seq_to_head_major(FAKE, FAKE, 1, 16, 4, 64, 3, 2, None)
    assert st == up.UPIPE_ERR_INVALID_ARG  # head range outside H
    st = up._lib.upipe_seq_to_head_major(FAKE, FAKE, 1, 16, 4, 60, 0, 2, None)
    assert st == up.UPIPE_ERR_INVALID_ARG  # D % 8
    st = up._lib.upipe_selftest_wait_timeout(0, None)
    assert st == up.UPIPE_ERR_INVALID_ARG


def test_status_strings():
    for s in range(6):
        assert up.upipe_status_string(s).startswith("UPIPE_")
    assert up.upipe_status_string(99) == "UPIPE_ERR_UNKNOWN"


def test_launch_count_and_profile_read_without_gpu():
    assert up.upipe_launch_count() >= 0
    up.upipe_profile_enable(False)
    stats = up.upipe_profile_read()
    assert set(stats) == set(up.KERNEL_CLASSES)


@pytest.mark.parametrize("name", WORKLOAD_ORDER)
def test_workspace_with_host_activations(name):
    """UPIPE_HOST_ACT adds head-group-sized staging only, so the chunked/unchunked ratio holds."""
    w = WORKLOADS[name]
    mask = (up.UPIPE_HOST_KV if w.kv_on_host else 0) | up.UPIPE_HOST_ACT
    fwd, bwd = _expected_ws(w.B, w.S, w.Hq, w.Hkv, w.D, w.head_chunk, w.seq_trunk, w.kv_on_host,
                            act_host=True)
    args = (w.B, w.S, w.Hq, w.Hkv, w.D, 1, w.head_chunk, w.seq_trunk)
    assert up.upipe_workspace_bytes(*args, up.UPIPE_PASS_FWD, mask) == fwd
    assert up.upipe_workspace_bytes(*args, up.UPIPE_PASS_BWD, mask) == bwd
    full = up.upipe_workspace_bytes(w.B, w.S, w.Hq, w.Hkv, w.D, 1, w.Hq, w.seq_trunk,
                                    up.UPIPE_PASS_BOTH, mask)
    part = up.upipe_workspace_bytes(*args, up.UPIPE_PASS_BOTH, mask)
    assert abs(part / full - w.head_chunk / w.Hq) < 1e-3


# ---- sequence-tiled loss ------------------------------------------------------------------

def _expected_ce_ws(S, Dm, V, T):
    al = lambda x: (x + 255) // 256 * 256  # noqa: E731
    Tt = min(T, S)
    Tp = (Tt + 127) // 128 * 128
    n_vt = (V + 255) // 256
    fwd = al(n_vt * Tp * 8) + al(Tp * 4)
    bwd = al(Tt * V * 2)
    return fwd, bwd


@pytest.mark.parametrize("S,Dm,V,T", [(131072, 4096, 128256, 8192), (1000, 256, 1088, 256),
                                      (1, 64, 64, 128), (300, 64, 320, 1024)])
def test_loss_workspace_matches_formula(S, Dm, V, T):
    fwd, bwd = _expected_ce_ws(S, Dm, V, T)
    assert up.upipe_ce_workspace_bytes(S, Dm, V, T, up.UPIPE_PASS_FWD) == fwd
    assert up.upipe_ce_workspace_bytes(S, Dm, V, T, up.UPIPE_PASS_BWD) == bwd
    assert up.upipe_ce_workspace_bytes(S, Dm, V, T, up.UPIPE_PASS_BOTH) == max(fwd, bwd)
    # host activations: two slots of a tile of h (forward), of h and dh (backward)
    slot = (min(T, S) * Dm * 2 + 255) // 256 * 256
    ha = up.UPIPE_HOST_ACT
    assert up.upipe_ce_workspace_bytes(S, Dm, V, T, up.UPIPE_PASS_FWD, ha) == fwd + 2 * slot
    assert up.upipe_ce_workspace_bytes(S, Dm, V, T, up.UPIPE_PASS_BWD, ha) == bwd + 4 * slot
    assert up.upipe_ce_workspace_bytes(S, Dm, V, T, up.UPIPE_PASS_BWD, up.UPIPE_HOST_KV) == 0


def test_loss_workspace_is_bounded_by_the_tile_not_the_sequence():
    # the point of sequence tiling: the dlogits block depends on seq_tile, not on S
    a = up.upipe_ce_workspace_bytes(131072, 4096, 128256, 8192, up.UPIPE_PASS_BWD)
    b = up.upipe_ce_workspace_bytes(1 << 22, 4096, 128256, 8192, up.UPIPE_PASS_BWD)
    assert a == b == 8192 * 128256 * 2


@pytest.mark.parametrize("S,Dm,V,T", [(0, 64, 64, 128), (128, 96, 64, 128), (128, 64, 100, 128),
                                      (128, 64, 64, 100), (128, 64, 1 << 31, 128)])
def test_loss_workspace_zero_for_invalid(S, Dm, V, T):
    assert up.upipe_ce_workspace_bytes(S, Dm, V, T, up.UPIPE_PASS_BOTH) == 0


def test_loss_calls_validate_before_device_access():
    lib = ctypes.CDLL(up.LIB_PATH)
    st = up._lib.upipe_ce_fwd(None, None, None, None, None, 128, 64, 64, 128, None, 0, None)
    assert st == up.UPIPE_ERR_INVALID_ARG
    st = up._lib.upipe_ce_fwd(None, None, None, None, None, 128, 96, 64, 128, None, 0, None)
    assert st == up.UPIPE_ERR_UNSUPPORTED
    st = up._lib.upipe_ce_bwd(None, None, None, None, None, None, None, 128, 64, 64, 128, None,
                              0, None)
    assert st == up.UPIPE_ERR_INVALID_ARG
    assert "NULL" in up.upipe_last_error_message()
    assert lib is not None


# ---- sequence-tiled gated MLP ---------------------------------------------------------------

@pytest.mark.parametrize("S,Dm,F,T", [(131072, 4096, 14336, 8192), (1000, 256, 384, 256),
                                      (1, 64, 128, 128)])
def test_mlp_workspace_matches_formula(S, Dm, F, T):
    al = lambda x: (x + 255) // 256 * 256  # noqa: E731
    Tt = min(T, S)
    tf = Tt * F * 2
    assert up.upipe_mlp_workspace_bytes(S, Dm, F, T, up.UPIPE_PASS_FWD) == al(tf)
    bwd = al(tf) + 2 * al(2 * tf)
    assert up.upipe_mlp_workspace_bytes(S, Dm, F, T, up.UPIPE_PASS_BWD) == bwd
    assert up.upipe_mlp_workspace_bytes(S, Dm, F, T, up.UPIPE_PASS_BOTH) == bwd
    slot = al(Tt * Dm * 2)
    ha = up.UPIPE_HOST_ACT
    assert up.upipe_mlp_workspace_bytes(S, Dm, F, T, up.UPIPE_PASS_FWD, ha) == al(tf) + 4 * slot
    assert up.upipe_mlp_workspace_bytes(S, Dm, F, T, up.UPIPE_PASS_BWD, ha) == bwd + 6 * slot
    # bounded by the tile: the same at 32x the sequence
    S1 = max(S, T)
    assert up.upipe_mlp_workspace_bytes(32 * S1, Dm, F, T, up.UPIPE_PASS_BWD) == \
        up.upipe_mlp_workspace_bytes(S1, Dm, F, T, up.UPIPE_PASS_BWD)


@pytest.mark.parametrize("S,Dm,F,T", [(0, 64, 128, 128), (128, 96, 128, 128),
                                      (128, 64, 192, 128), (128, 64, 128, 64)])
def test_mlp_workspace_zero_for_invalid(S, Dm, F, T):
    assert up.upipe_mlp_workspace_bytes(S, Dm, F, T, up.UPIPE_PASS_BOTH) == 0


def test_mlp_calls_validate_before_device_access():
    st = up._lib.upipe_mlp_fwd(None, None, None, None, 128, 64, 128, 128, None, 0, None)
    assert st == up.UPIPE_ERR_INVALID_ARG
    st = up._lib.upipe_mlp_bwd(None, None, None, None, None, None, None, 128, 64, 192, 128,
                               None, 0, None)
    assert st == up.UPIPE_ERR_UNSUPPORTED


def test_copy_failure_hook_arms_and_validates_without_gpu():
    assert up._lib.upipe_debug_fail_copy_after(-1) == up.UPIPE_ERR_INVALID_ARG
    up.upipe_debug_fail_copy_after(5)
    up.upipe_debug_fail_copy_after(0)  # disarmed again


@pytest.mark.parametrize("S,Dm,V,T", [(131072, 4096, 128256, 8192), (1000, 256, 1088, 256)])
def test_fused_loss_workspace_matches_formula(S, Dm, V, T):
    al = lambda x: (x + 255) // 256 * 256  # noqa: E731
    Tt = min(T, S)
    Tp = (Tt + 127) // 128 * 128
    fused = al((V + 255) // 256 * Tp * 8) + al(Tp * 4) + al(Tt * V * 4) + al(Tt * V * 2)
    assert up.upipe_ce_workspace_bytes(S, Dm, V, T, up.UPIPE_PASS_FUSED) == fused
    slot = al(Tt * Dm * 2)
    assert up.upipe_ce_workspace_bytes(S, Dm, V, T, up.UPIPE_PASS_FUSED, up.UPIPE_HOST_ACT) == \
        fused + 4 * slot
    # the attention and MLP workspaces have no fused pass
    assert up.upipe_workspace_bytes(1, 1024, 8, 2, 128, 1, 4, 1024, up.UPIPE_PASS_FUSED) == 0
    assert up.upipe_mlp_workspace_bytes(S, Dm, 128, T, up.UPIPE_PASS_FUSED) == 0


# ---- the forward without allocation ----------------------------------------------------------

@pytest.mark.parametrize("args,status", [
    ((1, 512, 6, 4, 64, 1, 6, 512), up.UPIPE_ERR_INVALID_ARG),      # Hq % Hkv
    ((1, 512, 32, 8, 128, 1, 2, 512), up.UPIPE_ERR_INVALID_ARG),    # head_chunk % (Hq/Hkv)
    ((1, 1024, 4, 4, 64, 1, 4, 300), up.UPIPE_ERR_INVALID_ARG),     # seq_trunk % 128
    ((1, 512, 4, 4, 64, 2, 4, 512), up.UPIPE_ERR_INVALID_ARG),      # causal not 0/1
    ((1, 512, 4, 4, 96, 1, 4, 512), up.UPIPE_ERR_UNSUPPORTED),      # D
    ((1, (1 << 30) + 128, 4, 4, 64, 1, 4, 512), up.UPIPE_ERR_UNSUPPORTED),  # S > 2^30
    ((1, 16384, 32, 8, 128, 1, 32, 16384), up.UPIPE_ERR_WORKSPACE_TOO_SMALL),  # > 32 MiB
])
def test_noalloc_status_codes_without_device_access(args, status):
    """The no-allocation forward validates shapes with the same plan as upipe_attn_fwd and
    returns the same status for the same bad shape, before touching any pointer; a problem
    too large for its static scratch is rejected before any device access too."""
    B, S, Hq, Hkv, D, causal, hc, T = args
    n0 = up.upipe_launch_count()
    st = up._lib.upipe_attn_fwd_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, B, S, Hq, Hkv, D, causal,
                                        hc, T, 0, None)
    assert st == status, up.upipe_last_error_message()
    msg = up.upipe_last_error_message()
    assert msg
    if status != up.UPIPE_ERR_WORKSPACE_TOO_SMALL:
        st2 = up._lib.upipe_attn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, B, S, Hq, Hkv, D, causal, hc,
                                     T, FAKE, 1 << 40, None)
        assert st2 == st
        assert up.upipe_last_error_message() == msg
    else:
        assert "32 MiB" in msg
    assert up.upipe_launch_count() == n0


def test_noalloc_rejects_null_and_misaligned_pointers():
    args = (1, 512, 4, 4, 64, 1, 4, 512)
    for ptrs in ((FAKE, FAKE, FAKE, FAKE, None),          # no prefill form: lse required
                 (None, FAKE, FAKE, FAKE, FAKE),
                 (FAKE, FAKE, FAKE + 8, FAKE, FAKE)):    # v not 16-byte aligned
        st = up._lib.upipe_attn_fwd_noalloc(*ptrs, *args, 0, None)
        assert st == up.UPIPE_ERR_INVALID_ARG
