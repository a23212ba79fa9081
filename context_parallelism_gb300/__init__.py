"""Python binding of libupipe: head-chunked, trunked causal (GQA) attention for one GB300.

Argument marshalling only: every step of the attention path runs in the library's CUDA
kernels, reached through the C ABI declared in ``include/upipe.h``. The functions named
``upipe_*`` mirror that ABI one to one (tensors may be passed where the ABI takes pointers);
``attention_forward`` / ``attention_backward`` allocate outputs and the workspace with torch
and call them. There is no fallback: if ``libupipe.so`` is missing, importing the binding
fails with an error that says how to build it.
"""
from __future__ import annotations

import ctypes
import os

import numpy as _np  # noqa: F401  (kept for users that pass numpy-backed pinned buffers)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libupipe.so")

UPIPE_OK = 0
UPIPE_ERR_INVALID_ARG = 1
UPIPE_ERR_UNSUPPORTED = 2
UPIPE_ERR_WORKSPACE_TOO_SMALL = 3
UPIPE_ERR_CUDA = 4
UPIPE_ERR_TIMEOUT = 5

UPIPE_PASS_FWD, UPIPE_PASS_BWD, UPIPE_PASS_BOTH, UPIPE_PASS_FUSED = 0, 1, 2, 3
UPIPE_HOST_KV, UPIPE_HOST_ACT = 1, 2

KERNEL_CLASSES = ["layout", "attn_fwd", "bwd_pre", "attn_bwd", "dq_convert", "other",
                  "loss_gemm", "loss_merge", "kv_h2d", "dkdv_d2h", "kv_wait"]

# Every symbol include/upipe.h declares, with (restype, argtypes).
_vp, _i, _i64, _sz, _u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_uint64


class KernelStat(ctypes.Structure):
    _fields_ = [("total_ms", ctypes.c_double), ("launches", ctypes.c_uint64)]


SIGNATURES = {
    "upipe_workspace_bytes": (_sz, [_i, _i64, _i, _i, _i, _i, _i, _i64, _i, _i]),
    "upipe_attn_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i64, _i, _i, _i, _i, _i, _i64, _vp,
                            _sz, _vp]),
    "upipe_attn_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i64, _i, _i, _i,
                            _i, _i, _i64, _vp, _sz, _vp]),
    "upipe_attn_fwd_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i64, _i, _i, _i, _i, _i, _i64,
                                    _i, _vp]),
    "upipe_seq_to_head_major": (_i, [_vp, _vp, _i, _i64, _i, _i, _i, _i, _vp]),
    "upipe_head_to_seq_major": (_i, [_vp, _vp, _i, _i64, _i, _i, _i, _i, _vp]),
    "upipe_sync_status": (_i, [_vp]),
    "upipe_status_string": (ctypes.c_char_p, [_i]),
    "upipe_last_error_message": (ctypes.c_char_p, []),
    "upipe_shutdown": (None, []),
    "upipe_launch_count": (_u64, []),
    "upipe_debug_fail_copy_after": (_i, [_i]),
    "upipe_profile_enable": (_i, [_i]),
    "upipe_profile_read": (_i, [ctypes.POINTER(KernelStat), _i]),
    "upipe_selftest_umma": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _vp]),
    "upipe_selftest_wait_timeout": (_i, [_i, _vp]),
    "upipe_ce_workspace_bytes": (_sz, [_i64, _i, _i64, _i64, _i, _i]),
    "upipe_ce_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i64, _i, _i64, _i64, _vp, _sz, _vp]),
    "upipe_ce_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i, _i64, _i64, _vp, _sz,
                          _vp]),
    "upipe_ce_fwd_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i, _i64, _i64, _vp,
                              _sz, _vp]),
    "upipe_mlp_workspace_bytes": (_sz, [_i64, _i, _i, _i64, _i, _i]),
    "upipe_mlp_fwd": (_i, [_vp, _vp, _vp, _vp, _i64, _i, _i, _i64, _vp, _sz, _vp]),
    "upipe_mlp_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i, _i, _i64, _vp, _sz,
                           _vp]),
}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; "
            f"g.build()\"` (or `python context_parallelism_gb300/build.py`)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


class UpipeError(RuntimeError):
    def __init__(self, status, where):
        msg = _lib.upipe_last_error_message().decode()
        name = _lib.upipe_status_string(status).decode()
        super().__init__(f"{where}: {name}: {msg}")
        self.status = status


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    raise TypeError(f"cannot pass {type(x)} as a pointer")


def _stream(stream, *tensors):
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    import torch
    for t in tensors:
        if hasattr(t, "is_cuda") and t.is_cuda:
            return torch.cuda.current_stream(t.device).cuda_stream
    return None


def _check(status, where):
    if status != UPIPE_OK:
        raise UpipeError(status, where)


# ---- one-to-one ABI wrappers ------------------------------------------------------------

def upipe_workspace_bytes(B, S, Hq, Hkv, D, causal, head_chunk, seq_trunk, pass_=UPIPE_PASS_BOTH,
                          host_mask=0):
    """host_mask: UPIPE_HOST_KV | UPIPE_HOST_ACT bits (True/1 keeps meaning host k/v)."""
    return int(_lib.upipe_workspace_bytes(B, S, Hq, Hkv, D, int(causal), head_chunk, seq_trunk,
                                          pass_, int(host_mask)))


def upipe_attn_fwd(q, k, v, o, lse, B, S, Hq, Hkv, D, causal, head_chunk, seq_trunk, workspace,
                   workspace_bytes=None, stream=None):
    wb = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    st = _lib.upipe_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, S, Hq, Hkv, D,
                             int(causal), head_chunk, seq_trunk, _ptr(workspace), wb,
                             _stream(stream, q, o, workspace))
    _check(st, "upipe_attn_fwd")


def upipe_attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, S, Hq, Hkv, D, causal, head_chunk,
                   seq_trunk, workspace, workspace_bytes=None, stream=None):
    wb = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    st = _lib.upipe_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                             _ptr(dk), _ptr(dv), B, S, Hq, Hkv, D, int(causal), head_chunk,
                             seq_trunk, _ptr(workspace), wb, _stream(stream, q, dq, lse, workspace))
    _check(st, "upipe_attn_bwd")


def upipe_attn_fwd_noalloc(q, k, v, o, lse, B, S, Hq, Hkv, D, causal, head_chunk, seq_trunk,
                           check_status=0, stream=None):
    """The forward with its scratch in the library's static device array (no allocation)."""
    st = _lib.upipe_attn_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, S, Hq, Hkv,
                                     D, int(causal), head_chunk, seq_trunk, int(check_status),
                                     _stream(stream, q, o))
    _check(st, "upipe_attn_fwd_noalloc")


def upipe_seq_to_head_major(src, dst, B, S, H, D, h_begin, h_count, stream=None):
    _check(_lib.upipe_seq_to_head_major(_ptr(src), _ptr(dst), B, S, H, D, h_begin, h_count,
                                        _stream(stream, src)), "upipe_seq_to_head_major")


def upipe_head_to_seq_major(src, dst, B, S, H, D, h_begin, h_count, stream=None):
    _check(_lib.upipe_head_to_seq_major(_ptr(src), _ptr(dst), B, S, H, D, h_begin, h_count,
                                        _stream(stream, src)), "upipe_head_to_seq_major")


def upipe_sync_status(stream=None):
    """Synchronise the stream and raise UpipeError if a kernel's bounded wait expired."""
    import torch
    s = stream if stream is not None else (torch.cuda.current_stream().cuda_stream
                                           if torch.cuda.is_available() else None)
    if s is not None and not isinstance(s, int):
        s = s.cuda_stream
    _check(_lib.upipe_sync_status(s), "upipe_sync_status")


def upipe_status_string(status):
    return _lib.upipe_status_string(status).decode()


def upipe_last_error_message():
    return _lib.upipe_last_error_message().decode()


def upipe_shutdown():
    _lib.upipe_shutdown()


def upipe_launch_count():
    return int(_lib.upipe_launch_count())


def upipe_debug_fail_copy_after(n):
    """Test hook: the n-th staging copy from now on fails (0 disarms)."""
    _check(_lib.upipe_debug_fail_copy_after(int(n)), "upipe_debug_fail_copy_after")


def upipe_profile_enable(on=True):
    _check(_lib.upipe_profile_enable(int(on)), "upipe_profile_enable")


def upipe_profile_read():
    """Returns {class name: (total_ms, launches)} for the launches recorded since last read."""
    arr = (KernelStat * len(KERNEL_CLASSES))()
    _check(_lib.upipe_profile_read(arr, len(KERNEL_CLASSES)), "upipe_profile_read")
    return {n: (arr[i].total_ms, int(arr[i].launches)) for i, n in enumerate(KERNEL_CLASSES)}


def upipe_selftest_umma(a, b, c, N, K, a_mn_major, b_mn_major, a_manual=0, lbo=16384, sbo=1024,
                        stream=None):
    _check(_lib.upipe_selftest_umma(_ptr(a), _ptr(b), _ptr(c), N, K, int(a_mn_major),
                                    int(b_mn_major), int(a_manual), lbo, sbo,
                                    _stream(stream, a)), "upipe_selftest_umma")


def upipe_selftest_wait_timeout(limit_us, stream=None):
    _check(_lib.upipe_selftest_wait_timeout(limit_us, _stream(stream)),
           "upipe_selftest_wait_timeout")


def upipe_ce_workspace_bytes(S, Dm, V, seq_tile, pass_=UPIPE_PASS_BOTH, host_mask=0):
    return int(_lib.upipe_ce_workspace_bytes(S, Dm, V, seq_tile, pass_, int(host_mask)))


def upipe_ce_fwd(h, w, target, loss, lse, S, Dm, V, seq_tile, workspace, workspace_bytes=None,
                 stream=None):
    wb = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    st = _lib.upipe_ce_fwd(_ptr(h), _ptr(w), _ptr(target), _ptr(loss), _ptr(lse), S, Dm, V,
                           seq_tile, _ptr(workspace), wb, _stream(stream, h, loss, workspace))
    _check(st, "upipe_ce_fwd")


def upipe_ce_bwd(h, w, target, lse, dloss, dh, dw, S, Dm, V, seq_tile, workspace,
                 workspace_bytes=None, stream=None):
    wb = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    st = _lib.upipe_ce_bwd(_ptr(h), _ptr(w), _ptr(target), _ptr(lse), _ptr(dloss), _ptr(dh),
                           _ptr(dw), S, Dm, V, seq_tile, _ptr(workspace), wb,
                           _stream(stream, h, dh, workspace))
    _check(st, "upipe_ce_bwd")


def upipe_ce_fwd_bwd(h, w, target, dloss, loss, lse, dh, dw, S, Dm, V, seq_tile, workspace,
                     workspace_bytes=None, stream=None):
    wb = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    st = _lib.upipe_ce_fwd_bwd(_ptr(h), _ptr(w), _ptr(target), _ptr(dloss), _ptr(loss),
                               _ptr(lse), _ptr(dh), _ptr(dw), S, Dm, V, seq_tile,
                               _ptr(workspace), wb, _stream(stream, h, loss, workspace))
    _check(st, "upipe_ce_fwd_bwd")


def upipe_mlp_workspace_bytes(S, Dm, F, seq_tile, pass_=UPIPE_PASS_BOTH, host_mask=0):
    return int(_lib.upipe_mlp_workspace_bytes(S, Dm, F, seq_tile, pass_, int(host_mask)))


def upipe_mlp_fwd(x, w_gu, w_d, y, S, Dm, F, seq_tile, workspace, workspace_bytes=None,
                  stream=None):
    wb = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    st = _lib.upipe_mlp_fwd(_ptr(x), _ptr(w_gu), _ptr(w_d), _ptr(y), S, Dm, F, seq_tile,
                            _ptr(workspace), wb, _stream(stream, x, y, workspace))
    _check(st, "upipe_mlp_fwd")


def upipe_mlp_bwd(x, w_gu, w_d, dy, dx, dw_gu, dw_d, S, Dm, F, seq_tile, workspace,
                  workspace_bytes=None, stream=None):
    wb = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    st = _lib.upipe_mlp_bwd(_ptr(x), _ptr(w_gu), _ptr(w_d), _ptr(dy), _ptr(dx), _ptr(dw_gu),
                            _ptr(dw_d), S, Dm, F, seq_tile, _ptr(workspace), wb,
                            _stream(stream, x, dx, workspace))
    _check(st, "upipe_mlp_bwd")


# ---- convenience: allocate outputs / workspace with torch, then call the ABI -------------

def _dims(q, k):
    B, S, Hq, D = q.shape
    return B, S, Hq, k.shape[2], D


def _device_of(*tensors):
    import torch
    for t in tensors:
        if t is not None and t.is_cuda:
            return t.device
    return torch.device("cuda", torch.cuda.current_device())


def attention_forward(q, k, v, causal=True, head_chunk=None, seq_trunk=None, workspace=None,
                      stream=None, with_lse=True, o_on_host=False):
    """o, lse = attention over token-major bf16 q [B,S,Hq,D], k/v [B,S,Hkv,D].
    q, k/v may be pinned host tensors (staged head group by head group, trunk by trunk);
    o_on_host returns o as a pinned host tensor, copied out group by group. with_lse=False is
    the prefill (inference) form: lse is neither allocated nor written and None is returned."""
    import torch
    B, S, Hq, Hkv, D = _dims(q, k)
    hc = head_chunk or Hq
    T = seq_trunk or S
    dev = _device_of(q, k)
    kv_host = not k.is_cuda
    mask = (UPIPE_HOST_KV if kv_host else 0) | (UPIPE_HOST_ACT if (not q.is_cuda or o_on_host)
                                                else 0)
    if o_on_host:
        o = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    else:
        o = torch.empty(q.shape, dtype=q.dtype, device=dev)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device=dev) if with_lse else None
    need = upipe_workspace_bytes(B, S, Hq, Hkv, D, causal, hc, T, UPIPE_PASS_FWD, mask)
    if need == 0:
        upipe_attn_fwd(q, k, v, o, lse, B, S, Hq, Hkv, D, causal, hc, T, 0, 0, stream)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    upipe_attn_fwd(q, k, v, o, lse, B, S, Hq, Hkv, D, causal, hc, T, workspace, None, stream)
    return o, lse


def attention_backward(q, k, v, o, lse, dout, causal=True, head_chunk=None, seq_trunk=None,
                       workspace=None, stream=None, dkdv_on_host=False, dq_on_host=False):
    """dq, dk, dv for the forward above. q, o, dout may be pinned host tensors (staged head
    group by head group); dq_on_host returns dq as a pinned host tensor, copied out group by
    group. dk/dv are device tensors, or pinned host tensors when dkdv_on_host (which needs host
    k/v): then each trunk's dK/dV is copied out as it finishes."""
    import torch
    B, S, Hq, Hkv, D = _dims(q, k)
    hc = head_chunk or Hq
    T = seq_trunk or S
    dev = _device_of(q, k, lse)
    kv_host = not k.is_cuda
    act_host = dq_on_host or not (q.is_cuda and o.is_cuda and dout.is_cuda)
    mask = (UPIPE_HOST_KV if kv_host else 0) | (UPIPE_HOST_ACT if act_host else 0)
    if dq_on_host:
        dq = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    else:
        dq = torch.empty(q.shape, dtype=q.dtype, device=dev)
    if dkdv_on_host:
        dk = torch.empty((B, S, Hkv, D), dtype=q.dtype, pin_memory=True)
        dv = torch.empty((B, S, Hkv, D), dtype=q.dtype, pin_memory=True)
    else:
        dk = torch.empty((B, S, Hkv, D), dtype=q.dtype, device=dev)
        dv = torch.empty((B, S, Hkv, D), dtype=q.dtype, device=dev)
    need = upipe_workspace_bytes(B, S, Hq, Hkv, D, causal, hc, T, UPIPE_PASS_BWD, mask)
    if need == 0:
        upipe_attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, S, Hq, Hkv, D, causal, hc, T, 0, 0,
                       stream)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    upipe_attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, S, Hq, Hkv, D, causal, hc, T, workspace,
                   None, stream)
    return dq, dk, dv


def _tiled_device(*tensors):
    import torch
    for t in tensors:
        if t is not None and t.is_cuda:
            return t.device
    return torch.device("cuda", torch.cuda.current_device())


def _empty_like_on(shape, dtype, dev, on_host):
    import torch
    if on_host:
        return torch.empty(shape, dtype=dtype, pin_memory=True)
    return torch.empty(shape, dtype=dtype, device=dev)


def ce_loss_forward(h, w, target, seq_tile=8192, workspace=None, stream=None):
    """loss, lse (float32 [S]) of the readout h [S, Dm] @ w[V, Dm]^T followed by token-level
    cross-entropy against target [S] (int64, negative = ignored), computed seq_tile tokens at
    a time without storing logits. h may be a pinned host tensor (staged tile by tile)."""
    import torch
    S, Dm = h.shape
    V = w.shape[0]
    dev = _tiled_device(w, target)
    loss = torch.empty(S, dtype=torch.float32, device=dev)
    lse = torch.empty(S, dtype=torch.float32, device=dev)
    mask = 0 if h.is_cuda else UPIPE_HOST_ACT
    need = upipe_ce_workspace_bytes(S, Dm, V, seq_tile, UPIPE_PASS_FWD, mask)
    if need == 0:
        upipe_ce_fwd(h, w, target, loss, lse, S, Dm, V, seq_tile, 0, 0, stream)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    upipe_ce_fwd(h, w, target, loss, lse, S, Dm, V, seq_tile, workspace, None, stream)
    return loss, lse


def ce_loss_backward(h, w, target, lse, dloss, seq_tile=8192, workspace=None, stream=None,
                     dh_on_host=False):
    """dh (bf16 [S, Dm]) and dw (float32 [V, Dm]) of sum_i dloss[i] * loss[i] for the forward
    above; lse is the forward's. h may be a pinned host tensor; dh_on_host returns dh as one."""
    import torch
    S, Dm = h.shape
    V = w.shape[0]
    dev = _tiled_device(w, target)
    dh = _empty_like_on((S, Dm), h.dtype, dev, dh_on_host)
    dw = torch.empty((V, Dm), dtype=torch.float32, device=dev)
    mask = UPIPE_HOST_ACT if (dh_on_host or not h.is_cuda) else 0
    need = upipe_ce_workspace_bytes(S, Dm, V, seq_tile, UPIPE_PASS_BWD, mask)
    if need == 0:
        upipe_ce_bwd(h, w, target, lse, dloss, dh, dw, S, Dm, V, seq_tile, 0, 0, stream)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    upipe_ce_bwd(h, w, target, lse, dloss, dh, dw, S, Dm, V, seq_tile, workspace, None, stream)
    return dh, dw


def ce_loss_fused(h, w, target, dloss, seq_tile=8192, workspace=None, stream=None,
                  dh_on_host=False):
    """loss, lse, dh, dw in one call when the upstream gradient dloss is known up front (the
    loss is the last operation). Bitwise the results of ce_loss_forward + ce_loss_backward,
    without the backward's logits recompute; needs seq_tile * V * 6 more bytes of workspace."""
    import torch
    S, Dm = h.shape
    V = w.shape[0]
    dev = _tiled_device(w, target)
    loss = torch.empty(S, dtype=torch.float32, device=dev)
    lse = torch.empty(S, dtype=torch.float32, device=dev)
    dh = _empty_like_on((S, Dm), h.dtype, dev, dh_on_host)
    dw = torch.empty((V, Dm), dtype=torch.float32, device=dev)
    mask = UPIPE_HOST_ACT if (dh_on_host or not h.is_cuda) else 0
    need = upipe_ce_workspace_bytes(S, Dm, V, seq_tile, UPIPE_PASS_FUSED, mask)
    if need == 0:
        upipe_ce_fwd_bwd(h, w, target, dloss, loss, lse, dh, dw, S, Dm, V, seq_tile, 0, 0, stream)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    upipe_ce_fwd_bwd(h, w, target, dloss, loss, lse, dh, dw, S, Dm, V, seq_tile, workspace, None,
                     stream)
    return loss, lse, dh, dw


def mlp_forward(x, w_gu, w_d, seq_tile=8192, workspace=None, stream=None, y_on_host=False):
    """y = (silu(x Wg^T) * x Wu^T) Wd^T for x [S, Dm], w_gu = [Wg; Wu] [2F, Dm], w_d [Dm, F]
    (bf16), seq_tile tokens at a time. x may be a pinned host tensor; y_on_host returns y as
    one."""
    import torch
    S, Dm = x.shape
    F = w_d.shape[1]
    dev = _tiled_device(w_gu)
    y = _empty_like_on((S, Dm), x.dtype, dev, y_on_host)
    mask = UPIPE_HOST_ACT if (y_on_host or not x.is_cuda) else 0
    need = upipe_mlp_workspace_bytes(S, Dm, F, seq_tile, UPIPE_PASS_FWD, mask)
    if need == 0:
        upipe_mlp_fwd(x, w_gu, w_d, y, S, Dm, F, seq_tile, 0, 0, stream)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    upipe_mlp_fwd(x, w_gu, w_d, y, S, Dm, F, seq_tile, workspace, None, stream)
    return y


def mlp_backward(x, w_gu, w_d, dy, seq_tile=8192, workspace=None, stream=None,
                 dx_on_host=False):
    """dx (bf16 [S, Dm]), dw_gu (float32 [2F, Dm]) and dw_d (float32 [Dm, F]) for the forward
    above and the upstream gradient dy [S, Dm]. x and dy may be pinned host tensors;
    dx_on_host returns dx as one."""
    import torch
    S, Dm = x.shape
    F = w_d.shape[1]
    dev = _tiled_device(w_gu)
    dx = _empty_like_on((S, Dm), x.dtype, dev, dx_on_host)
    dw_gu = torch.empty((2 * F, Dm), dtype=torch.float32, device=dev)
    dw_d = torch.empty((Dm, F), dtype=torch.float32, device=dev)
    mask = UPIPE_HOST_ACT if (dx_on_host or not x.is_cuda or not dy.is_cuda) else 0
    need = upipe_mlp_workspace_bytes(S, Dm, F, seq_tile, UPIPE_PASS_BWD, mask)
    if need == 0:
        upipe_mlp_bwd(x, w_gu, w_d, dy, dx, dw_gu, dw_d, S, Dm, F, seq_tile, 0, 0, stream)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    upipe_mlp_bwd(x, w_gu, w_d, dy, dx, dw_gu, dw_d, S, Dm, F, seq_tile, workspace, None,
                  stream)
    return dx, dw_gu, dw_d
