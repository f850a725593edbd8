"""Thin Python binding of ``libxt_attn.so`` (the C ABI in ``include/xt_attn.h``).

Argument marshalling only: the functions here allocate outputs with PyTorch
(device memory is PyTorch's job), pass ``data_ptr()`` values and the current
CUDA stream to the library, and turn non-zero status codes into exceptions.
Every step of the computation runs in the library's kernels. There is no
fallback: if the library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

XT_OK, XT_EINVAL, XT_EUNSUPPORTED, XT_ECUDA, XT_EWORKSPACE, XT_ETIMEOUT = range(6)
XT_F32, XT_BF16 = 0, 1

_lib = None


class XtError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {xt_status_str(status)} (status {status})"
        if status == XT_ECUDA and _lib is not None:
            msg += f", cudaError {_lib.xt_last_cuda_error()}"
        super().__init__(msg)


def library_path() -> str:
    return _build.LIB_PATH


def lib():
    """Loads libxt_attn.so (built in-tree by ``build.build()``); raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it first (causal_gqa_attention_xt_gb300.build)")
    L = ctypes.CDLL(path)
    i, d, sz, vp = ctypes.c_int, ctypes.c_double, ctypes.c_size_t, ctypes.c_void_p
    L.xt_attn_workspace_bytes.argtypes = [i, i, i, i, i, i, i]
    L.xt_attn_workspace_bytes.restype = sz
    L.xt_attn_fwd.argtypes = [i, i, i, i, i, d, d, vp, vp, vp, vp, vp, i, vp, vp, vp, vp, vp, vp,
                              vp, sz, vp]
    L.xt_attn_fwd.restype = i
    L.xt_attn_bwd.argtypes = [i, i, i, i, i, d, d, vp, vp, vp, vp, vp, i, vp, vp, vp, vp, vp, vp,
                              vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.xt_attn_bwd.restype = i
    L.xt_attn_bwd_noalloc.argtypes = [i, i, i, i, i, d, d, vp, vp, vp, vp, vp, i, vp, vp, vp, vp,
                                      vp, vp, vp, vp, vp, vp, vp, vp, vp]
    L.xt_attn_bwd_noalloc.restype = i
    L.xt_attn_varlen_workspace_bytes.argtypes = [i, i, i, i, i, i, i, i]
    L.xt_attn_varlen_workspace_bytes.restype = sz
    L.xt_attn_fwd_varlen.argtypes = [i, i, i, i, i, i, d, d, vp, vp, vp, vp, vp, vp, i, vp, vp,
                                     vp, vp, vp, vp, vp, sz, vp]
    L.xt_attn_fwd_varlen.restype = i
    L.xt_attn_bwd_varlen.argtypes = [i, i, i, i, i, i, d, d, vp, vp, vp, vp, vp, vp, i, vp, vp,
                                     vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.xt_attn_bwd_varlen.restype = i
    L.xt_attn_decode_workspace_bytes.argtypes = [i, i, i, i, i, i]
    L.xt_attn_decode_workspace_bytes.restype = sz
    L.xt_attn_decode.argtypes = [i, i, i, i, i, d, d, vp, vp, vp, vp, vp, vp, i, vp, vp, vp, vp,
                                 vp, sz, vp]
    L.xt_attn_decode.restype = i
    L.xt_attn_check.argtypes = [vp]
    L.xt_attn_check.restype = i
    L.xt_status_str.argtypes = [i]
    L.xt_status_str.restype = ctypes.c_char_p
    L.xt_last_cuda_error.restype = i
    L.xt_timing_enable.argtypes = [i]
    L.xt_timing_query.argtypes = [i, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_long)]
    L.xt_kernel_count.restype = i
    L.xt_test_inject_stall.argtypes = [i]
    L.xt_test_inject_stall.restype = i
    L.xt_kernel_name.argtypes = [i]
    L.xt_kernel_name.restype = ctypes.c_char_p
    _lib = L
    return L


def xt_status_str(status: int) -> str:
    return lib().xt_status_str(int(status)).decode()


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return XT_F32
    if t == torch.bfloat16:
        return XT_BF16
    raise TypeError(f"unsupported dtype {t}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("tensors must be contiguous CUDA tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def xt_attn_workspace_bytes(B, S, n_heads, n_kv_heads, head_dim, dtype, backward) -> int:
    code = dtype if isinstance(dtype, int) else _dtype_code(dtype)
    return int(lib().xt_attn_workspace_bytes(B, S, n_heads, n_kv_heads, head_dim, code,
                                             int(bool(backward))))


def xt_attn_fwd(q, k, v, gamma_q, gamma_k, eps, theta, *, out=None, lse=None, q_hat=None,
                k_hat=None, rstd_q=None, rstd_k=None, workspace=None, stream=None):
    """Forward of the attention core on CUDA tensors.

    q [B,S,H,D], k/v [B,S,G,D] (bf16 or fp32), gamma_q/gamma_k [D] fp32.
    Returns a dict: out [B,S,H,D], lse [B,H,S], q_hat [B,H,S,D], k_hat [B,G,S,D],
    rstd_q [B,S,H], rstd_k [B,S,G]. Outputs may be passed in preallocated.
    """
    B, S, H, D = q.shape
    G = k.shape[2]
    dev, dt = q.device, q.dtype
    f32 = dict(device=dev, dtype=torch.float32)
    out = out if out is not None else torch.empty((B, S, H, D), device=dev, dtype=dt)
    lse = lse if lse is not None else torch.empty((B, H, S), **f32)
    q_hat = q_hat if q_hat is not None else torch.empty((B, H, S, D), device=dev, dtype=dt)
    k_hat = k_hat if k_hat is not None else torch.empty((B, G, S, D), device=dev, dtype=dt)
    rstd_q = rstd_q if rstd_q is not None else torch.empty((B, S, H), **f32)
    rstd_k = rstd_k if rstd_k is not None else torch.empty((B, S, G), **f32)
    code = _dtype_code(dt)
    need = xt_attn_workspace_bytes(B, S, H, G, D, code, False)
    if workspace is None and need > 0:
        workspace = torch.empty(need, device=dev, dtype=torch.uint8)
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().xt_attn_fwd(B, S, H, G, D, float(eps), float(theta), _ptr(q), _ptr(k), _ptr(v),
                           _ptr(gamma_q), _ptr(gamma_k), code, _ptr(out), _ptr(lse), _ptr(q_hat),
                           _ptr(k_hat), _ptr(rstd_q), _ptr(rstd_k), _ptr(workspace), wbytes,
                           _stream(stream))
    if st != XT_OK:
        raise XtError(st, "xt_attn_fwd")
    return dict(out=out, lse=lse, q_hat=q_hat, k_hat=k_hat, rstd_q=rstd_q, rstd_k=rstd_k)


def xt_attn_bwd(q, k, v, gamma_q, gamma_k, saved, dout, eps, theta, *, dq=None, dk=None, dv=None,
                dgamma_q=None, dgamma_k=None, workspace=None, stream=None):
    """Backward of the attention core; ``saved`` is the dict xt_attn_fwd returned.

    Returns a dict: dq [B,S,H,D], dk/dv [B,S,G,D] (input dtype), dgamma_q,
    dgamma_k [D] fp32 (overwritten).
    """
    B, S, H, D = q.shape
    G = k.shape[2]
    dev, dt = q.device, q.dtype
    dq = dq if dq is not None else torch.empty_like(q)
    dk = dk if dk is not None else torch.empty_like(k)
    dv = dv if dv is not None else torch.empty_like(v)
    dgamma_q = dgamma_q if dgamma_q is not None else torch.empty(D, device=dev, dtype=torch.float32)
    dgamma_k = dgamma_k if dgamma_k is not None else torch.empty(D, device=dev, dtype=torch.float32)
    code = _dtype_code(dt)
    need = xt_attn_workspace_bytes(B, S, H, G, D, code, True)
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=dev, dtype=torch.uint8)
    wbytes = workspace.numel() * workspace.element_size()
    st = lib().xt_attn_bwd(B, S, H, G, D, float(eps), float(theta), _ptr(q), _ptr(k), _ptr(v),
                           _ptr(gamma_q), _ptr(gamma_k), code, _ptr(saved["out"]),
                           _ptr(saved["lse"]), _ptr(saved["q_hat"]), _ptr(saved["k_hat"]),
                           _ptr(saved["rstd_q"]), _ptr(saved["rstd_k"]), _ptr(dout), _ptr(dq),
                           _ptr(dk), _ptr(dv), _ptr(dgamma_q), _ptr(dgamma_k), _ptr(workspace),
                           wbytes, _stream(stream))
    if st != XT_OK:
        raise XtError(st, "xt_attn_bwd")
    return dict(dq=dq, dk=dk, dv=dv, dgamma_q=dgamma_q, dgamma_k=dgamma_k)


def xt_attn_bwd_noalloc(q, k, v, gamma_q, gamma_k, saved, dout, eps, theta, *, dq=None, dk=None,
                        dv=None, dgamma_q=None, dgamma_k=None, stream=None):
    """xt_attn_bwd without a workspace: the library's fixed 16 MiB device array is
    its scratch (for callers that cannot allocate). Outputs are the caller's,
    allocated here only when not passed in. Raises XtError(XT_EWORKSPACE) for
    problems that need more scratch than the array holds."""
    B, S, H, D = q.shape
    G = k.shape[2]
    dev = q.device
    dq = dq if dq is not None else torch.empty_like(q)
    dk = dk if dk is not None else torch.empty_like(k)
    dv = dv if dv is not None else torch.empty_like(v)
    dgamma_q = dgamma_q if dgamma_q is not None else torch.empty(D, device=dev, dtype=torch.float32)
    dgamma_k = dgamma_k if dgamma_k is not None else torch.empty(D, device=dev, dtype=torch.float32)
    st = lib().xt_attn_bwd_noalloc(B, S, H, G, D, float(eps), float(theta), _ptr(q), _ptr(k),
                                   _ptr(v), _ptr(gamma_q), _ptr(gamma_k), _dtype_code(q.dtype),
                                   _ptr(saved["out"]), _ptr(saved["lse"]), _ptr(saved["q_hat"]),
                                   _ptr(saved["k_hat"]), _ptr(saved["rstd_q"]),
                                   _ptr(saved["rstd_k"]), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                                   _ptr(dgamma_q), _ptr(dgamma_k), _stream(stream))
    if st != XT_OK:
        raise XtError(st, "xt_attn_bwd_noalloc")
    return dict(dq=dq, dk=dk, dv=dv, dgamma_q=dgamma_q, dgamma_k=dgamma_k)


def xt_attn_varlen_workspace_bytes(total, nseq, max_seqlen, n_heads, n_kv_heads, head_dim,
                                   dtype, backward) -> int:
    code = dtype if isinstance(dtype, int) else _dtype_code(dtype)
    return int(lib().xt_attn_varlen_workspace_bytes(total, nseq, max_seqlen, n_heads, n_kv_heads,
                                                    head_dim, code, int(bool(backward))))


def _check_cu(cu_seqlens):
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2:
        raise ValueError("cu_seqlens must be a 1-D int32 CUDA tensor of nseq + 1 offsets")
    return cu_seqlens.numel() - 1


def xt_attn_fwd_varlen(q, k, v, gamma_q, gamma_k, cu_seqlens, max_seqlen, eps, theta, *,
                       out=None, lse=None, q_hat=None, k_hat=None, rstd_q=None, rstd_k=None,
                       workspace=None, stream=None):
    """Forward over a packed batch: sample s on rows cu_seqlens[s]..cu_seqlens[s+1]-1.

    q [T,H,D], k/v [T,G,D], cu_seqlens int32 [nseq+1] on the device, max_seqlen
    the longest sample (host int). Returns a dict: out [T,H,D], lse [H,T],
    q_hat [H,T,D], k_hat [G,T,D], rstd_q [T,H], rstd_k [T,G].
    """
    T, H, D = q.shape
    G = k.shape[1]
    nseq = _check_cu(cu_seqlens)
    dev, dt = q.device, q.dtype
    f32 = dict(device=dev, dtype=torch.float32)
    out = out if out is not None else torch.empty((T, H, D), device=dev, dtype=dt)
    lse = lse if lse is not None else torch.empty((H, T), **f32)
    q_hat = q_hat if q_hat is not None else torch.empty((H, T, D), device=dev, dtype=dt)
    k_hat = k_hat if k_hat is not None else torch.empty((G, T, D), device=dev, dtype=dt)
    rstd_q = rstd_q if rstd_q is not None else torch.empty((T, H), **f32)
    rstd_k = rstd_k if rstd_k is not None else torch.empty((T, G), **f32)
    code = _dtype_code(dt)
    need = xt_attn_varlen_workspace_bytes(T, nseq, max_seqlen, H, G, D, code, False)
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=dev, dtype=torch.uint8)
    wbytes = workspace.numel() * workspace.element_size()
    st = lib().xt_attn_fwd_varlen(T, nseq, int(max_seqlen), H, G, D, float(eps), float(theta),
                                  _ptr(cu_seqlens), _ptr(q), _ptr(k), _ptr(v), _ptr(gamma_q),
                                  _ptr(gamma_k), code, _ptr(out), _ptr(lse), _ptr(q_hat),
                                  _ptr(k_hat), _ptr(rstd_q), _ptr(rstd_k), _ptr(workspace),
                                  wbytes, _stream(stream))
    if st != XT_OK:
        raise XtError(st, "xt_attn_fwd_varlen")
    return dict(out=out, lse=lse, q_hat=q_hat, k_hat=k_hat, rstd_q=rstd_q, rstd_k=rstd_k)


def xt_attn_bwd_varlen(q, k, v, gamma_q, gamma_k, cu_seqlens, max_seqlen, saved, dout, eps,
                       theta, *, dq=None, dk=None, dv=None, dgamma_q=None, dgamma_k=None,
                       workspace=None, stream=None):
    """Backward over a packed batch; ``saved`` is the dict xt_attn_fwd_varlen returned."""
    T, H, D = q.shape
    G = k.shape[1]
    nseq = _check_cu(cu_seqlens)
    dev, dt = q.device, q.dtype
    dq = dq if dq is not None else torch.empty_like(q)
    dk = dk if dk is not None else torch.empty_like(k)
    dv = dv if dv is not None else torch.empty_like(v)
    dgamma_q = dgamma_q if dgamma_q is not None else torch.empty(D, device=dev, dtype=torch.float32)
    dgamma_k = dgamma_k if dgamma_k is not None else torch.empty(D, device=dev, dtype=torch.float32)
    code = _dtype_code(dt)
    need = xt_attn_varlen_workspace_bytes(T, nseq, max_seqlen, H, G, D, code, True)
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=dev, dtype=torch.uint8)
    wbytes = workspace.numel() * workspace.element_size()
    st = lib().xt_attn_bwd_varlen(T, nseq, int(max_seqlen), H, G, D, float(eps), float(theta),
                                  _ptr(cu_seqlens), _ptr(q), _ptr(k), _ptr(v), _ptr(gamma_q),
                                  _ptr(gamma_k), code, _ptr(saved["out"]), _ptr(saved["lse"]),
                                  _ptr(saved["q_hat"]), _ptr(saved["k_hat"]),
                                  _ptr(saved["rstd_q"]), _ptr(saved["rstd_k"]), _ptr(dout),
                                  _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dgamma_q), _ptr(dgamma_k),
                                  _ptr(workspace), wbytes, _stream(stream))
    if st != XT_OK:
        raise XtError(st, "xt_attn_bwd_varlen")
    return dict(dq=dq, dk=dk, dv=dv, dgamma_q=dgamma_q, dgamma_k=dgamma_k)


def xt_attn_decode_workspace_bytes(B, S_max, n_heads, n_kv_heads, head_dim, dtype) -> int:
    code = dtype if isinstance(dtype, int) else _dtype_code(dtype)
    return int(lib().xt_attn_decode_workspace_bytes(B, S_max, n_heads, n_kv_heads, head_dim, code))


def xt_attn_decode(pos, q, k, v, gamma_q, gamma_k, k_cache, v_cache, eps, theta, *, out=None,
                   lse=None, workspace=None, stream=None):
    """One decode step: the new token of each batch element (q [B, H, D], k and v
    [B, G, D]) at position pos[b] (int32 CUDA tensor [B]) is appended to the
    caches (k_cache, v_cache [B, G, S_max, D], updated in place) and attends over
    rows 0..pos[b]. Returns dict(out [B, H, D], lse [B, H] fp32)."""
    B, H, D = q.shape
    G = k.shape[1]
    S_max = k_cache.shape[2]
    if pos.dtype != torch.int32 or pos.numel() != B:
        raise ValueError("pos must be an int32 tensor of B positions")
    dev = q.device
    code = _dtype_code(q.dtype)
    out = out if out is not None else torch.empty_like(q)
    lse = lse if lse is not None else torch.empty(B, H, device=dev, dtype=torch.float32)
    need = xt_attn_decode_workspace_bytes(B, S_max, H, G, D, code)
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=dev, dtype=torch.uint8)
    wbytes = workspace.numel() * workspace.element_size()
    st = lib().xt_attn_decode(B, S_max, H, G, D, float(eps), float(theta), _ptr(pos), _ptr(q),
                              _ptr(k), _ptr(v), _ptr(gamma_q), _ptr(gamma_k), code,
                              _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(lse),
                              _ptr(workspace), wbytes, _stream(stream))
    if st != XT_OK:
        raise XtError(st, "xt_attn_decode")
    return dict(out=out, lse=lse)


def xt_attn_check(stream=None) -> int:
    """Synchronizes the stream and returns the library's device status
    (XT_OK, XT_ETIMEOUT, or XT_EINVAL for an out-of-range decode position)."""
    return int(lib().xt_attn_check(_stream(stream)))


# ---- per-launch timing hooks -------------------------------------------

STALL_FWD_TC, STALL_DKDV_TC, STALL_DQ_TC = 1, 2, 4


def xt_test_inject_stall(kernel_mask: int) -> int:
    """Fault injection for the timeout path (see include/xt_attn.h): the
    tensor-core kernels in kernel_mask stall until their bounded wait runs
    out; 0 turns it off."""
    return lib().xt_test_inject_stall(int(kernel_mask))


def xt_timing_enable(on: bool = True):
    lib().xt_timing_enable(int(bool(on)))


def xt_timing_reset():
    lib().xt_timing_reset()


def xt_timing_query() -> dict:
    """{kernel name: (total ms, launches)} for every kernel that launched."""
    L = lib()
    res = {}
    for kid in range(L.xt_kernel_count()):
        ms, n = ctypes.c_double(0.0), ctypes.c_long(0)
        L.xt_timing_query(kid, ctypes.byref(ms), ctypes.byref(n))
        if n.value:
            res[L.xt_kernel_name(kid).decode()] = (ms.value, n.value)
    return res


class XtAttention(torch.autograd.Function):
    """Autograd wrapper: forward and backward both run in the library."""

    @staticmethod
    def forward(ctx, q, k, v, gamma_q, gamma_k, eps, theta):
        saved = xt_attn_fwd(q, k, v, gamma_q, gamma_k, eps, theta)
        ctx.save_for_backward(q, k, v, gamma_q, gamma_k, saved["out"], saved["lse"],
                              saved["q_hat"], saved["k_hat"], saved["rstd_q"], saved["rstd_k"])
        ctx.eps, ctx.theta = eps, theta
        return saved["out"]

    @staticmethod
    def backward(ctx, dout):
        q, k, v, gq, gk, out, lse, qh, kh, rq, rk = ctx.saved_tensors
        saved = dict(out=out, lse=lse, q_hat=qh, k_hat=kh, rstd_q=rq, rstd_k=rk)
        g = xt_attn_bwd(q, k, v, gq, gk, saved, dout.contiguous(), ctx.eps, ctx.theta)
        return g["dq"], g["dk"], g["dv"], g["dgamma_q"], g["dgamma_k"], None, None
