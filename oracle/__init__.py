"""Plain double-precision CPU oracle of the causal GQA attention core.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline / reference leg of ``bench.py`` may import this package. The CUDA
library never links, loads or calls it, and the two share no code.

The arithmetic lives in ``xt_oracle.c`` (compiled here with gcc, no fast-math,
no FMA contraction); this module only marshals numpy arrays. Every function
follows a passage of the pages:

* RMSNorm forward/backward -- Mint project report, 5.5.1 and 5.5.2; xtrain
  "Phase T9: Export to xserv", Decision 1 (per-head QK-norm, one [head_dim]
  gamma shared by all heads, before RoPE).
* rotate_half RoPE -- Mint report 5.4.1 (pair (i, i + D/2)), 5.4.2 (angle
  pos * theta^(-2i/D)), 5.4.4 (backward = rotation by the negative angle);
  xtrain T9 architecture-diff table (pos = row, theta from the config).
* causal SDPA -- xtrain "Phase T5: Tiny Transformer", Key Design Decisions
  (additive -1e9 mask above the diagonal) and its per-head layout pipeline;
  Mint report 5.3.1 (scale 1/sqrt(d_k), max-subtracted softmax, P V).
* GQA -- xtrain "Phase T15: GQA", "What is GQA" (q head qh reads kv head
  qh/group) and Decision 2 (repeat_kv copy; backward = in-order group sum).
* softmax backward -- the pages give none; the oracle uses the exact Jacobian
  dS = P o (dP - rowsum(dP o P)).
* packed batches -- Mint report 8.2 (a chat batch flattened to [total] rows,
  RoPE positions numbered inside each sample, block-causal mask: other
  samples' rows hidden, causal inside a sample).

Parity status: every function here is pinned by tests in
``tests/test_oracle_pins.py`` (library routines, closed forms, invariants,
finite differences and a hand-worked example); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "xt_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liborc.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile xt_oracle.c into oracle/_build/liborc.so (plain gcc, -O2)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-pthread", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            lib = ctypes.CDLL(path)
            dp = ctypes.POINTER(ctypes.c_double)
            lp = ctypes.POINTER(ctypes.c_long)
            I, L, Dd = ctypes.c_int, ctypes.c_long, ctypes.c_double
            lib.orc_rmsnorm_rows.argtypes = [L, I, dp, dp, Dd, dp, dp]
            lib.orc_rmsnorm_rows_bwd.argtypes = [L, I, dp, dp, Dd, dp, dp, dp]
            lib.orc_rope_rows.argtypes = [L, I, Dd, lp, dp, dp, I]
            lib.orc_repeat_kv.argtypes = [I, I, I, L, dp, dp]
            lib.orc_repeat_kv_bwd.argtypes = [I, I, I, L, dp, dp]
            lib.orc_sdpa_head_fwd.argtypes = [I, I, dp, dp, dp, dp, dp, dp]
            lib.orc_sdpa_head_bwd.argtypes = [I, I, dp, dp, dp, dp, dp, dp, dp, dp]
            lib.orc_attn_fwd.argtypes = [I, I, I, I, I, Dd, Dd, dp, dp, dp, dp, dp,
                                         dp, dp, dp, dp, dp, dp, I]
            lib.orc_attn_fwd.restype = I
            lib.orc_attn_bwd.argtypes = [I, I, I, I, I, Dd, Dd, dp, dp, dp, dp, dp, dp,
                                         dp, dp, dp, dp, dp, I]
            lib.orc_attn_bwd.restype = I
            lib.orc_attn_fwd_packed.argtypes = [I, lp, I, I, I, Dd, Dd, dp, dp, dp, dp, dp,
                                                dp, dp, dp, dp, dp, dp, I]
            lib.orc_attn_fwd_packed.restype = I
            lib.orc_attn_bwd_packed.argtypes = [I, lp, I, I, I, Dd, Dd, dp, dp, dp, dp, dp, dp,
                                                dp, dp, dp, dp, dp, I]
            lib.orc_attn_bwd_packed.restype = I
            lib.orc_attn_fwd_rows.argtypes = [I, I, I, I, I, Dd, Dd, dp, dp, dp, dp, dp,
                                              L, lp, dp, dp, I]
            lib.orc_attn_fwd_rows.restype = I
            lib.orc_attn_dq_rows.argtypes = [I, I, I, I, I, Dd, Dd, dp, dp, dp, dp, dp, dp,
                                             L, lp, dp, I]
            lib.orc_attn_dq_rows.restype = I
            lib.orc_attn_dkdv_rows.argtypes = [I, I, I, I, I, Dd, Dd, dp, dp, dp, dp, dp, dp,
                                               L, lp, dp, dp, I]
            lib.orc_attn_dkdv_rows.restype = I
            _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def host_available_bytes():
    """MemAvailable of the host (bytes), or None where /proc/meminfo is absent."""
    try:
        with open("/proc/meminfo") as f:
            for ln in f:
                if ln.startswith("MemAvailable:"):
                    return int(ln.split()[1]) * 1024
    except (OSError, ValueError, IndexError):
        pass
    return None


def head_threads(nthreads, S, n_square, n_heads):
    """Thread count for a whole-head call: each thread holds n_square [S, S]
    fp64 buffers, so the count is capped to keep them within half of the
    host's available memory (the results do not depend on the count)."""
    n = int(nthreads or default_threads())
    n = max(1, min(n, int(n_heads)))
    avail = host_available_bytes()
    if avail is not None:
        per_thread = n_square * 8 * int(S) * int(S) + (1 << 20)
        n = max(1, min(n, int(0.5 * avail // per_thread)))
    return n


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a: np.ndarray):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _lp(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_long))


# --- single steps ---------------------------------------------------------

def rmsnorm_rows(x, gamma, eps):
    """y = x * rsqrt(mean(x^2) + eps) * gamma over the last axis; also 1/rms."""
    x = _f64(x)
    D = x.shape[-1]
    rows = x.size // D
    g = _f64(gamma)
    y = np.empty_like(x)
    rstd = np.empty(x.shape[:-1], dtype=np.float64)
    _load().orc_rmsnorm_rows(rows, D, _p(x), _p(g), float(eps), _p(y), _p(rstd))
    return y, rstd


def rmsnorm_rows_bwd(x, gamma, eps, dy):
    """(dx, dgamma) of the RMSNorm above for upstream gradient dy."""
    x, dy, g = _f64(x), _f64(dy), _f64(gamma)
    D = x.shape[-1]
    dx = np.empty_like(x)
    dg = np.zeros(D, dtype=np.float64)
    _load().orc_rmsnorm_rows_bwd(x.size // D, D, _p(x), _p(g), float(eps), _p(dy), _p(dx), _p(dg))
    return dx, dg


def rope_rows(x, pos, theta, inverse=False):
    """rotate_half RoPE of rows x[..., D] at positions pos[...] (same leading shape)."""
    x = _f64(x)
    D = x.shape[-1]
    rows = x.size // D
    pos = np.ascontiguousarray(np.broadcast_to(np.asarray(pos, dtype=np.int64),
                                               x.shape[:-1])).astype(np.int64).reshape(-1)
    y = np.empty_like(x)
    _load().orc_rope_rows(rows, D, float(theta), _lp(pos), _p(x), _p(y), int(bool(inverse)))
    return y


def repeat_kv(x, H):
    """[B, G, S, D] -> [B, H, S, D], kv head g copied to q heads g*group .. +group-1."""
    x = _f64(x)
    B, G, S, D = x.shape
    out = np.empty((B, H, S, D), dtype=np.float64)
    _load().orc_repeat_kv(B, H, G, S * D, _p(x), _p(out))
    return out


def repeat_kv_bwd(dout, G):
    """[B, H, S, D] -> [B, G, S, D] group-row sum."""
    dout = _f64(dout)
    B, H, S, D = dout.shape
    din = np.empty((B, G, S, D), dtype=np.float64)
    _load().orc_repeat_kv_bwd(B, H, G, S * D, _p(dout), _p(din))
    return din


def sdpa_head_fwd(q, k, v):
    """One head's causal SDPA on [S, D]: returns (o, lse, p)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    S, D = q.shape
    p = np.empty((S, S), dtype=np.float64)
    o = np.empty((S, D), dtype=np.float64)
    lse = np.empty(S, dtype=np.float64)
    _load().orc_sdpa_head_fwd(S, D, _p(q), _p(k), _p(v), _p(p), _p(o), _p(lse))
    return o, lse, p


def sdpa_head_bwd(q, k, v, dout):
    """One head's causal SDPA backward on [S, D]: returns (dq, dk, dv)."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    S, D = q.shape
    _, _, p = sdpa_head_fwd(q, k, v)
    dq, dk, dv = (np.empty((S, D), dtype=np.float64) for _ in range(3))
    _load().orc_sdpa_head_bwd(S, D, _p(q), _p(k), _p(v), _p(p), _p(dout), _p(dq), _p(dk), _p(dv))
    return dq, dk, dv


# --- whole pipeline -------------------------------------------------------

def attn_fwd(q, k, v, gamma_q, gamma_k, eps, theta, nthreads=None):
    """Forward of the attention core.

    q [B,S,H,D], k/v [B,S,G,D], gammas [D]. Returns a dict with out [B,S,H,D],
    lse [B,H,S], qhat [B,H,S,D], khat [B,G,S,D], rstd_q [B,S,H], rstd_k [B,S,G].
    """
    q, k, v, gq, gk = map(_f64, (q, k, v, gamma_q, gamma_k))
    B, S, H, D = q.shape
    G = k.shape[2]
    out = np.empty((B, S, H, D))
    lse = np.empty((B, H, S))
    qhat = np.empty((B, H, S, D))
    khat = np.empty((B, G, S, D))
    rq = np.empty((B, S, H))
    rk = np.empty((B, S, G))
    rc = _load().orc_attn_fwd(B, S, H, G, D, float(eps), float(theta), _p(q), _p(k), _p(v),
                              _p(gq), _p(gk), _p(out), _p(lse), _p(qhat), _p(khat), _p(rq),
                              _p(rk), head_threads(nthreads, S, 1, B * H))
    if rc:
        raise ValueError("oracle: invalid shape")
    return dict(out=out, lse=lse, qhat=qhat, khat=khat, rstd_q=rq, rstd_k=rk)


def attn_bwd(q, k, v, gamma_q, gamma_k, dout, eps, theta, nthreads=None):
    """Backward of the attention core for upstream gradient dout [B,S,H,D].

    Returns a dict with dq [B,S,H,D], dk/dv [B,S,G,D], dgamma_q/dgamma_k [D].
    """
    q, k, v, gq, gk, do = map(_f64, (q, k, v, gamma_q, gamma_k, dout))
    B, S, H, D = q.shape
    G = k.shape[2]
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    dgq = np.empty(D)
    dgk = np.empty(D)
    rc = _load().orc_attn_bwd(B, S, H, G, D, float(eps), float(theta), _p(q), _p(k), _p(v),
                              _p(gq), _p(gk), _p(do), _p(dq), _p(dk), _p(dv), _p(dgq), _p(dgk),
                              head_threads(nthreads, S, 2, B * H))
    if rc:
        raise ValueError("oracle: invalid shape")
    return dict(dq=dq, dk=dk, dv=dv, dgamma_q=dgq, dgamma_k=dgk)


def _cu(cu_seqlens) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64).reshape(-1))


def attn_fwd_packed(q, k, v, gamma_q, gamma_k, cu_seqlens, eps, theta, nthreads=None):
    """Forward over a packed batch: sample s on rows cu[s]..cu[s+1]-1.

    q [T,H,D], k/v [T,G,D]. Returns a dict with out [T,H,D], lse [H,T],
    qhat [H,T,D], khat [G,T,D], rstd_q [T,H], rstd_k [T,G].
    """
    q, k, v, gq, gk = map(_f64, (q, k, v, gamma_q, gamma_k))
    cu = _cu(cu_seqlens)
    T, H, D = q.shape
    G = k.shape[1]
    out = np.empty((T, H, D))
    lse = np.empty((H, T))
    qhat = np.empty((H, T, D))
    khat = np.empty((G, T, D))
    rq = np.empty((T, H))
    rk = np.empty((T, G))
    if cu[-1] != T:
        raise ValueError("oracle: cu_seqlens[-1] must equal the row count")
    rc = _load().orc_attn_fwd_packed(len(cu) - 1, _lp(cu), H, G, D, float(eps), float(theta),
                                     _p(q), _p(k), _p(v), _p(gq), _p(gk), _p(out), _p(lse),
                                     _p(qhat), _p(khat), _p(rq), _p(rk),
                                     head_threads(nthreads, T, 1, H))
    if rc:
        raise ValueError("oracle: invalid shape or offsets")
    return dict(out=out, lse=lse, qhat=qhat, khat=khat, rstd_q=rq, rstd_k=rk)


def attn_bwd_packed(q, k, v, gamma_q, gamma_k, cu_seqlens, dout, eps, theta, nthreads=None):
    """Backward over a packed batch for upstream gradient dout [T,H,D]."""
    q, k, v, gq, gk, do = map(_f64, (q, k, v, gamma_q, gamma_k, dout))
    cu = _cu(cu_seqlens)
    T, H, D = q.shape
    G = k.shape[1]
    if cu[-1] != T:
        raise ValueError("oracle: cu_seqlens[-1] must equal the row count")
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    dgq = np.empty(D)
    dgk = np.empty(D)
    rc = _load().orc_attn_bwd_packed(len(cu) - 1, _lp(cu), H, G, D, float(eps), float(theta),
                                     _p(q), _p(k), _p(v), _p(gq), _p(gk), _p(do), _p(dq), _p(dk),
                                     _p(dv), _p(dgq), _p(dgk), head_threads(nthreads, T, 2, H))
    if rc:
        raise ValueError("oracle: invalid shape or offsets")
    return dict(dq=dq, dk=dk, dv=dv, dgamma_q=dgq, dgamma_k=dgk)


def _idx(rows) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    return a


def attn_fwd_rows(q, k, v, gamma_q, gamma_k, eps, theta, rows, nthreads=None):
    """O rows and LSE for query rows (b, h, t); returns (o [n, D], lse [n])."""
    q, k, v, gq, gk = map(_f64, (q, k, v, gamma_q, gamma_k))
    B, S, H, D = q.shape
    G = k.shape[2]
    idx = _idx(rows)
    n = idx.shape[0]
    o = np.empty((n, D))
    lse = np.empty(n)
    rc = _load().orc_attn_fwd_rows(B, S, H, G, D, float(eps), float(theta), _p(q), _p(k), _p(v),
                                   _p(gq), _p(gk), n, _lp(idx), _p(o), _p(lse),
                                   int(nthreads or default_threads()))
    if rc:
        raise ValueError("oracle: invalid shape")
    return o, lse


def attn_dq_rows(q, k, v, gamma_q, gamma_k, dout, eps, theta, rows, nthreads=None):
    """dq rows for query rows (b, h, t); returns [n, D]."""
    q, k, v, gq, gk, do = map(_f64, (q, k, v, gamma_q, gamma_k, dout))
    B, S, H, D = q.shape
    G = k.shape[2]
    idx = _idx(rows)
    n = idx.shape[0]
    dq = np.empty((n, D))
    rc = _load().orc_attn_dq_rows(B, S, H, G, D, float(eps), float(theta), _p(q), _p(k), _p(v),
                                  _p(gq), _p(gk), _p(do), n, _lp(idx), _p(dq),
                                  int(nthreads or default_threads()))
    if rc:
        raise ValueError("oracle: invalid shape")
    return dq


def attn_dkdv_rows(q, k, v, gamma_q, gamma_k, dout, eps, theta, rows, nthreads=None):
    """dk and dv rows for key rows (b, g, j); returns (dk [n, D], dv [n, D])."""
    q, k, v, gq, gk, do = map(_f64, (q, k, v, gamma_q, gamma_k, dout))
    B, S, H, D = q.shape
    G = k.shape[2]
    idx = _idx(rows)
    n = idx.shape[0]
    dk = np.empty((n, D))
    dv = np.empty((n, D))
    rc = _load().orc_attn_dkdv_rows(B, S, H, G, D, float(eps), float(theta), _p(q), _p(k),
                                    _p(v), _p(gq), _p(gk), _p(do), n, _lp(idx), _p(dk), _p(dv),
                                    int(nthreads or default_threads()))
    if rc:
        raise ValueError("oracle: invalid shape")
    return dk, dv
