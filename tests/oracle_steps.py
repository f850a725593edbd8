"""The oracle's forward and backward composed from its single steps, with an
optional rounding of Q-hat and K-hat between the prologue and the attention.

Test infrastructure (tests only). The steps are the oracle's own functions in
the pages' op order (xtrain "Phase T9", Decision 1: per-head RMSNorm, then
rotate_half RoPE at position s; "Phase T15": repeat_kv, per-head causal SDPA,
the group-row sum in the backward; Mint project report 5.4.4 and 5.5.2: RoPE
backward by the negative angle, RMSNorm backward). Without rounding the
composition equals the whole-pipeline oracle bitwise (a CPU pin checks this).

With ``round_hat`` (a function on float64 arrays) the normed-and-rotated rows
are rounded before they enter the attention, which is where xtrain "Phase
T12: bf16 mixed precision" stores activations in bf16: the rounding the GPU
path applies by design. Comparing the GPU with this composition isolates the
attention arithmetic from that prescribed rounding, which matters when large
gammas scale the scores (an ulp of bf16 in Q-hat then moves a probability by
more than the 2e-2 band).
"""
import numpy as np

import oracle


def _positions(B, S, NH):
    return np.broadcast_to(np.arange(S, dtype=np.int64)[None, :, None], (B, S, NH))


def _hat(x, gamma, eps, theta):
    """[B, S, NH, D] -> (hat [B, NH, S, D], rstd [B, S, NH])"""
    B, S, NH, _ = x.shape
    y, rstd = oracle.rmsnorm_rows(x, gamma, eps)
    yr = oracle.rope_rows(y, _positions(B, S, NH), theta)
    return np.ascontiguousarray(yr.transpose(0, 2, 1, 3)), rstd


def forward_backward(x, eps, theta, round_hat=None):
    """x: float64 inputs q, k, v, dout, gamma_q, gamma_k in the boundary
    layouts. Returns (fwd dict like oracle.attn_fwd, bwd dict like
    oracle.attn_bwd)."""
    q, k, v, do = x["q"], x["k"], x["v"], x["dout"]
    B, S, H, D = q.shape
    G = k.shape[2]
    qhat, rq = _hat(q, x["gamma_q"], eps, theta)
    khat, rk = _hat(k, x["gamma_k"], eps, theta)
    if round_hat is not None:
        qhat, khat = round_hat(qhat), round_hat(khat)
    vh = np.ascontiguousarray(v.transpose(0, 2, 1, 3))
    krep = oracle.repeat_kv(khat, H)
    vrep = oracle.repeat_kv(vh, H)
    doh = np.ascontiguousarray(do.transpose(0, 2, 1, 3))
    out = np.empty((B, H, S, D))
    lse = np.empty((B, H, S))
    dqh = np.empty((B, H, S, D))
    dkrep = np.empty((B, H, S, D))
    dvrep = np.empty((B, H, S, D))
    for b in range(B):
        for h in range(H):
            out[b, h], lse[b, h], _ = oracle.sdpa_head_fwd(qhat[b, h], krep[b, h], vrep[b, h])
            dqh[b, h], dkrep[b, h], dvrep[b, h] = oracle.sdpa_head_bwd(
                qhat[b, h], krep[b, h], vrep[b, h], doh[b, h])
    dkh = oracle.repeat_kv_bwd(dkrep, G)
    dv = oracle.repeat_kv_bwd(dvrep, G).transpose(0, 2, 1, 3)
    dyq = oracle.rope_rows(dqh.transpose(0, 2, 1, 3), _positions(B, S, H), theta, inverse=True)
    dyk = oracle.rope_rows(dkh.transpose(0, 2, 1, 3), _positions(B, S, G), theta, inverse=True)
    dq, dgq = oracle.rmsnorm_rows_bwd(q, x["gamma_q"], eps, dyq)
    dk, dgk = oracle.rmsnorm_rows_bwd(k, x["gamma_k"], eps, dyk)
    fwd = dict(out=np.ascontiguousarray(out.transpose(0, 2, 1, 3)), lse=lse, qhat=qhat,
               khat=khat, rstd_q=rq, rstd_k=rk)
    bwd = dict(dq=dq, dk=dk, dv=np.ascontiguousarray(dv), dgamma_q=dgq, dgamma_k=dgk)
    return fwd, bwd
