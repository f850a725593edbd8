"""Pins of the CPU oracle to things other than itself.

Each check is chosen so that a plausible slip in the oracle (a dropped term,
a wrong sign or index, a transposed operand, a wrong group mapping) fails:
library routines (torch fp64 rms_norm / SDPA / autograd), closed forms,
invariants stated on the pages, central finite differences of the whole
forward, brute force on tiny inputs, and a hand-worked example.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rng(seed=0):
    return np.random.default_rng(seed)


# --------------------------------------------------------------------------
# RMSNorm (Mint report 5.5.1 / 5.5.2; xtrain T9 Decision 1)
# --------------------------------------------------------------------------

def test_rmsnorm_matches_torch_rms_norm_fwd_and_autograd():
    r = rng(1)
    x = r.standard_normal((37, 24))
    g = 1 + 0.1 * r.standard_normal(24)
    dy = r.standard_normal((37, 24))
    eps = 1e-5
    y, rstd = oracle.rmsnorm_rows(x, g, eps)
    xt = torch.tensor(x, requires_grad=True)
    gt = torch.tensor(g, requires_grad=True)
    yt = F.rms_norm(xt, (24,), weight=gt, eps=eps)
    np.testing.assert_allclose(y, yt.detach().numpy(), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(rstd, 1 / np.sqrt((x ** 2).mean(-1) + eps), rtol=1e-13)
    yt.backward(torch.tensor(dy))
    dx, dg = oracle.rmsnorm_rows_bwd(x, g, eps, dy)
    np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(dg, gt.grad.numpy(), rtol=1e-11, atol=1e-13)


@pytest.mark.parametrize("eps", [1e-5, 1e-6, 0.3])
def test_rmsnorm_unit_gamma_closed_form(eps):
    # with gamma = 1: mean(y^2) = ms / (ms + eps)
    x = rng(2).standard_normal((50, 16)) * 0.01
    y, _ = oracle.rmsnorm_rows(x, np.ones(16), eps)
    ms = (x ** 2).mean(-1)
    np.testing.assert_allclose((y ** 2).mean(-1), ms / (ms + eps), rtol=1e-13)


def test_rmsnorm_scale_invariance_without_eps():
    x = rng(3).standard_normal((9, 8))
    g = 1 + 0.1 * rng(4).standard_normal(8)
    y1, _ = oracle.rmsnorm_rows(x, g, 0.0)
    y2, _ = oracle.rmsnorm_rows(7.5 * x, g, 0.0)
    np.testing.assert_allclose(y1, y2, rtol=1e-14, atol=1e-15)


def test_rmsnorm_backward_identity():
    # sum_j x_j dx_j = eps * dot / rms^3, from dx_j = g dy / rms - x dot / (d rms^3)
    r = rng(5)
    x = r.standard_normal((20, 32))
    g = 1 + 0.1 * r.standard_normal(32)
    dy = r.standard_normal((20, 32))
    eps = 0.05
    dx, _ = oracle.rmsnorm_rows_bwd(x, g, eps, dy)
    rms = np.sqrt((x ** 2).mean(-1) + eps)
    dot = (g * dy * x).sum(-1)
    np.testing.assert_allclose((x * dx).sum(-1), eps * dot / rms ** 3, rtol=1e-9, atol=1e-13)


# --------------------------------------------------------------------------
# RoPE (Mint report 5.4.1-5.4.4; xtrain T9 diff table)
# --------------------------------------------------------------------------

def test_rope_position_zero_is_identity_bitwise():
    x = rng(6).standard_normal((11, 16))
    y = oracle.rope_rows(x, np.zeros(11, dtype=np.int64), 1e4)
    assert np.array_equal(x, y)


@pytest.mark.parametrize("D,theta", [(16, 1e4), (64, 1e4), (128, 1e6), (2, 1e4)])
def test_rope_equals_complex_rotation(D, theta):
    # pair (i, i + D/2) as the complex number z = x_i + i x_{i+D/2}, rotated by
    # exp(i * pos * theta^(-2i/D))
    r = rng(7)
    pos = r.integers(0, 20000, size=13)
    x = r.standard_normal((13, D))
    y = oracle.rope_rows(x, pos, theta)
    half = D // 2
    freq = theta ** (-2.0 * np.arange(half) / D)
    z = (x[:, :half] + 1j * x[:, half:]) * np.exp(1j * pos[:, None] * freq[None, :])
    # angles reach 2e4 rad, so one ulp of the angle is ~4e-12 of the result
    np.testing.assert_allclose(y[:, :half], z.real, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(y[:, half:], z.imag, rtol=1e-10, atol=1e-10)


def test_rope_preserves_norm_and_inverts():
    r = rng(8)
    x = r.standard_normal((40, 64))
    pos = r.integers(0, 16384, size=40)
    y = oracle.rope_rows(x, pos, 1e6)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-14)
    back = oracle.rope_rows(y, pos, 1e6, inverse=True)
    np.testing.assert_allclose(back, x, rtol=1e-12, atol=1e-12)


def test_rope_relative_position_property():
    # q_t^R . k_j^R depends only on t - j (Mint report 5.4.3)
    r = rng(9)
    q = r.standard_normal(32)
    k = r.standard_normal(32)
    for t, j, c in [(5, 2, 100), (17, 17, 3), (300, 7, 1234)]:
        a = oracle.rope_rows(q[None], [t], 1e4)[0] @ oracle.rope_rows(k[None], [j], 1e4)[0]
        b = oracle.rope_rows(q[None], [t + c], 1e4)[0] @ oracle.rope_rows(k[None], [j + c], 1e4)[0]
        assert abs(a - b) < 1e-11 * max(1.0, abs(a))


# --------------------------------------------------------------------------
# repeat_kv (xtrain T15 "What is GQA" and Decision 2)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("B,H,G", [(2, 6, 2), (1, 8, 2), (3, 4, 4), (1, 16, 1)])
def test_repeat_kv_forward_and_group_sum(B, H, G):
    r = rng(10)
    S, D = 5, 4
    x = r.standard_normal((B, G, S, D))
    out = oracle.repeat_kv(x, H)
    group = H // G
    for qh in range(H):
        assert np.array_equal(out[:, qh], x[:, qh // group])  # adjacent grouping
    dout = r.standard_normal((B, H, S, D))
    din = oracle.repeat_kv_bwd(dout, G)
    brute = np.zeros_like(x)
    for b in range(B):
        for kvh in range(G):
            for rr in range(group):
                brute[b, kvh] += dout[b, kvh * group + rr]
    np.testing.assert_allclose(din, brute, rtol=1e-15, atol=0)
    # and it is the adjoint of the forward (autograd of repeat_interleave)
    xt = torch.tensor(x, requires_grad=True)
    torch.repeat_interleave(xt, group, dim=1).backward(torch.tensor(dout))
    np.testing.assert_allclose(din, xt.grad.numpy(), rtol=1e-15, atol=1e-15)
    if group == 1:
        assert np.array_equal(din, dout)


# --------------------------------------------------------------------------
# One head's causal SDPA (xtrain T5 pipeline; Mint report 5.3.1)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("S,D", [(1, 4), (7, 8), (33, 16), (64, 64)])
def test_sdpa_head_matches_torch_sdpa_and_autograd(S, D):
    r = rng(11)
    q, k, v, do = (r.standard_normal((S, D)) for _ in range(4))
    o, lse, p = oracle.sdpa_head_fwd(q, k, v)
    qt, kt, vt = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    ot = F.scaled_dot_product_attention(qt[None], kt[None], vt[None], is_causal=True)[0]
    np.testing.assert_allclose(o, ot.detach().numpy(), rtol=1e-12, atol=1e-13)
    scores = (torch.tensor(q) @ torch.tensor(k).T) / math.sqrt(D)
    scores = scores.masked_fill(torch.triu(torch.ones(S, S, dtype=torch.bool), 1), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(scores, -1).numpy(), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(p.sum(1), 1.0, rtol=1e-14)
    assert np.all(np.triu(p, 1) == 0.0)
    ot.backward(torch.tensor(do))
    dq, dk, dv = oracle.sdpa_head_bwd(q, k, v, do)
    np.testing.assert_allclose(dq, qt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, kt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, vt.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_sdpa_closed_forms():
    r = rng(12)
    S, D = 19, 8
    q = r.standard_normal((S, D))
    v = r.standard_normal((S, D))
    kvec = r.standard_normal(D)
    k = np.tile(kvec, (S, 1))  # constant key: uniform attention over the prefix
    o, lse, p = oracle.sdpa_head_fwd(q, k, v)
    t = np.arange(S)
    np.testing.assert_allclose(o, np.cumsum(v, 0) / (t + 1)[:, None], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, q @ kvec / math.sqrt(D) + np.log(t + 1), rtol=1e-12, atol=1e-12)
    # row 0 has exactly one admissible key
    k2 = r.standard_normal((S, D))
    o2, lse2, _ = oracle.sdpa_head_fwd(q, k2, v)
    assert np.array_equal(o2[0], v[0])
    assert lse2[0] == pytest.approx(q[0] @ k2[0] / math.sqrt(D), rel=1e-14)


def test_sdpa_backward_sum_rules():
    # rows of dS sum to 0  => sum_j dk_j = 0 ; rows of P sum to 1 => sum_j dv_j = sum_t do_t
    r = rng(13)
    S, D = 23, 16
    q, k, v, do = (r.standard_normal((S, D)) for _ in range(4))
    dq, dk, dv = oracle.sdpa_head_bwd(q, k, v, do)
    np.testing.assert_allclose(dk.sum(0), 0.0, atol=1e-12)
    np.testing.assert_allclose(dv.sum(0), do.sum(0), rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# Whole pipeline
# --------------------------------------------------------------------------

def _problem(B, S, H, G, D, seed, gamma_scale=0.1):
    r = rng(seed)
    q = r.standard_normal((B, S, H, D))
    k = r.standard_normal((B, S, G, D))
    v = r.standard_normal((B, S, G, D))
    do = r.standard_normal((B, S, H, D))
    gq = 1 + gamma_scale * r.standard_normal(D)
    gk = 1 + gamma_scale * r.standard_normal(D)
    return q, k, v, do, gq, gk


def _loss(q, k, v, gq, gk, do, eps, theta):
    return float((oracle.attn_fwd(q, k, v, gq, gk, eps, theta, nthreads=1)["out"] * do).sum())


@pytest.mark.parametrize("B,S,H,G,D,eps,theta", [
    (2, 5, 6, 2, 8, 1e-5, 1e4),      # group 3, B > 1
    (1, 16, 2, 2, 16, 1e-5, 1e4),    # the tiny MHA fp32 shape
    (1, 7, 4, 1, 4, 1e-6, 1e6),      # MQA, non-square
])
def test_whole_pipeline_central_finite_differences(B, S, H, G, D, eps, theta):
    q, k, v, do, gq, gk = _problem(B, S, H, G, D, seed=14)
    g = oracle.attn_bwd(q, k, v, gq, gk, do, eps, theta, nthreads=1)
    h = 1e-6
    args = dict(q=q, k=k, v=v, gq=gq, gk=gk)
    grads = dict(q=g["dq"], k=g["dk"], v=g["dv"], gq=g["dgamma_q"], gk=g["dgamma_k"])
    for name, arr in args.items():
        fd = np.zeros_like(arr)
        for i in np.ndindex(arr.shape):
            plus = {n: a.copy() for n, a in args.items()}
            minus = {n: a.copy() for n, a in args.items()}
            plus[name][i] += h
            minus[name][i] -= h
            lp = _loss(plus["q"], plus["k"], plus["v"], plus["gq"], plus["gk"], do, eps, theta)
            lm = _loss(minus["q"], minus["k"], minus["v"], minus["gq"], minus["gk"], do, eps, theta)
            fd[i] = (lp - lm) / (2 * h)
        scale = max(np.abs(fd).max(), 1e-3)
        err = np.abs(fd - grads[name]).max() / scale
        assert err < 2e-7, (name, err)


def test_group_one_equals_mha_composition_bitwise():
    # G = H: the pipeline equals norm -> rope -> per-head SDPA with no repeat_kv
    B, S, H, D = 2, 9, 3, 8
    q, k, v, do, gq, gk = _problem(B, S, H, H, D, seed=15)
    eps, theta = 1e-5, 1e4
    f = oracle.attn_fwd(q, k, v, gq, gk, eps, theta, nthreads=3)
    pos = np.broadcast_to(np.arange(S)[None, :, None], (B, S, H))
    qn, _ = oracle.rmsnorm_rows(q, gq, eps)
    kn, _ = oracle.rmsnorm_rows(k, gk, eps)
    qr = oracle.rope_rows(qn, pos, theta)
    kr = oracle.rope_rows(kn, pos, theta)
    for b in range(B):
        for h in range(H):
            o, lse, _ = oracle.sdpa_head_fwd(qr[b, :, h], kr[b, :, h], v[b, :, h])
            assert np.array_equal(f["out"][b, :, h], o)
            assert np.array_equal(f["lse"][b, h], lse)
            assert np.array_equal(f["qhat"][b, h], qr[b, :, h])


def test_gqa_equals_mha_on_repeated_kv():
    B, S, H, G, D = 2, 11, 6, 2, 8
    q, k, v, do, gq, gk = _problem(B, S, H, G, D, seed=16)
    eps, theta = 1e-5, 1e4
    group = H // G
    kr = np.repeat(k, group, axis=2)
    vr = np.repeat(v, group, axis=2)
    a = oracle.attn_fwd(q, k, v, gq, gk, eps, theta)
    m = oracle.attn_fwd(q, kr, vr, gq, gk, eps, theta)
    assert np.array_equal(a["out"], m["out"])
    assert np.array_equal(a["lse"], m["lse"])
    ga = oracle.attn_bwd(q, k, v, gq, gk, do, eps, theta)
    gm = oracle.attn_bwd(q, kr, vr, gq, gk, do, eps, theta)
    assert np.array_equal(ga["dq"], gm["dq"])
    # the shared kv head receives the sum of its group's gradients
    np.testing.assert_allclose(ga["dv"], gm["dv"].reshape(B, S, G, group, D).sum(3), rtol=1e-12,
                               atol=1e-13)
    np.testing.assert_allclose(ga["dk"], gm["dk"].reshape(B, S, G, group, D).sum(3), rtol=1e-11,
                               atol=1e-12)
    np.testing.assert_allclose(ga["dgamma_k"], gm["dgamma_k"], rtol=1e-11)


def test_thread_count_does_not_change_results():
    q, k, v, do, gq, gk = _problem(2, 13, 4, 2, 8, seed=17)
    a = oracle.attn_bwd(q, k, v, gq, gk, do, 1e-5, 1e4, nthreads=1)
    b = oracle.attn_bwd(q, k, v, gq, gk, do, 1e-5, 1e4, nthreads=5)
    for key in a:
        assert np.array_equal(a[key], b[key]), key


def test_hand_worked_example():
    with open(os.path.join(GOLDEN, "hand_worked_s2_d2.json")) as f:
        gold = json.load(f)
    inp = gold["inputs"]
    f = oracle.attn_fwd(np.array(inp["q"]), np.array(inp["k"]), np.array(inp["v"]),
                        np.array(inp["gamma_q"]), np.array(inp["gamma_k"]),
                        inp["eps"], inp["theta"])
    env = {n: getattr(math, n) for n in ("sqrt", "sin", "cos", "exp", "log")}
    ex = gold["expected_expr"]
    for name in ("s10", "s11", "p10", "p11"):
        env[name] = eval(ex[name], {}, env)

    def ev(x):
        return np.array(x if not isinstance(x, str) else eval(x, {}, env)) if not isinstance(
            x, list) else np.array([ev(e) for e in x])

    for key in ("out", "lse", "qhat", "khat"):
        np.testing.assert_allclose(f[key], ev(ex[key]), rtol=1e-14, atol=1e-15, err_msg=key)


def test_rows_api_equals_whole_api():
    B, S, H, G, D = 2, 21, 6, 2, 8
    q, k, v, do, gq, gk = _problem(B, S, H, G, D, seed=18)
    eps, theta = 1e-5, 1e4
    f = oracle.attn_fwd(q, k, v, gq, gk, eps, theta)
    g = oracle.attn_bwd(q, k, v, gq, gk, do, eps, theta)
    qrows = [(b, h, t) for b in range(B) for h in range(H) for t in range(S)]
    o, lse = oracle.attn_fwd_rows(q, k, v, gq, gk, eps, theta, qrows)
    dq = oracle.attn_dq_rows(q, k, v, gq, gk, do, eps, theta, qrows)
    for i, (b, h, t) in enumerate(qrows):
        np.testing.assert_allclose(o[i], f["out"][b, t, h], rtol=1e-12, atol=1e-13)
        assert lse[i] == pytest.approx(f["lse"][b, h, t], rel=1e-13, abs=1e-13)
        np.testing.assert_allclose(dq[i], g["dq"][b, t, h], rtol=1e-10, atol=1e-12)
    krows = [(b, gg, j) for b in range(B) for gg in range(G) for j in range(S)]
    dk, dv = oracle.attn_dkdv_rows(q, k, v, gq, gk, do, eps, theta, krows)
    for i, (b, gg, j) in enumerate(krows):
        np.testing.assert_allclose(dk[i], g["dk"][b, j, gg], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(dv[i], g["dv"][b, j, gg], rtol=1e-10, atol=1e-12)


def test_oracle_rejects_bad_shapes():
    q, k, v, do, gq, gk = _problem(1, 4, 3, 2, 8, seed=19)  # 3 % 2 != 0
    with pytest.raises(ValueError):
        oracle.attn_fwd(q, k, v, gq, gk, 1e-5, 1e4)


def test_step_composition_equals_whole_pipeline_bitwise():
    # tests/oracle_steps.py composes the oracle's single steps (used, with a bf16
    # rounding of Q-hat and K-hat, by the large-score GPU stress test); without the
    # rounding it must reproduce the whole-pipeline oracle exactly
    import oracle_steps
    B, S, H, G, D = 2, 19, 6, 2, 8
    q, k, v, do, gq, gk = _problem(B, S, H, G, D, seed=20)
    eps, theta = 1e-5, 1e4
    x = dict(q=q, k=k, v=v, dout=do, gamma_q=gq, gamma_k=gk)
    cf, cg = oracle_steps.forward_backward(x, eps, theta)
    f = oracle.attn_fwd(q, k, v, gq, gk, eps, theta)
    g = oracle.attn_bwd(q, k, v, gq, gk, do, eps, theta)
    for key in f:
        assert np.array_equal(cf[key], f[key]), key
    for key in g:
        assert np.array_equal(cg[key], g[key]), key


def test_step_composition_rounding_reaches_the_attention():
    # the rounding hook acts between the prologue and the attention: rounding
    # Q-hat/K-hat to a coarse grid changes out, and the identity leaves it alone
    import oracle_steps
    q, k, v, do, gq, gk = _problem(1, 9, 2, 1, 8, seed=21)
    x = dict(q=q, k=k, v=v, dout=do, gamma_q=gq, gamma_k=gk)
    base, _ = oracle_steps.forward_backward(x, 1e-5, 1e4)
    same, _ = oracle_steps.forward_backward(x, 1e-5, 1e4, round_hat=lambda a: a.copy())
    coarse, _ = oracle_steps.forward_backward(x, 1e-5, 1e4, round_hat=lambda a: np.round(a, 1))
    assert np.array_equal(same["out"], base["out"])
    assert np.array_equal(coarse["qhat"], np.round(base["qhat"], 1))
    assert not np.allclose(coarse["out"], base["out"], rtol=1e-6, atol=0)
