"""Pins of the oracle's packed-batch functions (Mint project report, 8.2: a
chat batch flattened to [total] rows, RoPE positions numbered inside each
sample, a block-causal mask that hides other samples' rows and, inside a
sample, the later rows).

The packed functions apply the block-causal mask to one [total, total] score
matrix per head; the checks below compare them with the batched functions
(one causal [S, S] matrix per sample), which share no masking code path with
them, and with central finite differences.
"""
import numpy as np
import pytest

import oracle


def _packed_problem(lens, H, G, D, seed):
    r = np.random.default_rng(seed)
    T = int(sum(lens))
    q = r.standard_normal((T, H, D))
    k = r.standard_normal((T, G, D))
    v = r.standard_normal((T, G, D))
    do = r.standard_normal((T, H, D))
    gq = 1 + 0.1 * r.standard_normal(D)
    gk = 1 + 0.1 * r.standard_normal(D)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    return q, k, v, do, gq, gk, cu


def test_equal_samples_equal_the_batched_oracle_bitwise():
    # masked probabilities are exact zeros in double, so the packed [T, T]
    # softmax and the batched [S, S] one add the same terms in the same order
    B, S, H, G, D, eps, theta = 3, 5, 4, 2, 8, 1e-5, 1e4
    q, k, v, do, gq, gk, cu = _packed_problem([S] * B, H, G, D, seed=3)
    pf = oracle.attn_fwd_packed(q, k, v, gq, gk, cu, eps, theta, nthreads=2)
    bf = oracle.attn_fwd(q.reshape(B, S, H, D), k.reshape(B, S, G, D), v.reshape(B, S, G, D),
                         gq, gk, eps, theta, nthreads=2)
    assert np.array_equal(pf["out"], bf["out"].reshape(B * S, H, D))
    assert np.array_equal(pf["lse"], bf["lse"].transpose(1, 0, 2).reshape(H, B * S))
    assert np.array_equal(pf["qhat"], bf["qhat"].transpose(1, 0, 2, 3).reshape(H, B * S, D))
    assert np.array_equal(pf["khat"], bf["khat"].transpose(1, 0, 2, 3).reshape(G, B * S, D))
    assert np.array_equal(pf["rstd_q"], bf["rstd_q"].reshape(B * S, H))
    assert np.array_equal(pf["rstd_k"], bf["rstd_k"].reshape(B * S, G))
    pb = oracle.attn_bwd_packed(q, k, v, gq, gk, cu, do, eps, theta, nthreads=2)
    bb = oracle.attn_bwd(q.reshape(B, S, H, D), k.reshape(B, S, G, D), v.reshape(B, S, G, D),
                         gq, gk, do.reshape(B, S, H, D), eps, theta, nthreads=2)
    assert np.array_equal(pb["dq"], bb["dq"].reshape(B * S, H, D))
    assert np.array_equal(pb["dk"], bb["dk"].reshape(B * S, G, D))
    assert np.array_equal(pb["dv"], bb["dv"].reshape(B * S, G, D))
    # dgamma sums the rows in the same (sample, position, head) order
    assert np.array_equal(pb["dgamma_q"], bb["dgamma_q"])
    assert np.array_equal(pb["dgamma_k"], bb["dgamma_k"])


@pytest.mark.parametrize("lens,H,G,D", [
    ([3, 0, 4, 5], 6, 2, 8),     # an empty sample, group 3
    ([1, 7, 2], 4, 1, 16),       # a one-row sample, MQA
])
def test_unequal_samples_equal_separate_batched_runs(lens, H, G, D):
    eps, theta = 1e-6, 1e6
    q, k, v, do, gq, gk, cu = _packed_problem(lens, H, G, D, seed=5)
    pf = oracle.attn_fwd_packed(q, k, v, gq, gk, cu, eps, theta, nthreads=1)
    pb = oracle.attn_bwd_packed(q, k, v, gq, gk, cu, do, eps, theta, nthreads=1)
    dgq = np.zeros(D)
    dgk = np.zeros(D)
    for s, L in enumerate(lens):
        if L == 0:
            continue
        a, b = cu[s], cu[s + 1]
        one = lambda x: x[a:b][None]
        bf = oracle.attn_fwd(one(q), one(k), one(v), gq, gk, eps, theta, nthreads=1)
        assert np.array_equal(pf["out"][a:b], bf["out"][0])
        assert np.array_equal(pf["lse"][:, a:b], bf["lse"][0])
        assert np.array_equal(pf["qhat"][:, a:b], bf["qhat"][0])
        assert np.array_equal(pf["khat"][:, a:b], bf["khat"][0])
        bb = oracle.attn_bwd(one(q), one(k), one(v), gq, gk, one(do), eps, theta, nthreads=1)
        assert np.array_equal(pb["dq"][a:b], bb["dq"][0])
        assert np.array_equal(pb["dk"][a:b], bb["dk"][0])
        assert np.array_equal(pb["dv"][a:b], bb["dv"][0])
        dgq += bb["dgamma_q"]
        dgk += bb["dgamma_k"]
    # the packed dgamma is one running sum over all rows: same terms, other grouping
    np.testing.assert_allclose(pb["dgamma_q"], dgq, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(pb["dgamma_k"], dgk, rtol=1e-12, atol=1e-12)


def test_samples_do_not_see_each_other():
    lens = [4, 3, 5]
    H, G, D, eps, theta = 4, 2, 8, 1e-5, 1e4
    q, k, v, do, gq, gk, cu = _packed_problem(lens, H, G, D, seed=8)
    base = oracle.attn_fwd_packed(q, k, v, gq, gk, cu, eps, theta, nthreads=1)
    a, b = cu[1], cu[2]
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    r = np.random.default_rng(9)
    q2[a:b] = r.standard_normal(q2[a:b].shape)
    k2[a:b] = r.standard_normal(k2[a:b].shape)
    v2[a:b] = r.standard_normal(v2[a:b].shape)
    pert = oracle.attn_fwd_packed(q2, k2, v2, gq, gk, cu, eps, theta, nthreads=1)
    keep = np.r_[0:a, b:cu[-1]]
    assert np.array_equal(base["out"][keep], pert["out"][keep])
    assert np.array_equal(base["lse"][:, keep], pert["lse"][:, keep])
    assert not np.array_equal(base["out"][a:b], pert["out"][a:b])


def test_packed_central_finite_differences():
    lens = [2, 0, 3]
    H, G, D, eps, theta = 2, 1, 4, 1e-5, 1e4
    q, k, v, do, gq, gk, cu = _packed_problem(lens, H, G, D, seed=11)

    def loss(q_, k_, v_, gq_, gk_):
        return float((oracle.attn_fwd_packed(q_, k_, v_, gq_, gk_, cu, eps, theta,
                                             nthreads=1)["out"] * do).sum())

    g = oracle.attn_bwd_packed(q, k, v, gq, gk, cu, do, eps, theta, nthreads=1)
    args = dict(q=q, k=k, v=v, gq=gq, gk=gk)
    grads = dict(q=g["dq"], k=g["dk"], v=g["dv"], gq=g["dgamma_q"], gk=g["dgamma_k"])
    h = 1e-6
    for name, arr in args.items():
        fd = np.zeros_like(arr)
        for i in np.ndindex(arr.shape):
            plus = {n: x.copy() for n, x in args.items()}
            minus = {n: x.copy() for n, x in args.items()}
            plus[name][i] += h
            minus[name][i] -= h
            fd[i] = (loss(**{n + "_": x for n, x in plus.items()}) -
                     loss(**{n + "_": x for n, x in minus.items()})) / (2 * h)
        scale = max(np.abs(fd).max(), 1e-3)
        assert np.abs(fd - grads[name]).max() / scale < 2e-7, name


@pytest.mark.parametrize("cu", [[1, 3, 5], [0, 3, 2, 5], [0, 2, 4]])
def test_packed_rejects_bad_offsets(cu):
    q, k, v, do, gq, gk, _ = _packed_problem([5], 2, 1, 4, seed=0)
    with pytest.raises(ValueError):
        oracle.attn_fwd_packed(q, k, v, gq, gk, cu, 1e-5, 1e4)
