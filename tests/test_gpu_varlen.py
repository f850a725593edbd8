"""GPU parity of packed batches (Mint project report, 8.2: samples flattened
into one row dimension, positions numbered inside each sample, a
block-causal mask between samples) through the C ABI, against the oracle's
packed forward and backward on the same seeded inputs.

Bars as for the batched calls: max relative error <= 2e-2 (bf16) / 1e-4
(fp32) per output tensor and the same argmax along every output row (near-ties
excepted). The full-size packed batch is checked on rows the oracle computes
one by one (each sample is an independent problem).
"""
import numpy as np
import pytest
import torch

import oracle
from causal_gqa_attention_xt_gb300 import build as xbuild
from causal_gqa_attention_xt_gb300 import xt
from causal_gqa_attention_xt_gb300.inputs import (PACKED_WORKLOADS, PackedWorkload, Workload,
                                                  make_inputs, make_packed_inputs, to_f64)

from parity_metrics import TOL, as_f64, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    xbuild.build()
    xt.lib()


def run_varlen(w: PackedWorkload, cpu: dict):
    d = {k: v.cuda() for k, v in cpu.items()}
    cu = d["cu_seqlens"]
    f = xt.xt_attn_fwd_varlen(d["q"], d["k"], d["v"], d["gamma_q"], d["gamma_k"], cu, w.max_len,
                              w.eps, w.theta)
    g = xt.xt_attn_bwd_varlen(d["q"], d["k"], d["v"], d["gamma_q"], d["gamma_k"], cu, w.max_len,
                              f, d["dout"], w.eps, w.theta)
    assert xt.xt_attn_check() == xt.XT_OK
    return f, g


CASES = [
    # an empty sample, a one-row sample, tile-ragged lengths, group 4
    PackedWorkload("varlen_group4_d64_bf16", (1, 130, 0, 257, 64), 8, 2, 64, 1e4, 1e-5, "bf16"),
    PackedWorkload("varlen_mha_d128_bf16", (300, 17, 129), 4, 4, 128, 1e6, 1e-6, "bf16"),
    PackedWorkload("varlen_mqa_d128_bf16", (520, 200, 128), 16, 1, 128, 1e6, 1e-6, "bf16"),
    PackedWorkload("varlen_group2_d32_f32", (33, 1, 70), 4, 2, 32, 1e4, 1e-5, "f32"),
    PackedWorkload("varlen_group2_d32_bf16", (33, 1, 300, 130), 4, 2, 32, 1e4, 1e-5, "bf16"),
    PackedWorkload("varlen_d128_f32", (140, 0, 65), 2, 1, 128, 1e6, 1e-6, "f32"),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_packed_batch_every_output(w):
    cpu = make_packed_inputs(w)
    f, g = run_varlen(w, cpu)
    x = to_f64({k: v for k, v in cpu.items() if k != "cu_seqlens"})
    rf = oracle.attn_fwd_packed(x["q"], x["k"], x["v"], x["gamma_q"], x["gamma_k"], w.cu, w.eps,
                                w.theta)
    rg = oracle.attn_bwd_packed(x["q"], x["k"], x["v"], x["gamma_q"], x["gamma_k"], w.cu,
                                x["dout"], w.eps, w.theta)
    tol = TOL[w.dtype]
    for name, got, ref in [("out", f["out"], rf["out"]), ("lse", f["lse"], rf["lse"]),
                           ("q_hat", f["q_hat"], rf["qhat"]), ("k_hat", f["k_hat"], rf["khat"]),
                           ("rstd_q", f["rstd_q"], rf["rstd_q"]),
                           ("rstd_k", f["rstd_k"], rf["rstd_k"]),
                           ("dq", g["dq"], rg["dq"]), ("dk", g["dk"], rg["dk"]),
                           ("dv", g["dv"], rg["dv"]), ("dgamma_q", g["dgamma_q"], rg["dgamma_q"]),
                           ("dgamma_k", g["dgamma_k"], rg["dgamma_k"])]:
        assert_close(f"{w.name}:{name}", got, ref, tol)


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("bf16", 64), ("f32", 64)])
def test_equal_lengths_equal_the_batched_call_bitwise(dtype, D):
    # the packed call on B samples of S rows runs the same tiles as the batched
    # call (only the row offsets differ), so every output is bitwise the same
    B, S, H, G = 3, 300, 4, 2
    bw = Workload(f"bat_{dtype}_{D}", B, S, H, G, D, 1e4, 1e-5, dtype, seed=6)
    cpu = make_inputs(bw)
    d = {k: v.cuda() for k, v in cpu.items()}
    fb = xt.xt_attn_fwd(d["q"], d["k"], d["v"], d["gamma_q"], d["gamma_k"], bw.eps, bw.theta)
    gb = xt.xt_attn_bwd(d["q"], d["k"], d["v"], d["gamma_q"], d["gamma_k"], fb, d["dout"],
                        bw.eps, bw.theta)
    cu = torch.arange(0, (B + 1) * S, S, dtype=torch.int32, device="cuda")
    flat = lambda t: t.reshape(B * S, *t.shape[2:])
    fp = xt.xt_attn_fwd_varlen(flat(d["q"]), flat(d["k"]), flat(d["v"]), d["gamma_q"],
                               d["gamma_k"], cu, S, bw.eps, bw.theta)
    gp = xt.xt_attn_bwd_varlen(flat(d["q"]), flat(d["k"]), flat(d["v"]), d["gamma_q"],
                               d["gamma_k"], cu, S, fp, flat(d["dout"]), bw.eps, bw.theta)
    assert xt.xt_attn_check() == xt.XT_OK
    hm = lambda t: t.transpose(0, 1).reshape(t.shape[1], B * S, *t.shape[3:])   # [B,X,S,..] -> [X,BS,..]
    assert torch.equal(fp["out"], flat(fb["out"]))
    assert torch.equal(fp["lse"], hm(fb["lse"]))
    assert torch.equal(fp["q_hat"], hm(fb["q_hat"]))
    assert torch.equal(fp["k_hat"], hm(fb["k_hat"]))
    assert torch.equal(fp["rstd_q"], flat(fb["rstd_q"]))
    assert torch.equal(fp["rstd_k"], flat(fb["rstd_k"]))
    for name in ("dq", "dk", "dv"):
        assert torch.equal(gp[name], flat(gb[name])), name
    # dgamma: the same rows, summed over the same per-CTA partials
    for name in ("dgamma_q", "dgamma_k"):
        assert torch.equal(gp[name], gb[name]), name


def test_full_size_packed_batch_sampled_rows():
    w = PACKED_WORKLOADS["qwen3_like_varlen_bf16"]
    cpu = make_packed_inputs(w)
    f, g = run_varlen(w, cpu)
    x = to_f64({k: v for k, v in cpu.items() if k != "cu_seqlens"})
    tol = TOL[w.dtype]
    rng = np.random.default_rng(0)
    cu = w.cu
    for s, L in enumerate(w.lens):
        a, b = cu[s], cu[s + 1]
        one = {k: x[k][a:b][None] for k in ("q", "k", "v", "dout")}
        ts = sorted(set([0, L - 1] + list(rng.integers(0, L, 3))))
        hs = [0, w.H - 1]
        rows = [(0, h, t) for h in hs for t in ts]
        o, lse = oracle.attn_fwd_rows(one["q"], one["k"], one["v"], x["gamma_q"], x["gamma_k"],
                                      w.eps, w.theta, rows)
        got_o = np.stack([as_f64(f["out"][a + t, h]) for (_, h, t) in rows])
        got_l = np.array([float(f["lse"][h, a + t]) for (_, h, t) in rows])
        assert_close(f"sample{s}:out", got_o, o, tol)
        assert_close(f"sample{s}:lse", got_l, lse, tol)
        dq = oracle.attn_dq_rows(one["q"], one["k"], one["v"], x["gamma_q"], x["gamma_k"],
                                 one["dout"], w.eps, w.theta, rows)
        got_dq = np.stack([as_f64(g["dq"][a + t, h]) for (_, h, t) in rows])
        assert_close(f"sample{s}:dq", got_dq, dq, tol)
        krows = [(0, gg, t) for gg in (0, w.G - 1) for t in ts]
        dk, dv = oracle.attn_dkdv_rows(one["q"], one["k"], one["v"], x["gamma_q"], x["gamma_k"],
                                       one["dout"], w.eps, w.theta, krows)
        got_dk = np.stack([as_f64(g["dk"][a + t, gg]) for (_, gg, t) in krows])
        got_dv = np.stack([as_f64(g["dv"][a + t, gg]) for (_, gg, t) in krows])
        assert_close(f"sample{s}:dk", got_dk, dk, tol)
        assert_close(f"sample{s}:dv", got_dv, dv, tol)


def test_bad_offsets_are_reported_and_the_next_call_is_clean():
    w = PackedWorkload("bad_cu_bf16", (100, 60), 4, 2, 64, 1e4, 1e-5, "bf16")
    cpu = make_packed_inputs(w)
    d = {k: v.cuda() for k, v in cpu.items()}
    # the last offset is not the row count, and one sample is longer than max_seqlen
    for bad in ([0, 100, 150], [0, 120, 160]):
        cu = torch.tensor(bad, dtype=torch.int32, device="cuda")
        xt.xt_attn_fwd_varlen(d["q"], d["k"], d["v"], d["gamma_q"], d["gamma_k"], cu, 100, w.eps,
                              w.theta)
        assert xt.xt_attn_check() == xt.XT_EINVAL
    f, g = run_varlen(w, cpu)   # asserts XT_OK
    assert torch.isfinite(f["out"].float()).all()
