"""GPU parity: the CUDA path through the C ABI against the CPU oracle, on the
same seeded inputs.

Bars: max relative error (max |g - r| / max |r|) <= 1e-4 for fp32 and 2e-2
for bf16 per output tensor, and the same argmax along every output row
(near-ties excepted). Every workload (small shapes, dim768, Qwen3-like, long
MQA) is compared element by element on every output against the whole
oracle; the 2^21-position case, too long for the oracle's [S, S] matrices, is
compared on rows the oracle computes one by one.
"""
import numpy as np
import pytest
import torch

import oracle
from causal_gqa_attention_xt_gb300 import build as xbuild
from causal_gqa_attention_xt_gb300 import xt
from causal_gqa_attention_xt_gb300.inputs import WORKLOADS, Workload, make_inputs, to_f64

from parity_metrics import TOL, as_f64, assert_close, max_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    xbuild.build()
    xt.lib()


def run_gpu(w: Workload, cpu: dict):
    dev = {k: v.cuda() for k, v in cpu.items()}
    f = xt.xt_attn_fwd(dev["q"], dev["k"], dev["v"], dev["gamma_q"], dev["gamma_k"], w.eps, w.theta)
    g = xt.xt_attn_bwd(dev["q"], dev["k"], dev["v"], dev["gamma_q"], dev["gamma_k"], f,
                       dev["dout"], w.eps, w.theta)
    assert xt.xt_attn_check() == xt.XT_OK
    return f, g


def oracle_full(w: Workload, x: dict):
    f = oracle.attn_fwd(x["q"], x["k"], x["v"], x["gamma_q"], x["gamma_k"], w.eps, w.theta)
    g = oracle.attn_bwd(x["q"], x["k"], x["v"], x["gamma_q"], x["gamma_k"], x["dout"], w.eps,
                        w.theta)
    return f, g


def compare_all(w, f, g, rf, rg):
    tol = TOL[w.dtype]
    errs = {}
    for name, got, ref in [("out", f["out"], rf["out"]), ("lse", f["lse"], rf["lse"]),
                           ("q_hat", f["q_hat"], rf["qhat"]), ("k_hat", f["k_hat"], rf["khat"]),
                           ("rstd_q", f["rstd_q"], rf["rstd_q"]),
                           ("rstd_k", f["rstd_k"], rf["rstd_k"]),
                           ("dq", g["dq"], rg["dq"]), ("dk", g["dk"], rg["dk"]),
                           ("dv", g["dv"], rg["dv"]), ("dgamma_q", g["dgamma_q"], rg["dgamma_q"]),
                           ("dgamma_k", g["dgamma_k"], rg["dgamma_k"])]:
        errs[name] = assert_close(f"{w.name}:{name}", got, ref, tol)
    return errs


SMALL = [
    WORKLOADS["tiny_mha_f32"],
    WORKLOADS["gqa_bf16"],
    Workload("ragged_group3_bf16", 2, 200, 6, 2, 64, 1e4, 1e-5, "bf16"),
    Workload("ragged_mqa_d128_bf16", 1, 333, 4, 1, 128, 1e6, 1e-6, "bf16"),
    Workload("mha_d128_bf16", 1, 384, 2, 2, 128, 1e6, 1e-6, "bf16"),
    Workload("one_token_bf16", 3, 1, 4, 2, 64, 1e4, 1e-5, "bf16"),
    Workload("s129_bf16", 1, 129, 2, 1, 64, 1e4, 1e-5, "bf16"),
    Workload("s17_f32", 1, 17, 4, 2, 32, 1e4, 1e-5, "f32"),
    Workload("ragged_d128_f32", 1, 130, 2, 1, 128, 1e6, 1e-6, "f32"),
    Workload("d8_group1_f32", 2, 37, 3, 3, 8, 1e4, 1e-5, "f32"),
    # head counts whose per-position chunks in the streaming kernels are uneven
    # (a q chunk and a k chunk of different sizes, a partial q chunk)
    Workload("chunks_h20_g5_bf16", 1, 150, 20, 5, 64, 1e4, 1e-5, "bf16"),
    Workload("chunks_h48_g16_d128_bf16", 1, 140, 48, 16, 128, 1e6, 1e-6, "bf16"),
    Workload("chunks_h12_g4_f32", 1, 70, 12, 4, 64, 1e4, 1e-5, "f32"),
    # head_dim 32 on the tensor cores (64-byte swizzled tiles)
    Workload("d32_group3_ragged_bf16", 2, 200, 6, 2, 32, 1e4, 1e-5, "bf16"),
    Workload("d32_mqa_bf16", 1, 520, 8, 1, 32, 1e6, 1e-6, "bf16"),
    Workload("d32_one_tile_bf16", 3, 128, 4, 4, 32, 1e4, 1e-5, "bf16"),
    WORKLOADS["dim768_hd32_bf16"],
    # one kv head for many query heads: the dK/dV work of a key tile is split over
    # several CTAs and their partials summed in a fixed order
    Workload("split_mqa_d128_bf16", 1, 2048, 16, 1, 128, 1e6, 1e-6, "bf16"),
    Workload("split_mqa_ragged_d64_bf16", 1, 1000, 8, 1, 64, 1e4, 1e-5, "bf16"),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_small_shapes_every_output(w):
    cpu = make_inputs(w)
    f, g = run_gpu(w, cpu)
    rf, rg = oracle_full(w, to_f64(cpu))
    compare_all(w, f, g, rf, rg)


def test_sharp_scores_f32():
    # gammas near 4 scale the scores by ~16, so row maxima move from tile to tile
    w = Workload("sharp_f32", 1, 520, 4, 2, 64, 1e4, 1e-5, "f32", seed=3)
    cpu = make_inputs(w, gamma_offset=4.0, gamma_scale=0.5)
    f, g = run_gpu(w, cpu)
    rf, rg = oracle_full(w, to_f64(cpu))
    compare_all(w, f, g, rf, rg)


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("bf16", 64), ("f32", 64)])
def test_late_dominant_keys_force_running_max_jumps(dtype, D):
    # Every query row is the same vector u, and so is every key from position
    # 256 on. After QK-norm + RoPE the score of key j for query t is
    # n(u) . R(j - t) n(u) / sqrt(D): about sqrt(D) on and near the diagonal and
    # O(1) for the random keys before 256. Rows past 256 therefore see their
    # running max jump by several units at the diagonal tile. Element sizes
    # stay those of gamma ~ 1, so bf16 rounding of Qhat/Khat stays small.
    w = Workload(f"late_keys_{dtype}_d{D}", 2, 600, 4, 2, D, 1e4, 1e-5, dtype, seed=4)
    cpu = make_inputs(w)
    u = cpu["q"][0, 0, 0].clone()
    cpu["q"][:] = u
    cpu["k"][:, 256:] = u
    f, g = run_gpu(w, cpu)
    rf, rg = oracle_full(w, to_f64(cpu))
    compare_all(w, f, g, rf, rg)


def _bf16_round(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).double().numpy()


@pytest.mark.parametrize("D", [128, 64])
def test_large_scores_bf16_against_the_oracle_with_bf16_hat_rows(D):
    """bf16 with gammas near 3 (scores up to ~9 sqrt(D), ~100 at D = 128) and the
    late-key construction above: running maxima jump by tens of log2 units past
    the lazy-rescale threshold while every score is large. At these magnitudes
    the bf16 storage of Q-hat and K-hat that the precision table of xtrain
    "Phase T12" prescribes moves single probabilities by more than 2e-2, so the
    reference is the oracle composed from its steps with its own Q-hat/K-hat
    rounded to bf16 where the GPU stores them (tests/oracle_steps.py); every
    other step stays in double, and the bar stays 2e-2 with the argmax rule."""
    w = Workload(f"large_scores_bf16_d{D}", 1, 600, 4, 2, D, 1e4, 1e-5, "bf16", seed=8)
    cpu = make_inputs(w, gamma_offset=3.0, gamma_scale=0.3)
    u = cpu["q"][0, 0, 0].clone()
    cpu["q"][:, ::2] = u                      # every other query row is u
    cpu["k"][:, 256:] = u                     # late keys equal to it
    f, g = run_gpu(w, cpu)
    import oracle_steps
    rf, rg = oracle_steps.forward_backward(to_f64(cpu), w.eps, w.theta, round_hat=_bf16_round)
    compare_all(w, f, g, rf, rg)


def test_forward_and_backward_are_bitwise_deterministic():
    w = WORKLOADS["gqa_bf16"]
    cpu = make_inputs(w)
    f1, g1 = run_gpu(w, cpu)
    f2, g2 = run_gpu(w, cpu)
    for a, b in list(zip(f1.values(), f2.values())) + list(zip(g1.values(), g2.values())):
        assert torch.equal(a, b)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_gqa_forward_equals_mha_on_repeated_kv_bitwise(dtype):
    w = Workload("gqa_vs_mha", 2, 300, 8, 2, 64, 1e4, 1e-5, dtype, seed=5)
    cpu = make_inputs(w)
    rep = dict(cpu)
    rep["k"] = cpu["k"].repeat_interleave(4, dim=2).contiguous()
    rep["v"] = cpu["v"].repeat_interleave(4, dim=2).contiguous()
    f_g, g_g = run_gpu(w, cpu)
    f_m, g_m = run_gpu(w.with_(G=8), rep)
    assert torch.equal(f_g["out"], f_m["out"])
    assert torch.equal(f_g["lse"], f_m["lse"])
    assert torch.equal(f_g["q_hat"], f_m["q_hat"])
    # the shared kv head's gradient is the sum of the group's gradients
    B, S, _, D = cpu["q"].shape
    dv_sum = as_f64(g_m["dv"]).reshape(B, S, 2, 4, D).sum(3)
    assert max_rel_err(g_g["dv"], dv_sum) <= TOL[dtype]


def test_group_one_matches_oracle_mha():
    w = Workload("mha_group1", 2, 260, 4, 4, 64, 1e4, 1e-5, "bf16", seed=6)
    cpu = make_inputs(w)
    f, g = run_gpu(w, cpu)
    rf, rg = oracle_full(w, to_f64(cpu))
    compare_all(w, f, g, rf, rg)


# ------------------------------------------------------------------ full sizes

@pytest.mark.parametrize("name", ["dim768_mha_bf16", "dim768_gqa_bf16"])
def test_dim768_full_oracle(name):
    w = WORKLOADS[name]
    cpu = make_inputs(w)
    f, g = run_gpu(w, cpu)
    rf, rg = oracle_full(w, to_f64(cpu))
    compare_all(w, f, g, rf, rg)


def _gpu_to_host(f, g):
    """The GPU results on the host (frees their device memory before the oracle runs)."""
    f = {k: v.cpu() for k, v in f.items()}
    g = {k: v.cpu() for k, v in g.items()}
    torch.cuda.empty_cache()
    return f, g


@pytest.mark.parametrize("name", ["qwen3_like_bf16", "mqa_long_bf16"])
def test_full_size_oracle_every_output(name):
    """The Qwen3-like and the long-context MQA workloads at full size against the
    whole oracle, element by element on every output (out, lse, q_hat, k_hat,
    rstd_q, rstd_k, dq, dk, dv, dgamma_q, dgamma_k) with the argmax rule. At the
    MQA shape the early key tiles go through the split dK/dV path (chunk
    partials, their reduce and the separate k-row epilogue); dgamma sums
    4096 x 32 + 4096 x 8 rows per batch element (Qwen3-like) and
    16384 x 17 rows (MQA)."""
    w = WORKLOADS[name]
    cpu = make_inputs(w)
    f, g = _gpu_to_host(*run_gpu(w, cpu))
    rf, rg = oracle_full(w, to_f64(cpu))
    compare_all(w, f, g, rf, rg)


def test_positions_past_two_to_the_21():
    """RoPE angles of positions >= 2^21 are formed in double, below in fp32 with
    a compensated product: rows on both sides of the switch against the oracle
    (norm + RoPE of single rows, attention rows over the whole prefix)."""
    S = (1 << 21) + 192
    w = Workload("positions_2p21_bf16", 1, S, 1, 1, 64, 1e6, 1e-6, "bf16")
    tol = TOL[w.dtype]
    cpu = make_inputs(w)
    f, g = run_gpu(w, cpu)
    x = to_f64(cpu)
    pos = np.array([0, 1, 5000, (1 << 21) - 1, 1 << 21, (1 << 21) + 1, S - 1])
    for name, src, gam, got in [("q_hat", "q", "gamma_q", f["q_hat"]),
                                ("k_hat", "k", "gamma_k", f["k_hat"])]:
        y, _ = oracle.rmsnorm_rows(x[src][0, pos, 0], x[gam], w.eps)
        ref = oracle.rope_rows(y, pos, w.theta)
        assert_close(name, got[0, 0, torch.as_tensor(pos, device=got.device)], ref, tol)
    rows = [(0, 0, int(t)) for t in (S - 1, (1 << 21) + 3, (1 << 21) - 2)]
    o, lse = oracle.attn_fwd_rows(x["q"], x["k"], x["v"], x["gamma_q"], x["gamma_k"], w.eps,
                                  w.theta, rows)
    dq = oracle.attn_dq_rows(x["q"], x["k"], x["v"], x["gamma_q"], x["gamma_k"], x["dout"],
                             w.eps, w.theta, rows)
    go = np.stack([as_f64(f["out"][0, t, 0]) for _, _, t in rows])
    glse = np.array([float(f["lse"][0, 0, t]) for _, _, t in rows])
    gdq = np.stack([as_f64(g["dq"][0, t, 0]) for _, _, t in rows])
    assert_close("out rows", go, o, tol)
    assert_close("lse rows", glse, lse, tol)
    assert_close("dq rows", gdq, dq, tol)
    krows = [(0, 0, S - 1), (0, 0, (1 << 21) + 10)]
    dk, dv = oracle.attn_dkdv_rows(x["q"], x["k"], x["v"], x["gamma_q"], x["gamma_k"], x["dout"],
                                   w.eps, w.theta, krows)
    gdk = np.stack([as_f64(g["dk"][0, j, 0]) for _, _, j in krows])
    gdv = np.stack([as_f64(g["dv"][0, j, 0]) for _, _, j in krows])
    assert_close("dk rows", gdk, dk, tol)
    assert_close("dv rows", gdv, dv, tol)
