"""GPU parity: the CUDA path through the C ABI against the CPU oracle, on the
same seeded inputs.

Bars: max relative error (max |g - r| / max |r|) <= 1e-4 for fp32 and 2e-2
for bf16 per output tensor, and the same argmax along every output row
(near-ties excepted). Small shapes are compared element by element on every
output; the full-size workloads are compared on exact sub-problems (one batch
element and one key/value group form an independent problem), on rows the
oracle computes one by one, and through sum rules that hold at any size.
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


def _sub_problem(x: dict, b: int, kvh: int, group: int):
    """Inputs of one (batch element, kv group): an independent problem."""
    hs = slice(kvh * group, (kvh + 1) * group)
    return dict(q=x["q"][b:b + 1, :, hs], k=x["k"][b:b + 1, :, kvh:kvh + 1],
                v=x["v"][b:b + 1, :, kvh:kvh + 1], dout=x["dout"][b:b + 1, :, hs],
                gamma_q=x["gamma_q"], gamma_k=x["gamma_k"])


def test_qwen3_like_full_size_sub_problem_and_rows():
    w = WORKLOADS["qwen3_like_bf16"]
    tol = TOL[w.dtype]
    cpu = make_inputs(w)
    f, g = run_gpu(w, cpu)
    x = to_f64(cpu)
    b, kvh = 3, 5
    sub = _sub_problem(x, b, kvh, w.group)
    ws = w.with_(B=1, H=w.group, G=1)
    rf, rg = oracle_full(ws, sub)
    hs = slice(kvh * w.group, (kvh + 1) * w.group)
    assert_close("out", f["out"][b:b + 1, :, hs], rf["out"], tol)
    assert_close("lse", f["lse"][b:b + 1, hs], rf["lse"], tol)
    assert_close("dq", g["dq"][b:b + 1, :, hs], rg["dq"], tol)
    assert_close("dk", g["dk"][b:b + 1, :, kvh:kvh + 1], rg["dk"], tol)
    assert_close("dv", g["dv"][b:b + 1, :, kvh:kvh + 1], rg["dv"], tol)
    # rows elsewhere, spread over batch, heads and tiles
    rng = np.random.default_rng(0)
    rows = [(int(rng.integers(w.B)), int(rng.integers(w.H)), int(t))
            for t in rng.integers(0, w.S, size=24)] + [(0, 0, 0), (1, 31, w.S - 1)]
    o, lse = oracle.attn_fwd_rows(x["q"], x["k"], x["v"], x["gamma_q"], x["gamma_k"], w.eps,
                                  w.theta, rows)
    dq = oracle.attn_dq_rows(x["q"], x["k"], x["v"], x["gamma_q"], x["gamma_k"], x["dout"],
                             w.eps, w.theta, rows)
    go = np.stack([as_f64(f["out"][bb, t, h]) for bb, h, t in rows])
    glse = np.array([float(f["lse"][bb, h, t]) for bb, h, t in rows])
    gdq = np.stack([as_f64(g["dq"][bb, t, h]) for bb, h, t in rows])
    assert max_rel_err(go, o) <= tol
    assert max_rel_err(glse, lse) <= tol
    assert max_rel_err(gdq, dq) <= tol
    krows = [(0, 0, w.S - 1), (2, 7, w.S - 130), (1, 3, w.S - 300)]
    dk, dv = oracle.attn_dkdv_rows(x["q"], x["k"], x["v"], x["gamma_q"], x["gamma_k"], x["dout"],
                                   w.eps, w.theta, krows)
    gdk = np.stack([as_f64(g["dk"][bb, j, gg]) for bb, gg, j in krows])
    gdv = np.stack([as_f64(g["dv"][bb, j, gg]) for bb, gg, j in krows])
    assert max_rel_err(gdk, dk) <= tol
    assert max_rel_err(gdv, dv) <= tol


def test_mqa_long_full_size_rows_and_sum_rule():
    w = WORKLOADS["mqa_long_bf16"]
    tol = TOL[w.dtype]
    cpu = make_inputs(w)
    f, g = run_gpu(w, cpu)
    x = to_f64(cpu)
    rng = np.random.default_rng(1)
    rows = [(0, int(rng.integers(w.H)), int(t)) for t in rng.integers(0, w.S, size=20)]
    rows += [(0, 0, 0), (0, 15, w.S - 1), (0, 7, 8191)]
    o, lse = oracle.attn_fwd_rows(x["q"], x["k"], x["v"], x["gamma_q"], x["gamma_k"], w.eps,
                                  w.theta, rows)
    dq = oracle.attn_dq_rows(x["q"], x["k"], x["v"], x["gamma_q"], x["gamma_k"], x["dout"],
                             w.eps, w.theta, rows)
    go = np.stack([as_f64(f["out"][0, t, h]) for _, h, t in rows])
    glse = np.array([float(f["lse"][0, h, t]) for _, h, t in rows])
    gdq = np.stack([as_f64(g["dq"][0, t, h]) for _, h, t in rows])
    assert max_rel_err(go, o) <= tol
    assert max_rel_err(glse, lse) <= tol
    assert max_rel_err(gdq, dq) <= tol
    krows = [(0, 0, w.S - 1), (0, 0, w.S - 60)]
    dk, dv = oracle.attn_dkdv_rows(x["q"], x["k"], x["v"], x["gamma_q"], x["gamma_k"], x["dout"],
                                   w.eps, w.theta, krows)
    gdk = np.stack([as_f64(g["dk"][0, j, 0]) for _, _, j in krows])
    gdv = np.stack([as_f64(g["dv"][0, j, 0]) for _, _, j in krows])
    assert max_rel_err(gdk, dk) <= tol
    assert max_rel_err(gdv, dv) <= tol
    # rows of P sum to one, so summed over positions dV equals the group's summed dO
    dv_total = as_f64(g["dv"])[0, :, 0].sum(0)
    do_total = x["dout"][0].sum((0, 1))
    assert max_rel_err(dv_total, do_total) <= tol


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
    assert max_rel_err(go, o) <= tol
    assert max_rel_err(glse, lse) <= tol
    assert max_rel_err(gdq, dq) <= tol
    krows = [(0, 0, S - 1), (0, 0, (1 << 21) + 10)]
    dk, dv = oracle.attn_dkdv_rows(x["q"], x["k"], x["v"], x["gamma_q"], x["gamma_k"], x["dout"],
                                   w.eps, w.theta, krows)
    gdk = np.stack([as_f64(g["dk"][0, j, 0]) for _, _, j in krows])
    gdv = np.stack([as_f64(g["dv"][0, j, 0]) for _, _, j in krows])
    assert max_rel_err(gdk, dk) <= tol
    assert max_rel_err(gdv, dv) <= tol
