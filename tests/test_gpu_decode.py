"""GPU parity of the decode step (one new token against a key/value cache).

The decode output of the token at position p is the training attention's row p
(Mint project report, 10.3 "KV cache": equal to the full-sequence attention at
that row), so the oracle's single-row attention over the raw q, k, v is the
reference; the cache row the call writes at p is checked against the oracle's
norm + RoPE of k, and v is copied exactly. Cache rows at and after p are filled
with garbage first, so that the call must write its own row and must not read
later ones. Bars as in the other parity tests.
"""
import numpy as np
import pytest
import torch

import oracle
from causal_gqa_attention_xt_gb300 import build as xbuild
from causal_gqa_attention_xt_gb300 import xt
from causal_gqa_attention_xt_gb300.inputs import Workload, make_inputs, to_f64

from parity_metrics import TOL, as_f64, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    xbuild.build()
    xt.lib()


CASES = [
    (Workload("dec_gqa_bf16", 3, 300, 8, 2, 64, 1e4, 1e-5, "bf16"), [0, 150, 299]),
    (Workload("dec_d128_bf16", 2, 1000, 32, 8, 128, 1e6, 1e-6, "bf16"), [999, 517]),
    # a group of 40 query heads: ten head chunks per kv head
    (Workload("dec_mqa_group40_bf16", 1, 5000, 40, 1, 128, 1e6, 1e-6, "bf16"), [4321]),
    (Workload("dec_f32", 2, 77, 4, 4, 32, 1e4, 1e-5, "f32"), [76, 5]),
    # head_dim 32 in bf16 (half of each lane group's 16-byte chunks lie past the row)
    (Workload("dec_d32_bf16", 2, 400, 6, 2, 32, 1e4, 1e-5, "bf16"), [399, 17]),
]


def _prefilled_caches(w, dev):
    """Caches of all S positions from the training forward (k_hat, v in the
    head-major cache layout)."""
    f = xt.xt_attn_fwd(dev["q"], dev["k"], dev["v"], dev["gamma_q"], dev["gamma_k"], w.eps,
                       w.theta)
    # clone: with one kv head the transposed v is already contiguous, and
    # .contiguous() alone would alias the input that the new rows come from
    return f["k_hat"].clone(), dev["v"].transpose(1, 2).contiguous().clone()


def _step(w, dev, kc, vc, pos):
    pos_t = torch.tensor(pos, dtype=torch.int32, device="cuda")
    qn = torch.stack([dev["q"][b, p] for b, p in enumerate(pos)]).contiguous()
    kn = torch.stack([dev["k"][b, p] for b, p in enumerate(pos)]).contiguous()
    vn = torch.stack([dev["v"][b, p] for b, p in enumerate(pos)]).contiguous()
    r = xt.xt_attn_decode(pos_t, qn, kn, vn, dev["gamma_q"], dev["gamma_k"], kc, vc, w.eps,
                          w.theta)
    assert xt.xt_attn_check() == xt.XT_OK
    return r


def _check(w, x, r, kc, vc, pos):
    tol = TOL[w.dtype]
    rows = [(b, h, p) for b, p in enumerate(pos) for h in range(w.H)]
    o, lse = oracle.attn_fwd_rows(x["q"], x["k"], x["v"], x["gamma_q"], x["gamma_k"], w.eps,
                                  w.theta, rows)
    go = np.stack([as_f64(r["out"][b, h]) for b, h, _ in rows])
    glse = np.array([float(r["lse"][b, h]) for b, h, _ in rows])
    assert_close("decode out", go, o, tol)
    assert_close("decode lse", glse, lse, tol)
    for b, p in enumerate(pos):
        y, _ = oracle.rmsnorm_rows(x["k"][b, p], x["gamma_k"], w.eps)
        ref = oracle.rope_rows(y, p, w.theta)
        assert_close("cached k_hat row", kc[b, :, p], ref, tol)
        assert torch.equal(vc[b, :, p].cpu(), torch.as_tensor(x["v"][b, p]).to(vc.dtype))


@pytest.mark.parametrize("w,pos", CASES, ids=lambda c: getattr(c, "name", None))
def test_decode_matches_oracle_rows(w, pos):
    cpu = make_inputs(w)
    dev = {k: v.cuda() for k, v in cpu.items()}
    x = to_f64(cpu)
    kc, vc = _prefilled_caches(w, dev)
    for b, p in enumerate(pos):   # the call writes row p itself and reads no later row
        kc[b, :, p:] = 7.0
        vc[b, :, p:] = -3.0
    r = _step(w, dev, kc, vc, pos)
    _check(w, x, r, kc, vc, pos)


def test_two_consecutive_steps_append_to_the_cache():
    w = Workload("dec_steps_bf16", 2, 260, 8, 2, 128, 1e6, 1e-6, "bf16")
    cpu = make_inputs(w)
    dev = {k: v.cuda() for k, v in cpu.items()}
    x = to_f64(cpu)
    kc, vc = _prefilled_caches(w, dev)
    pos = [200, 63]
    for b, p in enumerate(pos):
        kc[b, :, p:] = float("nan")   # never read: each step writes its row before attending
        vc[b, :, p:] = float("nan")
    _step(w, dev, kc, vc, pos)
    nxt = [p + 1 for p in pos]
    r = _step(w, dev, kc, vc, nxt)
    _check(w, x, r, kc, vc, nxt)


def test_out_of_range_position_is_reported_and_skipped():
    w = Workload("dec_bad_bf16", 2, 64, 4, 2, 64, 1e4, 1e-5, "bf16")
    cpu = make_inputs(w)
    dev = {k: v.cuda() for k, v in cpu.items()}
    kc = torch.zeros(2, 2, 64, 64, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    pos_t = torch.tensor([10, 64], dtype=torch.int32, device="cuda")
    qn = dev["q"][:, 0].contiguous()
    kn = dev["k"][:, 0].contiguous()
    vn = dev["v"][:, 0].contiguous()
    xt.xt_attn_decode(pos_t, qn, kn, vn, dev["gamma_q"], dev["gamma_k"], kc, vc, w.eps, w.theta)
    assert xt.xt_attn_check() == xt.XT_EINVAL
    assert xt.xt_attn_check() == xt.XT_OK          # the error word was cleared
    assert bool(torch.all(kc[1] == 0)) and bool(torch.all(vc[1] == 0))   # element 1 untouched
