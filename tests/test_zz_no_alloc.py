"""The backward entry point that allocates nothing (xt_attn_bwd_noalloc).

It is for callers that cannot allocate device memory themselves; its scratch
is the library's fixed 16 MiB device array. Checked through the C ABI against
the regular workspace backward on the same inputs, on two calls in a row (the
array keeps the previous call's contents), for both dtypes, plus the refusal
of a problem that needs more scratch than the array holds. This file sorts
last so that a run stopping at the first failure has run every other test.
"""
import ctypes

import pytest
import torch

from causal_gqa_attention_xt_gb300 import build as xbuild
from causal_gqa_attention_xt_gb300 import xt
from causal_gqa_attention_xt_gb300.inputs import Workload, make_inputs

from parity_metrics import TOL, max_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    xbuild.build()
    xt.lib()


@pytest.mark.parametrize("w", [
    Workload("noalloc_gqa_bf16", 2, 300, 8, 2, 64, 1e4, 1e-5, "bf16", seed=11),
    Workload("noalloc_mqa_f32", 1, 129, 4, 1, 32, 1e6, 1e-6, "f32", seed=12),
    # the bench's Qwen3-like shape: the bf16 kernels finish dq and dk themselves, so its
    # scratch (RoPE table, Dlt, dgamma partials) fits the static array
    Workload("noalloc_qwen3_like_bf16", 4, 4096, 32, 8, 128, 1e6, 1e-6, "bf16", seed=13),
], ids=lambda w: w.name)
def test_noalloc_backward_matches_workspace_backward(w):
    d = {k_: v_.cuda() for k_, v_ in make_inputs(w).items()}
    assert xt.xt_attn_workspace_bytes(w.B, w.S, w.H, w.G, w.D, w.dtype == "bf16" and 1 or 0,
                                      True) <= 16 << 20
    f = xt.xt_attn_fwd(d["q"], d["k"], d["v"], d["gamma_q"], d["gamma_k"], w.eps, w.theta)
    ref = xt.xt_attn_bwd(d["q"], d["k"], d["v"], d["gamma_q"], d["gamma_k"], f, d["dout"],
                         w.eps, w.theta)
    assert xt.xt_attn_check() == xt.XT_OK
    ref = {k_: v_.clone() for k_, v_ in ref.items()}
    for call in range(2):
        got = xt.xt_attn_bwd_noalloc(d["q"], d["k"], d["v"], d["gamma_q"], d["gamma_k"], f,
                                     d["dout"], w.eps, w.theta)
        assert xt.xt_attn_check() == xt.XT_OK
        for name in ("dq", "dk", "dv", "dgamma_q", "dgamma_k"):
            err = max_rel_err(got[name], ref[name])
            assert err <= TOL[w.dtype], (call, name, err)


def test_noalloc_refuses_problems_beyond_the_static_scratch():
    B, S, H, G, D = 64, 4096, 32, 8, 128
    assert xt.xt_attn_workspace_bytes(B, S, H, G, D, xt.XT_BF16, True) > 16 << 20
    # the size check comes before any launch, so one small aligned buffer stands in
    # for every tensor argument
    buf = torch.empty(64, device="cuda", dtype=torch.uint8)
    p = ctypes.c_void_p(buf.data_ptr())
    st = xt.lib().xt_attn_bwd_noalloc(B, S, H, G, D, 1e-6, 1e6, p, p, p, p, p, xt.XT_BF16,
                                      p, p, p, p, p, p, p, p, p, p, p, p, None)
    assert st == xt.XT_EWORKSPACE
