"""The backward entry point that allocates nothing (xt_attn_bwd_noalloc).

It is for callers that cannot allocate device memory themselves; its scratch
is the library's fixed 16 MiB device array. Both calls run the same
deterministic kernels on the same inputs, so the no-allocation result must be
bitwise equal to the regular workspace backward's. It is checked through the
C ABI on two calls in a row; between them a no-allocation call of a different
shape and dtype leaves the shared array holding differently laid-out data, so
a read of a scratch byte that the second call did not write first would show.
For both dtypes, plus the refusal of a problem that needs more scratch than
the array holds. This file sorts last so that a run stopping at the first
failure has run every other test.
"""
import ctypes

import pytest
import torch

from causal_gqa_attention_xt_gb300 import build as xbuild
from causal_gqa_attention_xt_gb300 import xt
from causal_gqa_attention_xt_gb300.inputs import Workload, make_inputs


pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    xbuild.build()
    xt.lib()


NOALLOC = [
    Workload("noalloc_gqa_bf16", 2, 300, 8, 2, 64, 1e4, 1e-5, "bf16", seed=11),
    Workload("noalloc_mqa_f32", 1, 129, 4, 1, 32, 1e6, 1e-6, "f32", seed=12),
    # the bench's Qwen3-like shape: the bf16 kernels finish dq and dk themselves, so its
    # scratch (RoPE table, Dlt, dgamma partials) fits the static array
    Workload("noalloc_qwen3_like_bf16", 4, 4096, 32, 8, 128, 1e6, 1e-6, "bf16", seed=13),
]
# a call of another shape and dtype, made between the two checked calls
OTHER = {"bf16": Workload("noalloc_other_f32", 2, 77, 6, 3, 64, 1e4, 1e-5, "f32", seed=14),
         "f32": Workload("noalloc_other_bf16", 1, 500, 4, 2, 128, 1e6, 1e-6, "bf16", seed=15)}


def _dtype_code(w):
    return xt.XT_BF16 if w.dtype == "bf16" else xt.XT_F32


def _noalloc(w, d, f):
    return xt.xt_attn_bwd_noalloc(d["q"], d["k"], d["v"], d["gamma_q"], d["gamma_k"], f,
                                  d["dout"], w.eps, w.theta)


@pytest.mark.parametrize("w", NOALLOC, ids=lambda w: w.name)
def test_noalloc_backward_matches_workspace_backward(w):
    d = {k_: v_.cuda() for k_, v_ in make_inputs(w).items()}
    assert xt.xt_attn_workspace_bytes(w.B, w.S, w.H, w.G, w.D, _dtype_code(w), True) <= 16 << 20
    f = xt.xt_attn_fwd(d["q"], d["k"], d["v"], d["gamma_q"], d["gamma_k"], w.eps, w.theta)
    ref = xt.xt_attn_bwd(d["q"], d["k"], d["v"], d["gamma_q"], d["gamma_k"], f, d["dout"],
                         w.eps, w.theta)
    assert xt.xt_attn_check() == xt.XT_OK
    ref = {k_: v_.clone() for k_, v_ in ref.items()}
    wo = OTHER[w.dtype]
    do_ = {k_: v_.cuda() for k_, v_ in make_inputs(wo).items()}
    fo = xt.xt_attn_fwd(do_["q"], do_["k"], do_["v"], do_["gamma_q"], do_["gamma_k"], wo.eps,
                        wo.theta)
    for call in range(2):
        if call == 1:
            _noalloc(wo, do_, fo)   # the shared array now holds the other problem's scratch
            assert xt.xt_attn_check() == xt.XT_OK
        got = _noalloc(w, d, f)
        assert xt.xt_attn_check() == xt.XT_OK
        for name in ("dq", "dk", "dv", "dgamma_q", "dgamma_k"):
            assert torch.equal(got[name], ref[name]), (call, name)


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
