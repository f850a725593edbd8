"""The timeout path of the tensor-core kernels on the GPU, without a GPU fault.

Every barrier wait in those kernels is bounded; a wait that runs out raises the
library's device error word, and the CTA drains its own copies and MMAs, frees
its tensor memory and exits (Mint project report 9.7, error handling: a GPU
failure surfaces at a check point as an error, it is not swallowed). Here
xt_test_inject_stall makes the MMA thread of each CTA of one kernel wait on a
barrier that nothing arrives on, with a 20 ms limit: the call must still
return, xt_attn_check() must report XT_ETIMEOUT once (and then clear), and the
next normal call must be correct against the oracle.
"""
import time

import pytest
import torch

from causal_gqa_attention_xt_gb300 import build as xbuild
from causal_gqa_attention_xt_gb300 import xt
from causal_gqa_attention_xt_gb300.inputs import Workload, make_inputs, to_f64

from test_gpu_parity import compare_all, oracle_full, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    xbuild.build()
    xt.lib()
    yield
    xt.xt_test_inject_stall(0)


SMALL = Workload("timeout_gqa_bf16", 1, 300, 4, 2, 64, 1e4, 1e-5, "bf16", seed=9)
# one kv head for 8 query heads over 1000 rows: the dK/dV work is split into
# chunks (partials, their reduce and the separate k-row epilogue follow)
SPLIT = Workload("timeout_split_mqa_bf16", 1, 1000, 8, 1, 64, 1e4, 1e-5, "bf16", seed=10)


@pytest.mark.parametrize("mask,w", [(xt.STALL_FWD_TC, SMALL), (xt.STALL_DKDV_TC, SMALL),
                                    (xt.STALL_DQ_TC, SMALL), (xt.STALL_DKDV_TC, SPLIT),
                                    (xt.STALL_FWD_TC | xt.STALL_DKDV_TC | xt.STALL_DQ_TC, SMALL)],
                         ids=["fwd", "dkdv", "dq", "dkdv_split", "all"])
def test_stalled_kernel_reports_timeout_and_the_next_call_is_correct(mask, w):
    cpu = make_inputs(w)
    assert xt.xt_attn_check() == xt.XT_OK                 # nothing pending from earlier tests
    t0 = time.perf_counter()
    try:
        assert xt.xt_test_inject_stall(mask) == xt.XT_OK
        d = {k: v.cuda() for k, v in cpu.items()}
        f = xt.xt_attn_fwd(d["q"], d["k"], d["v"], d["gamma_q"], d["gamma_k"], w.eps, w.theta)
        xt.xt_attn_bwd(d["q"], d["k"], d["v"], d["gamma_q"], d["gamma_k"], f, d["dout"], w.eps,
                       w.theta)
        st = xt.xt_attn_check()
    finally:
        xt.xt_test_inject_stall(0)
    assert st == xt.XT_ETIMEOUT, xt.xt_status_str(st)
    assert time.perf_counter() - t0 < 30.0                # gave up, did not hang
    assert xt.xt_attn_check() == xt.XT_OK                 # the word was cleared
    f, g = run_gpu(w, cpu)                                # checks XT_OK itself
    rf, rg = oracle_full(w, to_f64(cpu))
    compare_all(w, f, g, rf, rg)

