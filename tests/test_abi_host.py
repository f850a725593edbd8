"""Host-side checks of the C ABI that need no GPU: the library loads, it
exports every function include/xt_attn.h declares, and argument validation
rejects bad calls before any CUDA work (faults are injected on the host)."""
import ctypes
import os
import re

import pytest

from causal_gqa_attention_xt_gb300 import build as xbuild
from causal_gqa_attention_xt_gb300 import xt

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    xbuild.build()
    return xt.lib()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names.update(re.findall(r"\b(xt_\w+)\s*\(", src))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("xt_attn_fwd", "xt_attn_bwd", "xt_attn_workspace_bytes", "xt_status_str",
              "xt_attn_check"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for n in declared_functions():
        assert hasattr(L, n), n


def test_status_strings(L):
    for code in range(6):
        assert xt.xt_status_str(code) not in ("", "unknown status")
    assert xt.xt_status_str(99) == "unknown status"


def _fwd(L, B=1, S=16, H=2, G=2, D=16, eps=1e-5, theta=1e4, dtype=0, ptr=16):
    p = ctypes.c_void_p(ptr)
    return L.xt_attn_fwd(B, S, H, G, D, eps, theta, p, p, p, p, p, dtype, p, p, p, p, p, p,
                         None, 0, None)


@pytest.mark.parametrize("kw,code", [
    (dict(B=0), xt.XT_EINVAL), (dict(S=-1), xt.XT_EINVAL), (dict(H=3, G=2), xt.XT_EINVAL),
    (dict(D=15), xt.XT_EINVAL), (dict(dtype=7), xt.XT_EINVAL), (dict(eps=-1.0), xt.XT_EINVAL),
    (dict(theta=0.0), xt.XT_EINVAL), (dict(eps=float("nan")), xt.XT_EINVAL),
    (dict(ptr=0), xt.XT_EINVAL), (dict(ptr=8), xt.XT_EINVAL),
    (dict(B=1 << 16, S=1 << 16, H=1, G=1, D=16), xt.XT_EINVAL),
    (dict(D=48, dtype=1), xt.XT_EUNSUPPORTED), (dict(D=136), xt.XT_EUNSUPPORTED),
    (dict(D=12), xt.XT_EUNSUPPORTED),
])
def test_forward_validation_rejects_before_launch(L, kw, code):
    assert _fwd(L, **kw) == code


def test_forward_needs_its_workspace(L):
    p = ctypes.c_void_p(16)
    need = xt.xt_attn_workspace_bytes(1, 16, 2, 2, 16, 0, False)
    args = [1, 16, 2, 2, 16, 1e-5, 1e4] + [p] * 5 + [0] + [p] * 6
    assert L.xt_attn_fwd(*args, None, need, None) == xt.XT_EWORKSPACE
    assert L.xt_attn_fwd(*args, p, need - 1, None) == xt.XT_EWORKSPACE
    assert L.xt_attn_fwd(*args, ctypes.c_void_p(24), need, None) == xt.XT_EWORKSPACE


def test_backward_validation_and_workspace(L):
    p = ctypes.c_void_p(16)
    need = xt.xt_attn_workspace_bytes(1, 16, 2, 2, 16, 0, True)
    assert need > 0 and need % 256 == 0
    fneed = xt.xt_attn_workspace_bytes(1, 16, 2, 2, 16, 0, False)
    assert 16 * 8 * 8 <= fneed <= need   # the [S][D/2] (cos, sin) table; the backward holds it too
    assert xt.xt_attn_workspace_bytes(1, 16, 3, 2, 16, 0, True) == 0
    args = [1, 16, 2, 2, 16, 1e-5, 1e4] + [p] * 5 + [0] + [p] * 7 + [p] * 5
    assert L.xt_attn_bwd(*args, p, need - 1, None) == xt.XT_EWORKSPACE
    assert L.xt_attn_bwd(*args, None, need, None) == xt.XT_EWORKSPACE
    bad = list(args)
    bad[2] = 3
    assert L.xt_attn_bwd(*bad, p, need, None) == xt.XT_EINVAL


def test_timing_hooks_without_launches(L):
    xt.xt_timing_reset()
    assert xt.xt_timing_query() == {}
    assert L.xt_kernel_count() >= 5


def test_head_count_limit(L):
    # n_heads + n_kv_heads above 8192 is refused before any launch
    assert _fwd(L, H=8192, G=1) == xt.XT_EUNSUPPORTED


def test_decode_validation_and_workspace(L):
    p = ctypes.c_void_p(16)
    need = xt.xt_attn_decode_workspace_bytes(2, 64, 4, 2, 16, 0)
    assert need > 0 and need % 256 == 0
    assert xt.xt_attn_decode_workspace_bytes(2, 64, 3, 2, 16, 0) == 0
    assert xt.xt_attn_decode_workspace_bytes(2, 64, 4, 2, 48, 1) == 0   # bf16 wants D 32 / 64 / 128
    args = [2, 64, 4, 2, 16, 1e-5, 1e4]
    tail = [p] * 5 + [0] + [p] * 4
    assert L.xt_attn_decode(*args, p, *tail, p, need - 1, None) == xt.XT_EWORKSPACE
    assert L.xt_attn_decode(*args, None, *tail, p, need, None) == xt.XT_EINVAL      # no positions
    assert L.xt_attn_decode(*args, ctypes.c_void_p(18), *tail, p, need, None) == xt.XT_EINVAL
    bad = list(args)
    bad[2] = 3
    assert L.xt_attn_decode(*bad, p, *tail, p, need, None) == xt.XT_EINVAL


def test_fp32_grid_limit(L):
    # the fp32 path runs one grid row per (batch element, head): at most 65535
    assert _fwd(L, B=65536 // 2, S=1, H=2, G=2, D=16) == xt.XT_EUNSUPPORTED
    assert _fwd(L, B=65536 // 2, S=1, H=2, G=2, D=64, dtype=1, ptr=0) == xt.XT_EINVAL   # bf16: not limited


def _fwd_varlen(L, total=64, nseq=3, max_seqlen=32, H=4, G=2, D=64, dtype=1, cu=16, ptr=16,
                ws=None, wbytes=0):
    p = ctypes.c_void_p(ptr)
    return L.xt_attn_fwd_varlen(total, nseq, max_seqlen, H, G, D, 1e-5, 1e4, ctypes.c_void_p(cu),
                                p, p, p, p, p, dtype, p, p, p, p, p, p, ws, wbytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(nseq=0), xt.XT_EINVAL), (dict(max_seqlen=0), xt.XT_EINVAL),
    (dict(max_seqlen=65), xt.XT_EINVAL), (dict(cu=0), xt.XT_EINVAL), (dict(cu=18), xt.XT_EINVAL),
    (dict(total=0), xt.XT_EINVAL), (dict(H=3), xt.XT_EINVAL), (dict(ptr=8), xt.XT_EINVAL),
    (dict(D=48), xt.XT_EUNSUPPORTED),
    (dict(nseq=20000, D=16, dtype=0), xt.XT_EUNSUPPORTED),   # fp32 grid limit: nseq * H
])
def test_varlen_validation_rejects_before_launch(L, kw, code):
    assert _fwd_varlen(L, **kw) == code


def test_bf16_backward_workspace_follows_the_dkdv_split(L):
    # bf16: the tensor-core kernels finish dq and dk themselves, so no fp32 dQhat is kept and
    # fp32 dKhat only where the dK/dV work of long key tiles is split (long MQA)
    B, S, H, G, D = 4, 4096, 32, 8, 128
    bf = xt.xt_attn_workspace_bytes(B, S, H, G, D, 1, True)
    f32 = xt.xt_attn_workspace_bytes(B, S, H, G, D, 0, True)
    dkhat = B * G * S * D * 4
    assert 0 < bf < dkhat
    assert f32 > B * H * S * D * 4 + dkhat
    # table + Dlt + one dgamma_q row per (b, head, query tile) + one dgamma_k row per (b, kv head, key tile)
    assert bf >= S * D // 2 * 8 + B * H * S * 4 + (B * H * 32 + B * G * 32) * D * 4
    mqa = xt.xt_attn_workspace_bytes(1, 16384, 16, 1, D, 1, True)
    assert mqa > 1 * 1 * 16384 * D * 4   # fp32 dKhat for the reduce and the k-row epilogue


def test_varlen_workspace(L):
    fneed = xt.xt_attn_varlen_workspace_bytes(1000, 5, 300, 4, 2, 64, 1, False)
    bneed = xt.xt_attn_varlen_workspace_bytes(1000, 5, 300, 4, 2, 64, 1, True)
    assert fneed >= 1000 * 32 * 8 and bneed > fneed   # one (cos, sin) row per packed row
    assert xt.xt_attn_varlen_workspace_bytes(1000, 5, 1001, 4, 2, 64, 1, False) == 0
    assert xt.xt_attn_varlen_workspace_bytes(1000, 0, 300, 4, 2, 64, 1, True) == 0
    # the bf16 backward keeps a dgamma_q partial row per (sample, head, query tile)
    more = xt.xt_attn_varlen_workspace_bytes(1000, 9, 300, 4, 2, 64, 1, True)
    assert more >= bneed + 4 * 4 * 3 * 64 * 4 - 256
    assert _fwd_varlen(L, ws=ctypes.c_void_p(16), wbytes=100) == xt.XT_EWORKSPACE
    p = ctypes.c_void_p(16)
    need = xt.xt_attn_varlen_workspace_bytes(64, 3, 32, 4, 2, 64, 1, True)
    args = [64, 3, 32, 4, 2, 64, 1e-5, 1e4, p] + [p] * 5 + [1] + [p] * 7 + [p] * 5
    assert L.xt_attn_bwd_varlen(*args, p, need - 1, None) == xt.XT_EWORKSPACE
    bad = list(args)
    bad[2] = 0
    assert L.xt_attn_bwd_varlen(*bad, p, need, None) == xt.XT_EINVAL


def test_stall_injection_mask_validation(L):
    # the fault-injection hook of the timeout path takes kernel bits 1|2|4 only
    assert L.xt_test_inject_stall(8) == 1
    assert L.xt_test_inject_stall(-1) == 1
    assert L.xt_test_inject_stall(7) == 0
    assert L.xt_test_inject_stall(0) == 0
