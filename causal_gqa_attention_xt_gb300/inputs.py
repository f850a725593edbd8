"""Seeded synthetic inputs for the attention core.

This module holds no arithmetic of the method: it only draws random numbers.
Both the CUDA path (through the tests and the benchmark) and the CPU oracle
receive the same arrays from here.

Recipe (one CPU ``torch.Generator`` per workload, ``manual_seed(seed)``):
q [B,S,H,D], k [B,S,G,D], v [B,S,G,D] and dout [B,S,H,D] ~ N(0, 1) in fp32,
drawn in that order, then gamma_q and gamma_k = 1 + 0.1 * N(0, 1) [D], fp32.
For bf16 workloads q, k, v and dout are rounded to bf16 (round to nearest
even, ``Tensor.to``); the gammas stay fp32.

Packed batches (samples of different lengths flattened into one row
dimension) draw q [T,H,D], k, v [T,G,D], dout [T,H,D] and the gammas the same
way, T the sum of the lengths. The benchmark's length mix draws each sample's
length uniformly from [lo, hi] with its own generator (seed + 1) until the
total is reached; the last sample takes the remainder.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    """One attention-core problem: shapes, RoPE theta, RMSNorm eps, dtype."""
    name: str
    B: int
    S: int
    H: int          # query heads
    G: int          # key/value heads (H % G == 0)
    D: int          # head dim
    theta: float
    eps: float
    dtype: str      # "f32" or "bf16"
    seed: int = 0
    note: str = field(default="", compare=False)

    @property
    def group(self) -> int:
        return self.H // self.G

    @property
    def fwd_flops(self) -> float:
        """Causal forward FLOPs, counted as 2 * B * H * S^2 * D."""
        return 2.0 * self.B * self.H * self.S * self.S * self.D

    @property
    def bwd_flops(self) -> float:
        """Backward FLOPs, counted as 2.5 x the forward."""
        return 2.5 * self.fwd_flops

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


# The workloads the attention core is specified on (xtrain's tiny MHA shape,
# a GQA bring-up shape, the dim768 training shape, a Qwen3-like shape and a
# long-context MQA shape).
WORKLOADS = {
    "tiny_mha_f32": Workload("tiny_mha_f32", 1, 16, 2, 2, 16, 1e4, 1e-5, "f32"),
    "gqa_bf16": Workload("gqa_bf16", 4, 256, 8, 2, 64, 1e4, 1e-5, "bf16"),
    "dim768_mha_bf16": Workload("dim768_mha_bf16", 32, 1024, 12, 12, 64, 1e4, 1e-5, "bf16"),
    "dim768_gqa_bf16": Workload("dim768_gqa_bf16", 32, 1024, 12, 4, 64, 1e4, 1e-5, "bf16"),
    "qwen3_like_bf16": Workload("qwen3_like_bf16", 4, 4096, 32, 8, 128, 1e6, 1e-6, "bf16"),
    "mqa_long_bf16": Workload("mqa_long_bf16", 1, 16384, 16, 1, 128, 1e6, 1e-6, "bf16"),
    # the pages' own dim768 run: 24 heads x head_dim 32 at seq 256, per-rank batch 32
    "dim768_hd32_bf16": Workload("dim768_hd32_bf16", 32, 256, 24, 24, 32, 1e4, 1e-5, "bf16"),
    # decode: 32 sequences, each the next token against a full 4096-row cache
    "qwen3_like_decode_bf16": Workload("qwen3_like_decode_bf16", 32, 4096, 32, 8, 128, 1e6, 1e-6,
                                       "bf16"),
}


def torch_dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def make_inputs(w: Workload, gamma_scale: float = 0.1, gamma_offset: float = 1.0):
    """Draw the seeded CPU tensors of workload ``w``.

    Returns a dict of CPU tensors: q, k, v, dout in the workload dtype and
    gamma_q, gamma_k in fp32.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    q = torch.randn((w.B, w.S, w.H, w.D), generator=g, dtype=torch.float32)
    k = torch.randn((w.B, w.S, w.G, w.D), generator=g, dtype=torch.float32)
    v = torch.randn((w.B, w.S, w.G, w.D), generator=g, dtype=torch.float32)
    dout = torch.randn((w.B, w.S, w.H, w.D), generator=g, dtype=torch.float32)
    gamma_q = gamma_offset + gamma_scale * torch.randn((w.D,), generator=g, dtype=torch.float32)
    gamma_k = gamma_offset + gamma_scale * torch.randn((w.D,), generator=g, dtype=torch.float32)
    dt = torch_dtype(w.dtype)
    return dict(q=q.to(dt), k=k.to(dt), v=v.to(dt), dout=dout.to(dt),
                gamma_q=gamma_q, gamma_k=gamma_k)


def to_f64(inputs: dict) -> dict:
    """The same tensors widened exactly to float64 numpy arrays."""
    return {k: v.to(torch.float64).numpy() for k, v in inputs.items()}


@dataclass(frozen=True)
class PackedWorkload:
    """Samples of the given lengths packed into one [T] row dimension."""
    name: str
    lens: tuple
    H: int
    G: int
    D: int
    theta: float
    eps: float
    dtype: str
    seed: int = 0

    @property
    def T(self) -> int:
        return int(sum(self.lens))

    @property
    def max_len(self) -> int:
        return int(max(self.lens))

    @property
    def cu(self) -> list:
        out = [0]
        for n in self.lens:
            out.append(out[-1] + int(n))
        return out

    @property
    def fwd_flops(self) -> float:
        """Causal forward FLOPs, counted per sample as 2 * H * len^2 * D."""
        return float(sum(2.0 * self.H * n * n * self.D for n in self.lens))

    @property
    def bwd_flops(self) -> float:
        return 2.5 * self.fwd_flops


def length_mix(total: int, lo: int, hi: int, seed: int) -> tuple:
    """Sample lengths drawn uniformly from [lo, hi] until they sum to total."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + 1)
    lens = []
    left = total
    while left > 0:
        n = int(torch.randint(lo, hi + 1, (1,), generator=g).item())
        n = min(n, left)
        lens.append(n)
        left -= n
    return tuple(lens)


PACKED_WORKLOADS = {
    # 16384 rows (the Qwen3-like batch's rows) as samples of 256..4096 rows
    "qwen3_like_varlen_bf16": PackedWorkload("qwen3_like_varlen_bf16",
                                             length_mix(16384, 256, 4096, 0), 32, 8, 128,
                                             1e6, 1e-6, "bf16"),
}


def make_packed_inputs(w: PackedWorkload, gamma_scale: float = 0.1, gamma_offset: float = 1.0):
    """CPU tensors of a packed batch: q, k, v, dout (workload dtype), gammas
    (fp32) and cu_seqlens (int32 [nseq + 1])."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    T = w.T
    q = torch.randn((T, w.H, w.D), generator=g, dtype=torch.float32)
    k = torch.randn((T, w.G, w.D), generator=g, dtype=torch.float32)
    v = torch.randn((T, w.G, w.D), generator=g, dtype=torch.float32)
    dout = torch.randn((T, w.H, w.D), generator=g, dtype=torch.float32)
    gamma_q = gamma_offset + gamma_scale * torch.randn((w.D,), generator=g, dtype=torch.float32)
    gamma_k = gamma_offset + gamma_scale * torch.randn((w.D,), generator=g, dtype=torch.float32)
    dt = torch_dtype(w.dtype)
    return dict(q=q.to(dt), k=k.to(dt), v=v.to(dt), dout=dout.to(dt), gamma_q=gamma_q,
                gamma_k=gamma_k, cu_seqlens=torch.tensor(w.cu, dtype=torch.int32))
