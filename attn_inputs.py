"""Seeded synthetic inputs for the attention forward and split-KV decode.

This module is shared by the tests, the bench and the smoke check to feed both
the CUDA library and the CPU oracle the same bits.  It holds workload shapes
and random-number recipes only -- none of the attention arithmetic.

Recipe: one CPU ``torch.Generator`` seeded with the given seed draws Q, then K,
then V, each as fp32 samples that are rounded to bf16 with round-to-nearest-
even (``Tensor.to(torch.bfloat16)``).  ``normal`` draws use the stated standard
deviation; ``uniform`` draws are U(-1, 1).  Layout is [B, H, S, D] contiguous.

The five workloads are the page's Llama-family attention shapes made concrete
("A Thread-Register Decoupled GPU Execution Model for Efficient Tensor
Computation", Methodology, Tbl. III: context 4096, head dim 128; GQA/MQA head
sharing; FlashDecoding for decode).  No dataset or weights are involved.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Sk: int
    D: int
    causal: bool
    q_std: float = 1.0
    k_std: float = 1.0
    v_dist: str = "normal"  # "normal" (std 1) or "uniform" (U(-1,1))
    num_splits: int = 0     # > 0: split-KV decode workload
    seed: int = 1000

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def is_decode(self) -> bool:
        return self.num_splits > 0

    def flops(self) -> float:
        """Counted FLOPs: 4*B*Hq*Sq*Sk*D, halved when causal."""
        f = 4.0 * self.B * self.Hq * self.Sq * self.Sk * self.D
        return f / 2 if self.causal else f

    def algorithmic_bytes(self) -> int:
        """Minimum HBM traffic: read Q, K, V once (bf16); write O and LSE (fp32)."""
        q = self.B * self.Hq * self.Sq * self.D * 2
        kv = 2 * self.B * self.Hkv * self.Sk * self.D * 2
        o = self.B * self.Hq * self.Sq * self.D * 4
        lse = self.B * self.Hq * self.Sq * 4
        return q + kv + o + lse

    def describe(self) -> str:
        kind = "decode" if self.is_decode else ("causal" if self.causal else "non-causal")
        s = (f"{self.name}: B={self.B} Hq={self.Hq} Hkv={self.Hkv} Sq={self.Sq} "
             f"Sk={self.Sk} D={self.D} {kind}")
        if self.is_decode:
            s += f" splits={self.num_splits}"
        return s


# The five workloads, numbered 1..5; seed = 1000 + index.
WORKLOADS = {
    1: Workload("mha_b1_h2_s128_d64", 1, 2, 2, 128, 128, 64, False, seed=1001),
    2: Workload("mha_b4_h16_s1024_d64_causal", 4, 16, 16, 1024, 1024, 64, True,
                seed=1002),
    3: Workload("gqa_b2_hq32_hkv8_s8192_d128_causal", 2, 32, 8, 8192, 8192, 128, True,
                seed=1003),
    # "N(0,2)" read as variance 2 (std sqrt 2): the N(mu, sigma^2) convention.
    4: Workload("mha_b1_h16_s16384_d128_peaky", 1, 16, 16, 16384, 16384, 128, False,
                q_std=math.sqrt(2.0), k_std=math.sqrt(2.0), v_dist="uniform",
                seed=1004),
    5: Workload("gqa_decode_b64_hq32_hkv8_sk4096_d128_split8", 64, 32, 8, 1, 4096, 128,
                False, num_splits=8, seed=1005),
}


def make_qkv(B: int, Hq: int, Hkv: int, Sq: int, Sk: int, D: int, seed: int,
             q_std: float = 1.0, k_std: float = 1.0, v_dist: str = "normal"):
    """Q [B,Hq,Sq,D], K and V [B,Hkv,Sk,D] as bf16 CPU tensors, drawn in that order."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    q = torch.randn((B, Hq, Sq, D), generator=g, dtype=torch.float32)
    if q_std != 1.0:
        q.mul_(q_std)
    k = torch.randn((B, Hkv, Sk, D), generator=g, dtype=torch.float32)
    if k_std != 1.0:
        k.mul_(k_std)
    if v_dist == "normal":
        v = torch.randn((B, Hkv, Sk, D), generator=g, dtype=torch.float32)
    elif v_dist == "uniform":
        v = torch.rand((B, Hkv, Sk, D), generator=g, dtype=torch.float32).mul_(2.0).sub_(1.0)
    else:
        raise ValueError(f"unknown v_dist {v_dist!r}")
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)


def workload_inputs(w: Workload, seed: int | None = None):
    """Seeded bf16 (q, k, v) for a workload."""
    return make_qkv(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, w.seed if seed is None else seed,
                    q_std=w.q_std, k_std=w.k_std, v_dist=w.v_dist)


def sample_rows(B: int, H: int, S: int, n_random: int, seed: int) -> torch.Tensor:
    """Flat row ids (b*H + h)*S + i for a parity sample.

    Every (b, h) contributes its edge rows {0, 1, 127, 128, S-1} (those that
    exist); ``n_random`` further rows are drawn uniformly from a generator
    seeded with ``seed``.
    """
    fixed = sorted({i for i in (0, 1, 127, 128, S - 1) if 0 <= i < S})
    bh = torch.arange(B * H, dtype=torch.int64)
    edge = (bh[:, None] * S + torch.tensor(fixed, dtype=torch.int64)[None, :]).reshape(-1)
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    rnd = torch.randint(0, B * H * S, (n_random,), generator=g, dtype=torch.int64)
    return torch.unique(torch.cat([edge, rnd]))
