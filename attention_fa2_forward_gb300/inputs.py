"""Seeded synthetic inputs shaped like the attention workloads.

This module draws random numbers and nothing else: it holds none of the
attention arithmetic, so both the CUDA path and the fp64 oracle can be fed
from it. Tensors are generated on the CPU with a seeded ``torch.Generator``
in fp32 (Q, then K, then V) and rounded to the target dtype (bf16 rounding is
round-to-nearest-even), so every consumer sees identical values.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    S: int
    H: int
    Hkv: int
    D: int
    dtype: str  # "bf16" or "f32"
    causal: bool
    window: int = -1  # -1: no sliding window
    q_std: float = 1.0
    k_std: float = 1.0
    v_dist: str = "normal"  # "normal": N(0,1); "uniform": U(-1, 1)
    seed: int = 1000

    @property
    def scale(self) -> float:
        return 1.0 / (self.D ** 0.5)

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def describe(self) -> str:
        mask = "causal" if self.causal else "none"
        if self.window > 0:
            mask += f"+window{self.window}"
        return (f"B{self.B} H{self.H} Hkv{self.Hkv} S{self.S} D{self.D} "
                f"{self.dtype} {mask}")


# The workloads: a tiny fp32 case the oracle finishes instantly, a short
# causal MHA case, a causal GQA case, a sliding-window GQA case and a
# long-context multi-query stress case with large logits.
WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", 1, 128, 2, 2, 64, "f32", False, seed=1000),
    "mha_s1024_d64": Workload("mha_s1024_d64", 4, 1024, 16, 16, 64, "bf16", True, seed=1001),
    "gqa_s4096_d128": Workload("gqa_s4096_d128", 2, 4096, 32, 8, 128, "bf16", True, seed=1002),
    "swa_s16384_w4096": Workload("swa_s16384_w4096", 1, 16384, 32, 8, 128, "bf16", True,
                                 window=4096, seed=1003),
    "mqa_s32768_stress": Workload("mqa_s32768_stress", 1, 32768, 16, 1, 128, "bf16", True,
                                  q_std=3.0, k_std=3.0, v_dist="uniform", seed=1004),
    # Other head dims: 96 (padded to the 128-column kernel), 256 (one-Q-tile kernel).
    "gqa_s4096_d96": Workload("gqa_s4096_d96", 2, 4096, 32, 8, 96, "bf16", True, seed=1005),
    "gqa_s4096_d256": Workload("gqa_s4096_d256", 2, 4096, 16, 8, 256, "bf16", True, seed=1006),
    # fp32 inputs on the tensor cores (three bf16 parts per value).
    "gqa_s4096_d128_f32": Workload("gqa_s4096_d128_f32", 2, 4096, 32, 8, 128, "f32", True,
                                   seed=1007),
}


def make_qkv(B: int, S: int, H: int, Hkv: int, D: int, dtype: torch.dtype, seed: int,
             q_std: float = 1.0, k_std: float = 1.0, v_dist: str = "normal"):
    """Return CPU tensors q [B,S,H,D], k [B,S,Hkv,D], v [B,S,Hkv,D] in ``dtype``."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    q = torch.randn((B, S, H, D), generator=g, dtype=torch.float32)
    k = torch.randn((B, S, Hkv, D), generator=g, dtype=torch.float32)
    if v_dist == "normal":
        v = torch.randn((B, S, Hkv, D), generator=g, dtype=torch.float32)
    elif v_dist == "uniform":
        v = torch.rand((B, S, Hkv, D), generator=g, dtype=torch.float32) * 2.0 - 1.0
    else:
        raise ValueError(f"unknown v_dist {v_dist!r}")
    if q_std != 1.0:
        q = q * q_std
    if k_std != 1.0:
        k = k * k_std
    return q.to(dtype), k.to(dtype), v.to(dtype)


def workload_inputs(w: Workload, S: int | None = None, B: int | None = None):
    """Inputs of a workload (optionally with a different S or B, same recipe)."""
    return make_qkv(B or w.B, S or w.S, w.H, w.Hkv, w.D, w.torch_dtype, w.seed,
                    q_std=w.q_std, k_std=w.k_std, v_dist=w.v_dist)


# ---------------------------------------------------------------- KV cache

@dataclass(frozen=True)
class KvWorkload:
    """One attention step over a KV cache: B sequences whose keys and values
    fill the first lens[b] rows of [B, S_cache, Hkv, D] caches, with Sq new
    query tokens each (Sq = 1: one decoding step)."""
    name: str
    B: int
    Sq: int
    S_cache: int
    H: int
    Hkv: int
    D: int
    causal: bool = True
    window: int = -1
    ragged: bool = False  # lens drawn uniformly from [Sq, S_cache]; else all S_cache
    seed: int = 2000

    @property
    def scale(self) -> float:
        return 1.0 / (self.D ** 0.5)

    def describe(self) -> str:
        mask = "causal" if self.causal else "none"
        if self.window > 0:
            mask += f"+window{self.window}"
        lens = "ragged" if self.ragged else "full"
        return (f"B{self.B} Sq{self.Sq} S_cache{self.S_cache} ({lens}) H{self.H} "
                f"Hkv{self.Hkv} D{self.D} bf16 {mask}")


# Decoding steps: many short sequences, one long sequence (the key range is
# cut into splits), and a ragged batch of 4-token (speculative) steps.
KV_WORKLOADS = {
    "decode_b16_l8192_gqa_d128": KvWorkload("decode_b16_l8192_gqa_d128", 16, 1, 8192, 32, 8,
                                            128, seed=2001),
    "decode_b1_l131072_gqa_d128": KvWorkload("decode_b1_l131072_gqa_d128", 1, 1, 131072, 32, 8,
                                             128, seed=2002),
    "decode_b8_l32768_sq4_ragged": KvWorkload("decode_b8_l32768_sq4_ragged", 8, 4, 32768, 32, 8,
                                              128, ragged=True, seed=2003),
}


def make_kv_cache(B: int, Sq: int, S_cache: int, H: int, Hkv: int, D: int, seed: int,
                  ragged: bool = False, lens=None):
    """CPU bf16 tensors q [B, Sq, H, D], k_cache and v_cache [B, S_cache, Hkv, D]
    (every row random, including rows past the lengths) and the int32 lengths
    [B]: ``lens`` if given, else drawn uniformly from [Sq, S_cache] when
    ``ragged``, else S_cache."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    q = torch.randn((B, Sq, H, D), generator=g, dtype=torch.float32)
    k = torch.randn((B, S_cache, Hkv, D), generator=g, dtype=torch.float32)
    v = torch.randn((B, S_cache, Hkv, D), generator=g, dtype=torch.float32)
    if lens is None:
        if ragged:
            lens = torch.randint(min(Sq, S_cache), S_cache + 1, (B,), generator=g)
        else:
            lens = torch.full((B,), S_cache)
    lens = torch.as_tensor(lens, dtype=torch.int32).reshape(B)
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16), lens


def kv_workload_inputs(w: KvWorkload):
    return make_kv_cache(w.B, w.Sq, w.S_cache, w.H, w.Hkv, w.D, w.seed, ragged=w.ragged)


# ---------------------------------------------------------------- top-K

@dataclass(frozen=True)
class TopkWorkload:
    """Top-K selection over B rows of V fp32 scores (next-token logits)."""
    name: str
    B: int
    V: int
    K: int
    seed: int = 3000

    def describe(self) -> str:
        return f"B{self.B} V{self.V} K{self.K} fp32"


TOPK_WORKLOADS = {
    # A batch of next-token logits over a 128k vocabulary, top 50.
    "topk_b64_v131072_k50": TopkWorkload("topk_b64_v131072_k50", 64, 131072, 50, seed=3001),
    # 256 rows over a 256k vocabulary (268 MB of logits, more than L2), top 50.
    "topk_b256_v262144_k50": TopkWorkload("topk_b256_v262144_k50", 256, 262144, 50, seed=3002),
}


def make_scores(B: int, V: int, seed: int) -> torch.Tensor:
    """CPU fp32 scores [B, V] drawn N(0, 1) with a seeded generator."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return torch.randn((B, V), generator=g, dtype=torch.float32)
