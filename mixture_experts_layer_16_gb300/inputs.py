"""Seeded synthetic inputs for the fused MoE layer (forward + backward).

This module is the one piece shared by the CUDA path's callers and by the CPU
oracle.  It holds none of the layer's arithmetic: it only draws the workload
that the Prime Mega MoE pages measure (Qwen3-30B-A3B / Qwen3-235B-A22B layer
shapes, 128 experts, top-8, random routing; "TL;DR" and "How fast is Prime
Mega MoE?" sections) and rounds it to bf16 so that both sides consume the same
bits.

Recipe (one numpy PCG64 stream per config, drawn in this fixed order):
  1. routing logits  [T, k]  ~ N(0,1)  ->  topk_w = softmax over the k chosen (fp32)
  2. topk_idx        [T, k]  int32, k distinct experts per token:
       'uniform'   : a uniform random k-subset of the E experts;
       'zipf'      : sequential weighted draws without replacement (Gumbel-top-k)
                     with p(rank) ~ rank^-s over a seeded permutation of experts;
       'zipf_trunc': as 'zipf' but only the first `zipf_ranks` ranks get mass,
                     so E - zipf_ranks experts receive no token at all.
  3. x               [T, H]  ~ N(0,1)     -> bf16
  4. W_gate          [E,I,H] ~ N(0,0.02)  -> bf16
  5. W_up            [E,I,H] ~ N(0,0.02)  -> bf16
  6. W_down          [E,H,I] ~ N(0,0.02)  -> bf16
  7. dy              [T, H]  ~ N(0,1)     -> bf16
Every bf16 tensor is returned twice: as uint16 bit patterns (for the device)
and as float32 values that are exactly those bf16 numbers (for the oracle).
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import numpy as np


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    routing: str = "uniform"      # 'uniform' | 'zipf' | 'zipf_trunc'
    zipf_s: float = 1.2
    zipf_ranks: int = 0           # only for 'zipf_trunc'
    seed: int = 0
    prec: str = "bf16"            # 'bf16' | 'mxfp8' | 'fp8_bwd' | 'fp8_block'

    @property
    def R(self) -> int:
        return self.T * self.k

    def flops_fwd(self) -> float:
        return 6.0 * self.R * self.H * self.I

    def flops_bwd(self) -> float:
        return 12.0 * self.R * self.H * self.I

    def replace(self, **kw) -> "MoEConfig":
        return dataclasses.replace(self, **kw)


# The workloads: a tiny case, the two Qwen3 layer shapes, a skewed-routing
# 16,384-token case, and the MXFP8 16,384-token case.
CONFIGS: Dict[str, MoEConfig] = {
    "tiny": MoEConfig("tiny", T=64, H=128, I=64, E=8, k=2, routing="uniform", seed=1),
    "qwen3_30b_4k": MoEConfig("qwen3_30b_4k", T=4096, H=2048, I=768, E=128, k=8,
                              routing="uniform", seed=2),
    "qwen3_30b_16k_zipf": MoEConfig("qwen3_30b_16k_zipf", T=16384, H=2048, I=768, E=128,
                                    k=8, routing="zipf", zipf_s=1.2, seed=3),
    "qwen3_30b_16k_zipf_empty": MoEConfig("qwen3_30b_16k_zipf_empty", T=16384, H=2048,
                                          I=768, E=128, k=8, routing="zipf_trunc",
                                          zipf_s=1.2, zipf_ranks=120, seed=4),
    # a smaller skewed case (same layer, 8,192 tokens) for profiler captures
    "qwen3_30b_8k_zipf": MoEConfig("qwen3_30b_8k_zipf", T=8192, H=2048, I=768, E=128, k=8,
                                   routing="zipf", zipf_s=1.2, seed=7),
    "qwen3_235b_8k": MoEConfig("qwen3_235b_8k", T=8192, H=4096, I=1536, E=128, k=8,
                               routing="uniform", seed=5),
    "qwen3_30b_16k_mxfp8": MoEConfig("qwen3_30b_16k_mxfp8", T=16384, H=2048, I=768,
                                     E=128, k=8, routing="uniform", seed=6, prec="mxfp8"),
    # the same inputs with a BF16 forward and an MXFP8 backward
    "qwen3_30b_16k_fp8_bwd": MoEConfig("qwen3_30b_16k_fp8_bwd", T=16384, H=2048, I=768,
                                       E=128, k=8, routing="uniform", seed=6, prec="fp8_bwd"),
    # a smaller MXFP8 case (8,192 tokens, uniform routing) for profiler captures
    "qwen3_30b_8k_mxfp8": MoEConfig("qwen3_30b_8k_mxfp8", T=8192, H=2048, I=768, E=128, k=8,
                                    routing="uniform", seed=8, prec="mxfp8"),
    # and in blockwise FP8 (forward and backward)
    "qwen3_30b_16k_fp8block": MoEConfig("qwen3_30b_16k_fp8block", T=16384, H=2048, I=768,
                                        E=128, k=8, routing="uniform", seed=6,
                                        prec="fp8_block"),
}

BF16_ROUND_BIAS = np.uint32(0x7FFF)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even) -> uint16 bits."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + BF16_ROUND_BIAS + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact float32 value of bf16 bit patterns."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _routing(rng: np.random.Generator, cfg: MoEConfig) -> np.ndarray:
    T, E, k = cfg.T, cfg.E, cfg.k
    if k > E:
        raise ValueError("k must not exceed E")
    if cfg.routing == "uniform":
        keys = rng.random((T, E), dtype=np.float64)
        idx = np.argpartition(keys, k - 1, axis=1)[:, :k]
        # a uniform random k-subset, presented in a uniformly random order
        order = np.argsort(np.take_along_axis(keys, idx, axis=1), axis=1)
        idx = np.take_along_axis(idx, order, axis=1)
        return idx.astype(np.int32)
    if cfg.routing in ("zipf", "zipf_trunc"):
        ranks = np.arange(1, E + 1, dtype=np.float64)
        p = ranks ** (-cfg.zipf_s)
        if cfg.routing == "zipf_trunc":
            if not 0 < cfg.zipf_ranks <= E or cfg.zipf_ranks < k:
                raise ValueError("zipf_ranks must be in [k, E]")
            p[cfg.zipf_ranks:] = 0.0
        p /= p.sum()
        expert_of_rank = rng.permutation(E)
        with np.errstate(divide="ignore"):
            logp = np.log(p)
        g = rng.gumbel(size=(T, E)) + logp[None, :]
        top = np.argpartition(-g, k - 1, axis=1)[:, :k]
        order = np.argsort(-np.take_along_axis(g, top, axis=1), axis=1)
        top = np.take_along_axis(top, order, axis=1)   # draw order
        return expert_of_rank[top].astype(np.int32)
    raise ValueError(f"unknown routing {cfg.routing!r}")


def _normal_bf16(rng: np.random.Generator, shape, std: float):
    v = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        v *= np.float32(std)
    bits = bf16_bits(v)
    return bits, bf16_to_f32(bits)


def make_inputs(cfg: MoEConfig, with_dy: bool = True,
                weights: bool = True) -> Dict[str, np.ndarray]:
    """Draw one config's inputs.  Keys: topk_idx, topk_w, x, W_gate, W_up, W_down,
    dy (float32 values of bf16 numbers) and the same names + '_bits' (uint16)."""
    rng = np.random.Generator(np.random.PCG64(cfg.seed))
    out: Dict[str, np.ndarray] = {}
    logits = rng.standard_normal(size=(cfg.T, cfg.k))
    ex = np.exp(logits - logits.max(axis=1, keepdims=True))
    out["topk_w"] = (ex / ex.sum(axis=1, keepdims=True)).astype(np.float32)
    out["topk_idx"] = _routing(rng, cfg)
    out["x_bits"], out["x"] = _normal_bf16(rng, (cfg.T, cfg.H), 1.0)
    if weights:
        for name, shape in (("W_gate", (cfg.E, cfg.I, cfg.H)),
                            ("W_up", (cfg.E, cfg.I, cfg.H)),
                            ("W_down", (cfg.E, cfg.H, cfg.I))):
            out[name + "_bits"], out[name] = _normal_bf16(rng, shape, 0.02)
    if with_dy:
        if not weights:
            # keep the stream order fixed: skip the weight draws
            for shape in ((cfg.E, cfg.I, cfg.H), (cfg.E, cfg.I, cfg.H), (cfg.E, cfg.H, cfg.I)):
                rng.standard_normal(size=shape, dtype=np.float32)
        out["dy_bits"], out["dy"] = _normal_bf16(rng, (cfg.T, cfg.H), 1.0)
    return out


def custom_inputs(T: int, H: int, I: int, E: int, k: int, seed: int = 0,
                  routing: str = "uniform", idx: Optional[np.ndarray] = None,
                  **kw) -> Dict[str, np.ndarray]:
    """Inputs for an ad-hoc shape (edge-case tests).  `idx` overrides the routing."""
    cfg = MoEConfig("custom", T=T, H=H, I=I, E=E, k=k, routing=routing, seed=seed, **kw)
    d = make_inputs(cfg)
    if idx is not None:
        d["topk_idx"] = np.ascontiguousarray(idx, dtype=np.int32)
    return d


def router_weights(E: int, H: int, seed: int = 0) -> Dict[str, np.ndarray]:
    """W_router [E, H] ~ N(0, 0.02), rounded to bf16 (bits and exact values); its own
    stream, so the layer's inputs do not change."""
    rng = np.random.default_rng(np.random.PCG64(1000003 + seed))
    bits = bf16_bits(rng.standard_normal((E, H)).astype(np.float32) * np.float32(0.02))
    return dict(W_router_bits=bits, W_router=bf16_to_f32(bits).astype(np.float64))
