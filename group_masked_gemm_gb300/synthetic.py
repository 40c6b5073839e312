"""Seeded synthetic inputs for the group-masked FFN / projection workloads.

This module only draws random numbers and rounds them to bf16; it holds none
of the method's arithmetic, so both the CUDA path and the CPU oracle can be
fed from it.  Everything is numpy (``default_rng(seed)``), drawn in a fixed
order so that a workload is a pure function of its parameters:

    1. X            ~ N(0, 1)                       [T, D]
    2. weights      ~ N(0, 0.02), stored [out, in] (nn.Linear layout)
    3. the mask's own draws (keep-rates, then one uniform per (t, g)),
       mask[t, g] = u[t, g] < keep[t, g]

Shapes and statistics follow the workloads of the WIDE paper (Sec. 4.1:
Llama3.1-8B and Llama3.2-3B backbones; Sec. 4.4 / Fig. 9: attention sparsity
~66%, FFN ~28.5% at G = 128).  The paper's evaluation data and trained
routers are not used: masks are Bernoulli draws with the stated keep-rates.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

WEIGHT_STD = 0.02


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    rnd = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + rnd) >> 16).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32 (exact)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def _normal_bf16(rng, shape, std=1.0):
    x = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return bf16_bits(x)


def _bernoulli(rng, keep, shape):
    u = rng.random(shape)
    return (u < keep).astype(np.uint8)


def _beta_rescaled(rng, n, target):
    """Beta(2,2) draws rescaled to the requested mean and clipped to [0, 1]."""
    p = rng.beta(2.0, 2.0, size=n)
    return np.clip(p * (target / p.mean()), 0.0, 1.0)


def correlated_keep(r_t: np.ndarray, k: float) -> np.ndarray:
    """Per-token keep probability with mean k, monotone in a shared r_t in [0,1].

    With r_t ~ Beta(2,2) (mean 1/2): k * r_t / 0.5 for k <= 1/2, else
    1 - (1 - k)(1 - r_t) / 0.5.  Both stay in [0, 1] and have mean exactly k,
    and tokens with a large r_t keep more groups in every module.
    """
    r_t = np.asarray(r_t, np.float64)
    if k <= 0.5:
        return k * r_t / 0.5
    return 1.0 - (1.0 - k) * (1.0 - r_t) / 0.5


@dataclass
class FFNInputs:
    """One masked-FFN workload; bf16 tensors are uint16 bit patterns."""
    name: str
    T: int
    D: int
    F: int
    G: int
    seed: int
    X: np.ndarray
    Wg: np.ndarray
    Wu: np.ndarray
    Wd: np.ndarray
    mask: np.ndarray
    meta: dict = field(default_factory=dict)

    @property
    def n_groups(self) -> int:
        return self.F // self.G

    def active_flops(self) -> float:
        """6 * D * G * sum(M): gate, up and down MACs of the active groups."""
        return 6.0 * self.D * self.G * float(self.mask.sum(dtype=np.int64))

    def dense_flops(self) -> float:
        return 6.0 * self.D * self.F * self.T


def ffn_inputs(T, D, F, G, seed, keep=0.5, mask_kind="iid", name="custom"):
    """Draw X, Wg, Wu, Wd and a mask [T, F/G].

    mask_kind: "iid" (Bernoulli(keep) per entry), "per_group" (group keep-rate
    ~ Beta(2,2) rescaled to mean ``keep``), "ones", "zeros".
    """
    if F % G:
        raise ValueError("F must be a multiple of G")
    rng = np.random.default_rng(seed)
    X = _normal_bf16(rng, (T, D))
    Wg = _normal_bf16(rng, (F, D), WEIGHT_STD)
    Wu = _normal_bf16(rng, (F, D), WEIGHT_STD)
    Wd = _normal_bf16(rng, (D, F), WEIGHT_STD)
    ng = F // G
    meta = {"mask_kind": mask_kind, "keep": keep}
    if mask_kind == "iid":
        mask = _bernoulli(rng, keep, (T, ng))
    elif mask_kind == "per_group":
        p_g = _beta_rescaled(rng, ng, keep)
        meta["group_keep"] = p_g
        mask = _bernoulli(rng, p_g[None, :], (T, ng))
    elif mask_kind == "ones":
        mask = np.ones((T, ng), np.uint8)
    elif mask_kind == "zeros":
        mask = np.zeros((T, ng), np.uint8)
    else:
        raise ValueError(mask_kind)
    return FFNInputs(name, T, D, F, G, seed, X, Wg, Wu, Wd, mask, meta)


def with_mask(inp: FFNInputs, mask: np.ndarray, name: str | None = None) -> FFNInputs:
    """Same tensors, another mask (e.g. the all-ones dense-path run)."""
    mask = np.ascontiguousarray(mask, np.uint8)
    assert mask.shape == (inp.T, inp.n_groups)
    return FFNInputs(name or inp.name, inp.T, inp.D, inp.F, inp.G, inp.seed,
                     inp.X, inp.Wg, inp.Wu, inp.Wd, mask, dict(inp.meta))


# --- the named workloads -----------------------------------------------------

def tiny_ffn() -> FFNInputs:
    """T=64, d_model=256, d_ffn=1024, G=128 (8 groups), Bernoulli(0.5), seed 0."""
    return ffn_inputs(64, 256, 1024, 128, 0, 0.5, "iid", "tiny_ffn_T64_D256_F1024_G128")


def llama3b_prefill() -> FFNInputs:
    """Llama3.2-3B FFN prefill: T=4096, D=3072, F=8192, G=128, per-group
    keep ~ Beta(2,2) rescaled to mean 0.5, seed 1."""
    return ffn_inputs(4096, 3072, 8192, 128, 1, 0.5, "per_group",
                      "llama3.2-3b_ffn_prefill_T4096_G128_per_group_p0.5")


def llama8b_prefill(keep=0.5) -> FFNInputs:
    """Llama3.1-8B FFN prefill: T=16384, D=4096, F=14336, G=128, i.i.d.
    Bernoulli(keep), seed 2 (keep 0.75 / 0.5 / 0.25 = 25 / 50 / 75% sparsity)."""
    return ffn_inputs(16384, 4096, 14336, 128, 2, keep, "iid",
                      f"llama3.1-8b_ffn_prefill_T16384_G128_keep{keep:g}")


def llama8b_decode(T, G) -> FFNInputs:
    """Llama3.1-8B FFN decode: T in {1,4,16}, G in {64,128,256,512}, p=0.5, seed 3."""
    return ffn_inputs(T, 4096, 14336, G, 3, 0.5, "iid",
                      f"llama3.1-8b_ffn_decode_T{T}_G{G}")


@dataclass
class LayerInputs:
    """Prunable Llama3.1-8B layer: q_proj / o_proj over 8 GQA head groups of
    512 columns and the FFN over 112 groups of 128."""
    T: int
    X: np.ndarray        # [T, 4096]
    Wq: np.ndarray       # [4096, 4096]
    Wo: np.ndarray       # [4096, 4096]
    A: np.ndarray        # [T, 4096] stand-in for the attention output
    ffn: FFNInputs
    mask_attn: np.ndarray  # [T, 8]
    G_attn: int = 512


def llama8b_layer(T=16384, seed=4, attn_keep=0.34, ffn_keep=0.72) -> LayerInputs:
    """Full prunable layer, seed 4: per-token r_t ~ Beta(2,2) shared by both
    modules, attention keep 0.34 (66% sparsity), FFN keep 0.72 (28%)."""
    D, F, G, Ga = 4096, 14336, 128, 512
    rng = np.random.default_rng(seed)
    X = _normal_bf16(rng, (T, D))
    Wq = _normal_bf16(rng, (D, D), WEIGHT_STD)
    Wo = _normal_bf16(rng, (D, D), WEIGHT_STD)
    A = _normal_bf16(rng, (T, D))
    Wg = _normal_bf16(rng, (F, D), WEIGHT_STD)
    Wu = _normal_bf16(rng, (F, D), WEIGHT_STD)
    Wd = _normal_bf16(rng, (D, F), WEIGHT_STD)
    r_t = rng.beta(2.0, 2.0, size=T)
    ka = correlated_keep(r_t, attn_keep)
    kf = correlated_keep(r_t, ffn_keep)
    mask_attn = _bernoulli(rng, ka[:, None], (T, D // Ga))
    mask_ffn = _bernoulli(rng, kf[:, None], (T, F // G))
    ffn = FFNInputs(f"llama3.1-8b_layer_ffn_T{T}", T, D, F, G, seed, X, Wg, Wu,
                    Wd, mask_ffn, {"mask_kind": "correlated", "keep": ffn_keep})
    return LayerInputs(T, X, Wq, Wo, A, ffn, mask_attn, Ga)


def random_mask(T, n_groups, keep, seed) -> np.ndarray:
    """A stand-alone Bernoulli mask (for reorder-only cases)."""
    rng = np.random.default_rng(seed)
    return _bernoulli(rng, keep, (T, n_groups))


def sample_rows(T: int, n: int, seed: int) -> np.ndarray:
    """A sorted seeded subset of token rows that always contains 0 and T-1."""
    rng = np.random.default_rng(seed)
    n = min(n, T)
    pick = rng.choice(T, size=n, replace=False)
    pick[0] = 0
    if n > 1:
        pick[1] = T - 1
    return np.unique(pick).astype(np.int32)
