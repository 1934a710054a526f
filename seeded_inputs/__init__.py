"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the CPU oracle.

This module holds no arithmetic of the method itself: it only draws seeded
normal variates, rounds them to the storage type (bf16 round-to-nearest-even,
or fp32), and names the five workloads' shapes.  Both sides of every parity
check take their inputs from here; nothing here imports either side.

Workloads (the shapes follow the tensor-parallel MLP and MoE layers of
"TileLink: Generating Efficient Compute-Communication Overlapping Kernels using
Tile-Centric Primitives", Table 4 (MLP-2 / MLP-5 rows), and "Triton-distributed:
Programming Overlapping Kernels on Distributed AI Systems with the Triton
Compiler", Table 4 (AG+MoE rows with hidden 2048 / ffn 1408)):

  ag_tiny   AG+GEMM,  W=2, A_r 128x256,  B 256x256,   N(0,1)/sqrt(256)
  ag_70b    AG+GEMM,  W=8, A_r 1024x8192, B 8192x3584, N(0,1)/sqrt(8192)
  rs_70b    GEMM+RS,  W=8, A_p 8192x3584, B_p 3584x8192, N(0,1)/sqrt(28672)
  mlp2_8b   MLP2,     W=4, X 4096x4096 N(0,1); W1_r 4096x3584, W2_r 3584x4096 N(0,0.02^2)
  moe_64e   MoE,      T=4096, H=2048, E=64, F=1408, top-2; X N(0,1); logits N(0,1) fp32;
                      Wg, Wu (E,H,F) and Wd (E,F,H) N(0,0.02^2)
  attn_16k  AG KV + self-attention, W=8, 32 heads, head dim 128, sequence 16k (2048 per rank):
                      Q [32, 2048, 128], K_r and V_r [32, 2048, 128] per rank, all N(0,1)
                      ("TileLink ...", Table 4, Attn-1 at 16k)

Each tensor is drawn from its own stream, seed*1000 + tensor_index, with numpy's
PCG64 generator (standard normal, float32), scaled by the standard deviation in
float32, then rounded to bf16 (RNE) where the tensor is bf16.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "WORKLOADS", "Workload", "normal_f32", "normal_bf16", "bf16_bits_to_f32",
    "bf16_bits_to_f64", "f32_to_bf16_bits", "make_inputs",
]


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round-to-nearest-even); return the 16-bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float64 (exact)."""
    return bf16_bits_to_f32(b).astype(np.float64)


def normal_f32(stream: int, shape, std: float) -> np.ndarray:
    """float32 N(0, std^2) draws from PCG64(stream)."""
    g = np.random.Generator(np.random.PCG64(stream))
    out = g.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        out *= np.float32(std)
    return out


def normal_bf16(stream: int, shape, std: float) -> np.ndarray:
    """bf16 (as uint16 bit patterns) N(0, std^2) draws from PCG64(stream)."""
    return f32_to_bf16_bits(normal_f32(stream, shape, std))


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str                 # "ag_gemm" | "gemm_rs" | "mlp2" | "moe"
    seed: int
    dims: dict = field(default_factory=dict)


WORKLOADS = {
    "ag_tiny": Workload("ag_tiny", "ag_gemm", 1, dict(W=2, m_per_rank=128, n=256, k=256)),
    "ag_70b": Workload("ag_70b", "ag_gemm", 2, dict(W=8, m_per_rank=1024, n=3584, k=8192)),
    "rs_70b": Workload("rs_70b", "gemm_rs", 3, dict(W=8, m=8192, n=8192, k_r=3584)),
    "mlp2_8b": Workload("mlp2_8b", "mlp2", 4, dict(W=4, tokens=4096, hidden=4096, f_r=3584)),
    "moe_64e": Workload("moe_64e", "moe", 5, dict(T=4096, H=2048, E=64, F=1408, topk=2)),
    "attn_16k": Workload("attn_16k", "ag_attn", 6, dict(W=8, heads=32, l_r=2048, d=128)),
}


def make_inputs(kind: str, seed: int, **d) -> dict:
    """Draw every input tensor of one workload instance.

    bf16 tensors are returned as uint16 bit-pattern arrays; fp32 tensors as float32.
    Shapes:
      ag_gemm: a_shards [W] (m_per_rank, k); b (k, n)
      gemm_rs: a [W] (m, k_r); b [W] (k_r, n)
      mlp2:    x_shards [W] (tokens/W, hidden); w1 [W] (hidden, f_r); w2 [W] (f_r, hidden)
      moe:     x (T, H); logits (T, E) fp32; w_gate, w_up (E, H, F); w_down (E, F, H)
      ag_attn: q (heads, l_r, d); k_shards, v_shards [W] (heads, l_r, d)
      reduce_scatter: partials [W] (m, n) fp32, N(0, 1)
    """
    base = seed * 1000
    if kind == "ag_gemm":
        W, mr, n, k = d["W"], d["m_per_rank"], d["n"], d["k"]
        s = 1.0 / math.sqrt(k)
        a = [normal_bf16(base + r, (mr, k), s) for r in range(W)]
        b = normal_bf16(base + 100, (k, n), s)
        return dict(a_shards=a, b=b)
    if kind == "gemm_rs":
        W, m, n, kr = d["W"], d["m"], d["n"], d["k_r"]
        s = 1.0 / math.sqrt(W * kr)
        a = [normal_bf16(base + p, (m, kr), s) for p in range(W)]
        b = [normal_bf16(base + 100 + p, (kr, n), s) for p in range(W)]
        return dict(a=a, b=b)
    if kind == "mlp2":
        W, T, h, fr = d["W"], d["tokens"], d["hidden"], d["f_r"]
        x = [normal_bf16(base + r, (T // W, h), 1.0) for r in range(W)]
        w1 = [normal_bf16(base + 100 + r, (h, fr), 0.02) for r in range(W)]
        w2 = [normal_bf16(base + 200 + r, (fr, h), 0.02) for r in range(W)]
        return dict(x_shards=x, w1=w1, w2=w2)
    if kind == "moe":
        T, H, E, F = d["T"], d["H"], d["E"], d["F"]
        return dict(
            x=normal_bf16(base + 0, (T, H), 1.0),
            logits=normal_f32(base + 1, (T, E), 1.0),
            w_gate=normal_bf16(base + 2, (E, H, F), 0.02),
            w_up=normal_bf16(base + 3, (E, H, F), 0.02),
            w_down=normal_bf16(base + 4, (E, F, H), 0.02),
        )
    if kind == "reduce_scatter":
        W, m, n = d["W"], d["m"], d["n"]
        return dict(partials=[normal_f32(base + p, (m, n), 1.0) for p in range(W)])
    if kind == "ag_attn":
        W, Hh, L, hd = d["W"], d["heads"], d["l_r"], d["d"]
        return dict(
            q=normal_bf16(base + 0, (Hh, L, hd), 1.0),
            k_shards=[normal_bf16(base + 100 + r, (Hh, L, hd), 1.0) for r in range(W)],
            v_shards=[normal_bf16(base + 200 + r, (Hh, L, hd), 1.0) for r in range(W)],
        )
    raise ValueError(f"unknown workload kind {kind!r}")


def workload_inputs(name: str, **overrides) -> dict:
    w = WORKLOADS[name]
    dims = dict(w.dims)
    dims.update(overrides)
    return make_inputs(w.kind, w.seed, **dims)
