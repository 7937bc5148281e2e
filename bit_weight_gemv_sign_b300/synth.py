"""Seeded synthetic inputs and workload shapes.

This module holds random-number draws and shape tables only: no packing,
no product, no patch arithmetic.  It is the one piece of code shared by the
CUDA path's tests/benchmark and the CPU oracle's checks, so both sides see
byte-identical inputs.

Input recipe (the pages' real Bonsai weights are not available, so seeded
synthetic tensors with the same format stand in for them):
  * sign bits  : i.i.d. uniform bytes, i.e. i.i.d. Bernoulli(0.5) bits;
  * scales     : |N(0, 0.02)| drawn in fp32, rounded to fp16 (RNE), plus an
                 optional offset (1e-3 for the tiny case);
  * activations: N(0, 1) drawn in fp32, rounded to bf16 (RNE);
  * ternary    : codes -1/0/+1 with 0 at probability 1/3 (a BitNet-like
                 share of zeros), or two independent uniform sign planes.
Every matrix has its own Philox stream keyed by ``seed``; activations use a
separate key space so that a matrix and its input never share a stream.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

X_SEED_OFFSET = 1 << 20


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(int(seed)))


def sign_bits(N: int, K: int, gen: np.random.Generator) -> np.ndarray:
    """Packed sign bits, [N, K/8] uint8, every bit Bernoulli(0.5)."""
    return gen.integers(0, 256, size=(N, K // 8), dtype=np.uint8)


def group_scales(N: int, K: int, gen: np.random.Generator, offset: float = 0.0,
                 sigma: float = 0.02) -> np.ndarray:
    """fp16 bit patterns [N, K/128] of |N(0, sigma)| + offset."""
    s = np.abs(gen.standard_normal(size=(N, K // 128), dtype=np.float32)) * np.float32(sigma)
    if offset:
        s = s + np.float32(offset)
    return s.astype(np.float16).view(np.uint16)


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 array -> bf16 bit patterns (round to nearest even, via torch)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def activations(B: int, K: int, gen: np.random.Generator) -> np.ndarray:
    """bf16 bit patterns [B, K] of N(0, 1)."""
    return to_bf16_bits(gen.standard_normal(size=(B, K), dtype=np.float32))


def matrix(N: int, K: int, seed: int, scale_offset: float = 0.0):
    """(bits, scales) of one synthetic packed matrix."""
    g = rng(seed)
    bits = sign_bits(N, K, g)
    scales = group_scales(N, K, g, offset=scale_offset)
    return bits, scales


def ternary_codes(N: int, K: int, gen: np.random.Generator, p_zero: float = 1.0 / 3.0) -> np.ndarray:
    """Ternary codes [N, K] int8: 0 with probability ``p_zero``, otherwise -1
    or +1 with equal probability."""
    p = (1.0 - p_zero) / 2.0
    return gen.choice(np.array([-1, 0, 1], dtype=np.int8), size=(N, K), p=[p, p_zero, p])


def ternary_matrix(N: int, K: int, seed: int):
    """(a, b, scales) of one synthetic ternary matrix given directly as two
    independent uniform sign planes (every pair of bits is a valid code, so
    this draws 0 with probability 1/2 and -1, +1 with 1/4 each)."""
    g = rng(seed)
    a = sign_bits(N, K, g)
    b = sign_bits(N, K, g)
    scales = group_scales(N, K, g)
    return a, b, scales


def x_for(B: int, K: int, seed: int) -> np.ndarray:
    return activations(B, K, rng(seed + X_SEED_OFFSET))


def fp_weights(N: int, K: int, seed: int, sigma: float = 0.02) -> np.ndarray:
    """fp32 weights N(0, sigma) [N, K] (input of the packing step)."""
    return rng(seed).standard_normal(size=(N, K), dtype=np.float32) * np.float32(sigma)


def distinct_rows(N: int, count: int, seed: int) -> np.ndarray:
    """``count`` distinct row indices in [0, N), int32."""
    return rng(seed).choice(N, size=count, replace=False).astype(np.int32)


# ---- workload shapes ----------------------------------------------------

@dataclass(frozen=True)
class Mat:
    name: str
    N: int   # outputs (rows)
    K: int   # inputs (columns, multiple of 128)
    swiglu: bool = False   # rows are interleaved (gate, up) pairs; N / 2 outputs

    @property
    def out(self) -> int:
        return self.N // 2 if self.swiglu else self.N


TINY = Mat("tiny", 256, 1024)

PROJ_8B = [Mat("up_gate", 12288, 4096), Mat("down", 4096, 12288),
           Mat("q_o", 4096, 4096), Mat("k_v", 1024, 4096)]

LM_HEAD_8B = Mat("lm_head", 151936, 4096)


def sweep_8b() -> list:
    """36 layers x {q, k, v, o, gate, up, down} + the 1-bit LM head, decode
    order (253 matrices; the embedding is a lookup and is not swept)."""
    out = []
    for layer in range(36):
        out += [Mat(f"L{layer}.q", 4096, 4096), Mat(f"L{layer}.k", 1024, 4096),
                Mat(f"L{layer}.v", 1024, 4096), Mat(f"L{layer}.o", 4096, 4096),
                Mat(f"L{layer}.gate", 12288, 4096), Mat(f"L{layer}.up", 12288, 4096),
                Mat(f"L{layer}.down", 4096, 12288)]
    out.append(Mat("lm_head", 151936, 4096))
    return out


def sweep_8b_fused_mlp() -> list:
    """The 8B-class sweep with each layer's gate and up projections stored as
    one interleaved 24576 x 4096 matrix whose product ends in the SwiGLU
    activation (36 x {q, k, v, o, gate_up, down} + the LM head, 217 matrices,
    the same weights and bytes as ``sweep_8b``)."""
    out = []
    for layer in range(36):
        out += [Mat(f"L{layer}.q", 4096, 4096), Mat(f"L{layer}.k", 1024, 4096),
                Mat(f"L{layer}.v", 1024, 4096), Mat(f"L{layer}.o", 4096, 4096),
                Mat(f"L{layer}.gate_up", 24576, 4096, swiglu=True),
                Mat(f"L{layer}.down", 4096, 12288)]
    out.append(Mat("lm_head", 151936, 4096))
    return out


def decode_chain_8b_fused() -> list:
    """The 8B-class decode step as a chain of fused matrices: per layer q|k|v
    as one 6144 x 4096 matrix (they share x), o, gate|up interleaved 24576 x
    4096 ending in SwiGLU, and down, whose input is that h; then the LM head
    (145 matrices, the same weights and bytes as ``sweep_8b``)."""
    out = []
    for layer in range(36):
        out += [Mat(f"L{layer}.qkv", 6144, 4096), Mat(f"L{layer}.o", 4096, 4096),
                Mat(f"L{layer}.gate_up", 24576, 4096, swiglu=True), Mat(f"L{layer}.down", 4096, 12288)]
    out.append(Mat("lm_head", 151936, 4096))
    return out


PROJ_NAMES_27B = ["q", "k", "v", "o", "gate", "up", "down"]


def sweep_27b() -> list:
    """64 layers x {q 5120x5120, k 1024x5120, v 1024x5120, o 5120x5120,
    gate 17408x5120, up 17408x5120, down 5120x17408} (448 matrices)."""
    out = []
    for layer in range(64):
        out += [Mat(f"L{layer}.q", 5120, 5120), Mat(f"L{layer}.k", 1024, 5120),
                Mat(f"L{layer}.v", 1024, 5120), Mat(f"L{layer}.o", 5120, 5120),
                Mat(f"L{layer}.gate", 17408, 5120), Mat(f"L{layer}.up", 17408, 5120),
                Mat(f"L{layer}.down", 5120, 17408)]
    return out


def patch_entries_27b(count: int = 100, seed: int = 0):
    """``count`` (layer, projection, row) entries over the 27B-class sweep,
    drawn with the given seed (distinct triples)."""
    mats = sweep_27b()
    g = rng(seed)
    seen = set()
    out = []
    while len(out) < count:
        layer = int(g.integers(0, 64))
        proj = int(g.integers(0, 7))
        m = mats[layer * 7 + proj]
        row = int(g.integers(0, m.N))
        key = (layer, proj, row)
        if key not in seen:
            seen.add(key)
            out.append(key)
    return out
