"""Seeded synthetic inputs for the W4A16-g128 projection matmul and the dense
BF16 split-K GEMM.

This module only draws random numbers and encodes them in the library's input
format; it holds none of the matmul arithmetic.  Both the CPU oracle and the
CUDA path consume the exact bytes produced here.

Input format (the W4A16-g128 affine format, MLX-style affine quantization):
  * A       BF16 [M, Kred], row-major (returned as uint16 bit patterns)
  * Wq      uint32 [Nout, Kred/8], row-major; word j of row n holds
            q[n, 8j + i] in bits 4i..4i+3 (low nibble first), q in 0..15
  * scales  BF16 [Nout, Kred/128]; biases BF16 [Nout, Kred/128]
  * the weight the matmul uses is w[n, k] = scale[n, k/128] * q[n, k] + bias[n, k/128]

Value distributions follow the workloads the library is measured on:
A ~ N(0, 1); q uniform on 0..15; scale ~ U[0.005, 0.02]; bias = -8*scale +
N(0, 0.001).  Draw order is fixed (A, q, scale, bias noise) so a seed names
one problem.  Shapes are those of the Qwen3-4B projections in the tiny-llm
book, "Week 2 Day 7: Split-K Prefill" (Task 1 and Task 4 benchmark sweeps).
"""
from __future__ import annotations

import numpy as np
import torch

GROUP = 128  # quantization group length along the reduction axis

# Qwen3-4B projection shapes, Kred -> Nout (tiny-llm "Week 2 Day 7: Split-K
# Prefill", Task 4 sweep over q, k, v, o, gate, up, down).
PROJECTIONS = {
    "q": (2560, 4096),
    "k": (2560, 1024),
    "v": (2560, 1024),
    "o": (4096, 2560),
    "gate": (2560, 9728),
    "up": (2560, 9728),
    "down": (9728, 2560),
}
# Partial last 32-column output tile ("Task 4: Reduce and Verify").
RAGGED = (2560, 1000)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 array -> BF16 bit patterns (uint16), round to nearest even."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """BF16 bit patterns (uint16) -> float32 (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def pack_nibbles(q: np.ndarray) -> np.ndarray:
    """q uint8 [Nout, Kred] in 0..15 -> uint32 [Nout, Kred/8], low nibble first."""
    nout, kred = q.shape
    assert kred % 8 == 0
    shifts = (4 * np.arange(8, dtype=np.uint32))[None, None, :]
    words = (q.reshape(nout, kred // 8, 8).astype(np.uint32) << shifts)
    return np.bitwise_or.reduce(words, axis=2).astype(np.uint32)


def make_w4a16(M: int, Kred: int, Nout: int, seed: int = 0) -> dict:
    """One seeded W4A16-g128 problem.  Returns numpy arrays:
    A (uint16 bf16 bits [M,Kred]), Wq (uint32 [Nout,Kred/8]), scales, biases
    (uint16 bf16 bits [Nout,Kred/128]) and the unpacked q (uint8 [Nout,Kred])."""
    if Kred % GROUP:
        raise ValueError("Kred must be a multiple of 128")
    G = Kred // GROUP
    rng = np.random.default_rng(seed)
    a = rng.standard_normal((M, Kred), dtype=np.float32)
    q = rng.integers(0, 16, size=(Nout, Kred), dtype=np.uint8)
    scale = rng.uniform(0.005, 0.02, size=(Nout, G)).astype(np.float32)
    noise = rng.normal(0.0, 0.001, size=(Nout, G)).astype(np.float32)
    scales = f32_to_bf16_bits(scale)
    bias = -8.0 * bf16_bits_to_f32(scales) + noise
    return {
        "A": f32_to_bf16_bits(a),
        "Wq": pack_nibbles(q),
        "scales": scales,
        "biases": f32_to_bf16_bits(bias),
        "q": q,
        "M": M, "Kred": Kred, "Nout": Nout,
    }


def make_dense(M: int, N: int, K: int, seed: int = 0) -> dict:
    """Dense BF16 GEMM problem C = A @ W.T: A [M,K] and W [N,K] ~ N(0,1)."""
    rng = np.random.default_rng(seed)
    a = rng.standard_normal((M, K), dtype=np.float32)
    w = rng.standard_normal((N, K), dtype=np.float32)
    return {"A": f32_to_bf16_bits(a), "W": f32_to_bf16_bits(w), "M": M, "N": N, "K": K}


# Qwen3-4B attention: 32 query heads, 8 KV heads (grouped-query, 4 per KV
# head), head dim 128.
ATTENTION_HEADS = {"Hq": 32, "Hkv": 8, "D": 128}


def make_attention(B: int, Hq: int, Hkv: int, Lmax: int, D: int, seed: int = 0,
                   lens=None, lmin: int = 1) -> dict:
    """One seeded decode-attention problem: q [B,Hq,D], K and V [B,Hkv,Lmax,D]
    (BF16 bits, ~ N(0, 1)) and per-sequence lengths lens [B] (int32), drawn
    uniformly from [lmin, Lmax] unless given -- a mix of context lengths, as a
    decode batch of requests has.  Draw order: q, K, V, lens."""
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, Hq, D), dtype=np.float32)
    K = rng.standard_normal((B, Hkv, Lmax, D), dtype=np.float32)
    V = rng.standard_normal((B, Hkv, Lmax, D), dtype=np.float32)
    if lens is None:
        lens = rng.integers(lmin, Lmax + 1, size=B)
    return {"q": f32_to_bf16_bits(q), "K": f32_to_bf16_bits(K), "V": f32_to_bf16_bits(V),
            "lens": np.asarray(lens, dtype=np.int32), "B": B, "Hq": Hq, "Hkv": Hkv,
            "Lmax": Lmax, "D": D}
