"""Seeded synthetic inputs: GGUF-layout weight bytes, activations, routing.

This module only draws random numbers and lays them out as bytes.  It holds
none of the product's arithmetic (no decoding, no dot products), so both the
CUDA path's tests and the CPU oracle can take their inputs from it.

Weight recipe (the block formats' fields drawn directly, since the pages
print no real weights):

* Q4_K (144-byte super-blocks of 256 weights): d and dmin uniform in
  [1e-4, 1e-3], stored as IEEE binary16; the 12 packed scale/min bytes and the
  128 quant bytes are uniform random bytes.  The 12-byte packing assigns each
  of its 96 bits to exactly one of the sixteen 6-bit fields, and each quant
  byte holds two 4-bit quants, so uniform bytes give scales/mins uniform on
  0..63 and quants uniform on 0..15, all independent.
* Q8_0 (34-byte blocks of 32 weights): d as above, quants uniform int8 on
  -127..127.
* Q5_K (176 bytes / 256): as Q4_K, with the 32 fifth-bit bytes uniform too.
* Q6_K (210 bytes / 256): the 128 low-bit and 64 high-bit bytes uniform
  (quants uniform on 0..63), sixteen int8 scales uniform on -128..127, d
  as above.
* IQ4_NL (18 bytes / 32): d as above, the 16 code bytes uniform.
* Activations: fp32 N(0, 1).  Prefill activations: N(0, 1) rounded to bf16.
* Router: logits N(0, 1) per (token, expert); p = softmax; the top_k largest
  p give the expert ids (distinct) and their p (not renormalised) the fp32
  routing weights.

All generators use numpy's PCG64 ``default_rng(seed)``.
"""
from __future__ import annotations

import numpy as np

Q8_0 = 8
Q4_K = 12
Q5_K = 13
Q6_K = 14
IQ4_NL = 20

Q4K_BLOCK_BYTES = 144
Q4K_BLOCK_WEIGHTS = 256
Q8_0_BLOCK_BYTES = 34
Q8_0_BLOCK_WEIGHTS = 32

# Llama-3.1-8B linear layers (N rows x K columns); q,k,v share one input,
# gate,up share one input.
LLAMA8B_SHAPES = (
    ("q", 4096, 4096),
    ("k", 1024, 4096),
    ("v", 1024, 4096),
    ("o", 4096, 4096),
    ("gate", 14336, 4096),
    ("up", 14336, 4096),
    ("down", 4096, 14336),
)
LLAMA8B_LAYERS = 32

# OLMoE-1B-7B expert FFN.
OLMOE_EXPERTS = 64
OLMOE_D_MODEL = 2048
OLMOE_D_FF = 1024
OLMOE_TOP_K = 8


# (block bytes, block weights) of the formats beyond Q4_K and Q8_0
_BLOCKS = {Q5_K: (176, 256), Q6_K: (210, 256), IQ4_NL: (18, 32)}


def row_bytes(fmt: int, K: int) -> int:
    if fmt in _BLOCKS:
        nbytes, nw = _BLOCKS[fmt]
        if K % nw:
            raise ValueError(f"format {fmt} needs K % {nw} == 0")
        return K // nw * nbytes
    if fmt == Q4_K:
        if K % Q4K_BLOCK_WEIGHTS:
            raise ValueError("Q4_K needs K % 256 == 0")
        return K // Q4K_BLOCK_WEIGHTS * Q4K_BLOCK_BYTES
    if fmt == Q8_0:
        if K % Q8_0_BLOCK_WEIGHTS:
            raise ValueError("Q8_0 needs K % 32 == 0")
        return K // Q8_0_BLOCK_WEIGHTS * Q8_0_BLOCK_BYTES
    raise ValueError(f"unknown format {fmt}")


def _fp16_scales(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.uniform(1e-4, 1e-3, size=shape).astype("<f2")


def q4k_matrix(N: int, K: int, seed: int) -> np.ndarray:
    """N x K weights as Q4_K bytes, shape [N, K/256*144] uint8."""
    nb = N * (K // Q4K_BLOCK_WEIGHTS)
    row_bytes(Q4_K, K)
    rng = np.random.default_rng(seed)
    raw = np.frombuffer(rng.bytes(nb * Q4K_BLOCK_BYTES), dtype=np.uint8)
    raw = raw.reshape(nb, Q4K_BLOCK_BYTES).copy()
    raw[:, 0:4] = _fp16_scales(rng, (nb, 2)).view(np.uint8).reshape(nb, 4)
    return raw.reshape(N, -1)


def q8_0_matrix(N: int, K: int, seed: int) -> np.ndarray:
    """N x K weights as Q8_0 bytes, shape [N, K/32*34] uint8."""
    nb = N * (K // Q8_0_BLOCK_WEIGHTS)
    row_bytes(Q8_0, K)
    rng = np.random.default_rng(seed)
    out = np.empty((nb, Q8_0_BLOCK_BYTES), np.uint8)
    out[:, 0:2] = _fp16_scales(rng, nb).view(np.uint8).reshape(nb, 2)
    out[:, 2:] = rng.integers(-127, 128, size=(nb, 32), dtype=np.int8).view(np.uint8)
    return out.reshape(N, -1)


def _raw_blocks(fmt: int, N: int, K: int, rng: np.random.Generator) -> np.ndarray:
    nbytes, nw = _BLOCKS[fmt]
    nb = N * (K // nw)
    row_bytes(fmt, K)
    return np.frombuffer(rng.bytes(nb * nbytes), dtype=np.uint8).reshape(nb, nbytes).copy()


def q5k_matrix(N: int, K: int, seed: int) -> np.ndarray:
    """N x K weights as Q5_K bytes, shape [N, K/256*176] uint8."""
    rng = np.random.default_rng(seed)
    raw = _raw_blocks(Q5_K, N, K, rng)
    raw[:, 0:4] = _fp16_scales(rng, (raw.shape[0], 2)).view(np.uint8).reshape(-1, 4)
    return raw.reshape(N, -1)


def q6k_matrix(N: int, K: int, seed: int) -> np.ndarray:
    """N x K weights as Q6_K bytes, shape [N, K/256*210] uint8 (the int8
    scales are uniform bytes)."""
    rng = np.random.default_rng(seed)
    raw = _raw_blocks(Q6_K, N, K, rng)
    raw[:, 208:210] = _fp16_scales(rng, raw.shape[0]).view(np.uint8).reshape(-1, 2)
    return raw.reshape(N, -1)


def iq4nl_matrix(N: int, K: int, seed: int) -> np.ndarray:
    """N x K weights as IQ4_NL bytes, shape [N, K/32*18] uint8."""
    rng = np.random.default_rng(seed)
    raw = _raw_blocks(IQ4_NL, N, K, rng)
    raw[:, 0:2] = _fp16_scales(rng, raw.shape[0]).view(np.uint8).reshape(-1, 2)
    return raw.reshape(N, -1)


def matrix(fmt: int, N: int, K: int, seed: int) -> np.ndarray:
    if fmt == Q4_K:
        return q4k_matrix(N, K, seed)
    if fmt == Q8_0:
        return q8_0_matrix(N, K, seed)
    return {Q5_K: q5k_matrix, Q6_K: q6k_matrix, IQ4_NL: iq4nl_matrix}[fmt](N, K, seed)


def activations(M: int, K: int, seed: int) -> np.ndarray:
    """fp32 N(0,1) activations [M, K]."""
    return np.random.default_rng(seed).standard_normal((M, K), dtype=np.float32)


def activations_bf16(M: int, K: int, seed: int) -> np.ndarray:
    """N(0,1) activations rounded to bfloat16; returns the uint16 bit patterns."""
    import torch
    x = activations(M, K, seed)
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def router(T: int, n_experts: int, top_k: int, seed: int):
    """Expert ids [T, top_k] int32 (distinct per token, by descending p) and
    routing weights [T, top_k] fp32 from a softmax over N(0,1) logits."""
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((T, n_experts))
    p = np.exp(logits - logits.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    order = np.argsort(-p, axis=1, kind="stable")[:, :top_k]
    ids = order.astype(np.int32)
    r = np.take_along_axis(p, order, axis=1).astype(np.float32)
    return ids, r


def layer_seed(seed: int, layer: int, which: int) -> int:
    """Distinct seed for matrix `which` of layer `layer`."""
    return (seed * 1_000_003 + layer * 101 + which) & 0x7FFFFFFF
