"""Seeded synthetic inputs shared by the tests, the bench and the smoke run.

This module holds none of the method's arithmetic: it only draws Q, K, V.
Shapes and distributions follow the long-sequence video-DiT workloads the
kvi8r pages describe (head dim 128, packed non-causal sequences): Q, K, V are
N(0, 1) in fp32 rounded to bf16, laid out [heads, seq, 128].  The "outlier"
variant multiplies 4 fixed channels of K by 20 before rounding, the kind of
outlier channels the Hadamard rotation is there to spread.

Seeds: Q uses ``seed``, K ``seed + 1``, V ``seed + 2``; the outlier channels
are the first four of a permutation of range(128) drawn with seed 3.
"""
from __future__ import annotations

import torch

HEAD_DIM = 128
OUTLIER_COUNT = 4
OUTLIER_GAIN = 20.0
OUTLIER_SEED = 3


def outlier_channels(d: int = HEAD_DIM) -> list[int]:
    g = torch.Generator().manual_seed(OUTLIER_SEED)
    return sorted(torch.randperm(d, generator=g)[:OUTLIER_COUNT].tolist())


def normal_f32(shape, seed: int, device="cpu") -> torch.Tensor:
    g = torch.Generator(device=device).manual_seed(int(seed))
    return torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)


def normal_bf16(shape, seed: int, device="cpu") -> torch.Tensor:
    return normal_f32(shape, seed, device).to(torch.bfloat16)


def make_k(heads: int, seq: int, seed: int, k_outliers: bool, device="cpu") -> torch.Tensor:
    k = normal_f32((heads, seq, HEAD_DIM), seed, device)
    if k_outliers:
        k[..., outlier_channels()] *= OUTLIER_GAIN
    return k.to(torch.bfloat16)


def make_qkv(heads: int, seq: int, seed: int = 0, k_outliers: bool = False,
             device="cpu", q_seq: int | None = None):
    """(Q, K, V) bf16 tensors [heads, q_seq or seq, 128] / [heads, seq, 128]."""
    q = normal_bf16((heads, seq if q_seq is None else q_seq, HEAD_DIM), seed, device)
    k = make_k(heads, seq, seed + 1, k_outliers, device)
    v = normal_bf16((heads, seq, HEAD_DIM), seed + 2, device)
    return q, k, v


# Named workloads: (heads, seq, k_outliers, q_chunk, kv_block).
WORKLOADS = {
    "tiny_1x1024": dict(heads=1, seq=1024, k_outliers=False, q_chunk=256, kv_block=512),
    "h8_l16384": dict(heads=8, seq=16384, k_outliers=False, q_chunk=4096, kv_block=8192),
    "h24_l32768_outlier": dict(heads=24, seq=32768, k_outliers=True, q_chunk=16384, kv_block=16384),
    "h32_l217088_outlier": dict(heads=32, seq=217088, k_outliers=True, q_chunk=16384, kv_block=16384),
    # the full-size sequence on 4 heads: small enough for counter captures,
    # with the same per-head store and launch pattern
    "h4_l217088_outlier": dict(heads=4, seq=217088, k_outliers=True, q_chunk=16384, kv_block=16384),
    "h32_l65536_sweep": dict(heads=32, seq=65536, k_outliers=False, q_chunk=16384, kv_block=16384),
}
