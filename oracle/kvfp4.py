"""fp64 CPU oracle for the kvfp4 K/V store (NVFP4: e2m1 values with one e4m3
scale per 16) and the attention over it.

THIS IS TEST INFRASTRUCTURE, under the same rule as ``oracle.kvi8r``: only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` may import it; the
CUDA path never calls it.

What is computed, and where it is stated
----------------------------------------
[P1] "H3 Streamed Blocks (exact low-VRAM, alpha)", Inputs table, kv_store row,
     kvfp4s: K/V kept as NVFP4 -- E2M1 values with one e4m3 scale per 16
     elements (0.5625 byte per element) -- with Q and K Hadamard-rotated, and
     no delta_s and no Q-centering.

Readings where the page leaves a step open:
  R20 e2m1 is the 4-bit float with 1 sign, 2 exponent and 1 mantissa bit:
      magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 (codes 0-7; bit 3 is the sign).
      Encoding rounds to nearest, ties to the even code, and saturates at
      +-6.  The e4m3 scale is the OCP format of the kvf8s oracle (R13).
  R21 Blocks are 16 consecutive values along the head dimension of one
      (token, head) row.  Scale s = e4m3(absmax / 6) of the block; codes =
      e2m1(x / s); a block whose scale is 0 has all codes 0.  There is no
      second-level (per-tensor) scale: the page names only the per-16 e4m3
      scale.
  R22 K is rotated (k' = k H, the kvi8r basis) before encoding; V is not
      (the page rotates "Q/K"), so the output needs no un-rotation.
  R23 The result is exact softmax attention of the rotated query over the
      dequantised store, O = softmax(q' K^T * scale) V.  A dequantised value
      code * scale is exact in fp16: the product of a 2-bit and a 4-bit
      significand has at most 6 bits, and 2^-10 <= |value| <= 2688 or value
      = 0, inside fp16's range (subnormals step by 2^-24), so a kernel may
      dequantise to fp16 without rounding.
"""

from __future__ import annotations

import numpy as np

from .kvf8s import e4m3_decode, e4m3_encode
from .kvi8r import HEAD_DIM, as_f64, default_scale, rotate, softmax_attention

BLOCK = 16
E2M1_MAX = 6.0
_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e2m1_values() -> np.ndarray:
    """The 16 e2m1 code values (fp64); code 8 is -0."""
    return np.concatenate([_MAG, -_MAG])


def e2m1_encode(x) -> np.ndarray:
    """Codes (uint8, 0-15) of fp64 values: nearest e2m1 value, ties to the
    even code, saturating at +-6; the sign bit (8) follows the sign of x."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E2M1_MAX)
    hi = np.minimum(np.searchsorted(_MAG, a, side="left"), len(_MAG) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo, d_hi = a - _MAG[lo], _MAG[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    mag = np.where(a == _MAG[hi], hi, np.where(pick_hi, hi, lo)).astype(np.uint8)
    return np.where(np.signbit(x), mag | np.uint8(8), mag).astype(np.uint8)


def e2m1_decode(codes) -> np.ndarray:
    return e2m1_values()[np.asarray(codes, dtype=np.uint8)]


def encode_blocks(x) -> tuple[np.ndarray, np.ndarray]:
    """NVFP4 encoding of rows [..., 128]: (codes [..., 128] uint8 0-15, e4m3
    scale codes [..., 8] uint8) per reading R21."""
    x = as_f64(x)
    g = x.reshape(*x.shape[:-1], x.shape[-1] // BLOCK, BLOCK)
    amax = np.max(np.abs(g), axis=-1)
    sc = e4m3_encode(amax / E2M1_MAX)
    s = e4m3_decode(sc)
    safe = np.where(s > 0, s, 1.0)[..., None]
    codes = np.where((s > 0)[..., None], e2m1_encode(g / safe), np.uint8(0)).astype(np.uint8)
    return codes.reshape(x.shape), sc


def dequant(codes: np.ndarray, scale_codes: np.ndarray) -> np.ndarray:
    """code value * block scale, [..., 128] fp64."""
    v = e2m1_decode(codes)
    s = np.repeat(e4m3_decode(scale_codes), BLOCK, axis=-1)
    return v * s


def build_store_kvfp4(K, V) -> dict:
    """The kvfp4 store of K and V ([heads, seq, 128] each): K rotated, V not."""
    kc, ks = encode_blocks(rotate(K))
    vc, vs = encode_blocks(as_f64(V))
    return {"k_codes": kc, "k_scales": ks, "v_codes": vc, "v_scales": vs}


def attend_kvfp4(Q, store: dict, scale: float | None = None, heads=None) -> np.ndarray:
    """O = softmax(q' K^T * scale) V over the dequantised store (R23); q' = Q H
    in fp64.  ``heads`` indexes the store's heads for the rows of Q."""
    Q = as_f64(Q)
    scale = default_scale(Q.shape[-1]) if scale is None else scale
    hs = range(Q.shape[0]) if heads is None else heads
    out = np.empty(Q.shape)
    for i, h in enumerate(hs):
        kd = dequant(store["k_codes"][h], store["k_scales"][h])
        vd = dequant(store["v_codes"][h], store["v_scales"][h])
        out[i] = softmax_attention(rotate(Q[i]), kd, vd, scale)
    return out


def pack_codes(codes: np.ndarray) -> np.ndarray:
    """Two codes per byte, element 2i in the low nibble: [..., 128] ->
    [..., 64] (the store's byte layout)."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def unpack_codes(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


__all__ = ["BLOCK", "E2M1_MAX", "HEAD_DIM", "e2m1_values", "e2m1_encode", "e2m1_decode", "encode_blocks",
           "dequant", "build_store_kvfp4", "attend_kvfp4", "pack_codes", "unpack_codes"]
