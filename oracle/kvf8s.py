"""fp64 CPU oracle for the kvf8s K/V store (fp8 e4m3 in the kvi8s layout) and
the attention over it.

THIS IS TEST INFRASTRUCTURE, under the same rule as ``oracle.kvi8r``: only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU-baseline leg
and ``--impl reference``) may import it; the CUDA path never calls it.

What is computed, and where it is stated
----------------------------------------
[P1] "H3 Streamed Blocks (exact low-VRAM, alpha)", Inputs table, kv_store row:
     kvi8s keeps the same K/V bytes in SageAttention's kernel layout -- K with
     one scale per 64-token block, V in fp8 with one scale per channel, Q and
     K Hadamard-rotated first -- and attends on int8/fp8 tensor cores straight
     from the store, with no dequantisation.
[P2] "Low VRAM, low RAM: the de-rope on a 16 GB card", "The K/V store
     options" table, kvi8s row: K is smoothed by its mean before the
     per-64-token-block scale; V is fp8 e4m3 per channel.  The roadmap's
     "fp8 K/V if a kernel takes it without dequant" is the rung built here.

Readings where the pages leave a step open:
  R13 kvf8s is kvi8s with the int8 K replaced by fp8 e4m3 (the fp8 tensor
      path; a K/V pair attended "straight from the store").  e4m3 is the OCP
      E4M3 format without infinities (bias 7, largest finite 448, smallest
      subnormal 2^-9).  Every encode rounds to nearest, ties to even, and
      saturates at +-448.
  R14 Rotation: q' = q H and k' = k H with the kvi8r basis (R1).  V is not
      rotated (the pages rotate "Q/K"), so the output needs no un-rotation.
  R15 Mean smoothing: mu = the mean over all tokens of k' (per head, per
      channel); the store encodes k' - mu.  Subtracting mu shifts every score
      of a query row by the same q'.mu, so the softmax is unchanged; mu is
      kept only as a diagnostic.
  R16 K scale: one fp32 scale per (head, 64-token block) s = absmax/448
      over the block's smoothed values (a tail block covers the tokens it
      has); codes = e4m3(x / s), the quotient rounded once, exactly, to the
      nearest e4m3 value (ties to even); a block with s = 0 has all codes 0.
  R17 V scale: one fp32 scale per (head, channel) s = absmax/448 over all
      tokens; codes = e4m3(v / s) rounded once from the exact quotient, as
      for K.
  R18 Q: one fp32 scale per rotated query row, s = absmax/448, codes =
      e4m3(q' / s) rounded from the exact quotient; the scores are
      S = (code_q . code_k) s_q s_k * scale.
      Reading for R16-R18: the pages name "fp8 e4m3 V per channel" and "fp8
      K/V if a kernel takes it without dequant" and give no arithmetic; the
      plainest reading of a scaled encode is the value divided by its scale,
      rounded once.  How a kernel forms the quotient (a reciprocal and a
      product, say) is its own precision step, bounded in its tests.
  R19 The result is exact softmax attention over the dequantised encodings
      (reading R7's blockwise combine changes nothing mathematically).  The
      fp8 P of a kernel's P.V product is a precision step of that kernel,
      bounded in its tests, not part of the definition.
"""

from __future__ import annotations

import numpy as np

from .kvi8r import HEAD_DIM, as_f64, default_scale, rotate, softmax_attention

E4M3_MAX = 448.0
K_BLOCK = 64


# --------------------------------------------------------------------------
# fp8 e4m3 (reading R13)
# --------------------------------------------------------------------------
def e4m3_values() -> np.ndarray:
    """The 256 e4m3 code values (fp64), NaN for the two NaN codes 0x7f and
    0xff.  Code bits: sign | 4 exponent bits (bias 7) | 3 mantissa bits; an
    exponent field of 0 is subnormal: (m/8) 2^-6."""
    out = np.empty(256)
    for c in range(256):
        sign = -1.0 if c & 0x80 else 1.0
        e, m = (c >> 3) & 0xF, c & 0x7
        if e == 0xF and m == 0x7:
            out[c] = np.nan
        elif e == 0:
            out[c] = sign * (m / 8.0) * 2.0 ** -6
        else:
            out[c] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return out


_POS = e4m3_values()[:0x7F]  # codes 0x00..0x7e: 0 and the 126 positive finite values, ascending


def e4m3_encode(x) -> np.ndarray:
    """Codes (uint8) of fp64 values: nearest e4m3 value, ties to the even
    code (the one whose last mantissa bit is 0), saturating at +-448.  The
    sign bit follows the sign of x, -0.0 included."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.searchsorted(_POS, a, side="left")          # first value >= a
    hi = np.minimum(hi, len(_POS) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo, d_hi = a - _POS[lo], _POS[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    mag = np.where(a == _POS[hi], hi, np.where(pick_hi, hi, lo)).astype(np.uint8)
    return np.where(np.signbit(x), mag | np.uint8(0x80), mag).astype(np.uint8)


def e4m3_decode(codes) -> np.ndarray:
    return e4m3_values()[np.asarray(codes, dtype=np.uint8)]


def fp32_round(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def e4m3_div(x, s) -> np.ndarray:
    """Codes (uint8) of x / s rounded once to the nearest e4m3 value, ties to
    the even code, saturating at +-448; the sign follows x (readings
    R16-R18).  x is fp64 and s a positive fp32 value (broadcast against x).

    The quotient is never rounded to fp64 first.  The two e4m3 values that
    bracket |x| / s are found from the fp64 quotient; the choice between them
    compares |x| with their midpoint times s.  A midpoint of two e4m3 values
    has at most 5 significant bits and s 24, so that product is exact in
    fp64, and the sign of the fp64 difference |x| - m s is the sign of the
    exact one."""
    x = np.asarray(x, dtype=np.float64)
    s = np.broadcast_to(np.asarray(s, dtype=np.float64), x.shape)
    a = np.abs(x)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = a / s
    lo = np.searchsorted(_POS, q, side="right") - 1    # _POS[lo] <= fp64 quotient
    lo = np.clip(lo, 0, len(_POS) - 1)
    hi = np.minimum(lo + 1, len(_POS) - 1)
    mid = (_POS[lo] + _POS[hi]) / 2                    # exact: 5 significant bits at most
    d = a - mid * s                                    # sign of |x| - mid s, exact
    pick_hi = (d > 0) | ((d == 0) & (hi % 2 == 0))
    mag = np.where(lo == hi, lo, np.where(pick_hi, hi, lo)).astype(np.uint8)  # lo == hi: 448, saturated
    return np.where(np.signbit(x), mag | np.uint8(0x80), mag).astype(np.uint8)


def _scaled_codes(x: np.ndarray, s: np.ndarray) -> np.ndarray:
    """e4m3(x / s) with s broadcast against x; all-zero codes where s = 0
    (readings R16-R18)."""
    s = np.broadcast_to(np.asarray(s, dtype=np.float64), np.shape(x))
    pos = s > 0
    return np.where(pos, e4m3_div(x, np.where(pos, s, 1.0)), np.uint8(0)).astype(np.uint8)


# --------------------------------------------------------------------------
# the store (readings R14-R17)
# --------------------------------------------------------------------------
def smooth_mean(Kr: np.ndarray) -> np.ndarray:
    """mu: mean over tokens of the rotated K, per head and channel (R15)."""
    return as_f64(Kr).mean(axis=-2)


def k_block_scales(Ks: np.ndarray, block: int = K_BLOCK) -> np.ndarray:
    """fp32 absmax/448 per (head, block of `block` tokens) of smoothed K (R16)."""
    H, L, _ = Ks.shape
    nb = (L + block - 1) // block
    s = np.empty((H, nb))
    for b in range(nb):
        s[:, b] = np.max(np.abs(Ks[:, b * block:(b + 1) * block]), axis=(1, 2))
    return fp32_round(s / E4M3_MAX)


def encode_k(K, block: int = K_BLOCK) -> dict:
    """Rotate, smooth and quantise K [heads, seq, 128] (R14-R16)."""
    Kr = rotate(K)
    mu = smooth_mean(Kr)
    Ks = Kr - mu[:, None, :]
    s = k_block_scales(Ks, block)
    s_tok = np.repeat(s, block, axis=1)[:, :Ks.shape[1]]
    return {"k_codes": _scaled_codes(Ks, s_tok[..., None]), "k_scales": s, "k_mean": mu}


def v_channel_scales(V) -> np.ndarray:
    """fp32 absmax/448 per (head, channel) over all tokens (R17); the fp32
    quotient of an exact bf16 absmax."""
    a = np.max(np.abs(as_f64(V)), axis=-2).astype(np.float32)
    return (a / np.float32(E4M3_MAX)).astype(np.float64)


def encode_v(V) -> dict:
    """V codes [heads, seq, 128] (token-major here) and fp32 per-channel
    scales [heads, 128]; codes e4m3(v / s) (R17)."""
    s = v_channel_scales(V)
    return {"v_codes": _scaled_codes(as_f64(V), s[:, None, :]), "v_scales": s}


def build_store_kvf8s(K, V, block: int = K_BLOCK) -> dict:
    """The kvf8s store of K and V ([heads, seq, 128] each)."""
    out = encode_k(K, block)
    out.update(encode_v(V))
    return out


def dequant_k(store: dict, h: int, block: int = K_BLOCK) -> np.ndarray:
    s = np.repeat(store["k_scales"][h], block)[:store["k_codes"].shape[1]]
    return e4m3_decode(store["k_codes"][h]) * s[:, None]


def dequant_v(store: dict, h: int) -> np.ndarray:
    return e4m3_decode(store["v_codes"][h]) * store["v_scales"][h][None, :]


# --------------------------------------------------------------------------
# the query and the attention (readings R18, R19)
# --------------------------------------------------------------------------
def encode_q(Q) -> tuple[np.ndarray, np.ndarray]:
    """Rotated query rows as (e4m3 codes, fp32 row scales)."""
    Qr = rotate(Q)
    s = fp32_round(np.max(np.abs(Qr), axis=-1) / E4M3_MAX)
    return _scaled_codes(Qr, s[..., None]), s


def attend_kvf8s(Q, store: dict, scale: float | None = None, heads=None, block: int = K_BLOCK) -> np.ndarray:
    """kvf8s attention: S = (Q codes . K codes) s_q s_k * scale, P = softmax(S)
    over every key, O = P (V codes * s_v), in the original basis (no
    un-rotation: V is not rotated).  ``heads`` indexes the store's heads for
    the rows of Q."""
    Q = as_f64(Q)
    scale = default_scale(Q.shape[-1]) if scale is None else scale
    hs = range(Q.shape[0]) if heads is None else heads
    qc, qs = encode_q(Q)
    out = np.empty(Q.shape)
    for i, h in enumerate(hs):
        qd = e4m3_decode(qc[i]) * qs[i][:, None]
        out[i] = softmax_attention(qd, dequant_k(store, h, block), dequant_v(store, h), scale)
    return out


__all__ = [
    "E4M3_MAX", "K_BLOCK", "HEAD_DIM", "e4m3_values", "e4m3_encode", "e4m3_decode", "e4m3_div", "fp32_round",
    "smooth_mean", "k_block_scales", "encode_k", "v_channel_scales", "encode_v", "build_store_kvf8s",
    "dequant_k", "dequant_v", "encode_q", "attend_kvf8s",
]
