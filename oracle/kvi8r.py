"""fp64 CPU oracle for the kvi8r K/V store and the attention over it.

THIS IS TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py`` (its CPU-baseline leg and ``--impl reference``) may import it.
The product path (the CUDA library and its binding) never imports, links or
calls anything here, and nothing here imports the product package.

What is computed, and where it is stated
----------------------------------------
[P1] "H3 Streamed Blocks (exact low-VRAM, alpha)" (comfy.icu node page),
     Inputs table:
       * kv_store row: kvi8r keeps K and V as int8 with one fp16 scale per row
         (per token, per head) in a fixed orthonormal 128-wide Hadamard-rotated
         basis of the head dim; the query chunk is rotated to match and the
         output is un-rotated once; a K/V block is dequantised as one
         int8->fp16 cast times the scale; attention runs blockwise over
         ``kv_block`` (default 16384) with an online-softmax combine.
       * q_chunk row: query tokens per attention call, exact at any value.
       * kv_block row: K/V attended in blocks with a log-sum-exp combine.
[P2] "Low VRAM, low RAM: the de-rope on a 16 GB card" (LOWVRAM.md):
       * "The K/V store options" table, kvi8r row (same definition; the
         dequant is "no GEMM").
       * the paragraph on why the rotation: the Hadamard spreads outlier
         channels before rounding, scores are invariant (q.k = (qH).(kH)) and
         P.V comes back through H^T once.
       * "What is exact, and what is not": the exact store is plain softmax
         attention, chunked.

Readings where the pages leave a step open (each the plainest one the rest of
the pages supports):
  R1  H is the Sylvester-ordered Hadamard matrix of order 128 divided by
      sqrt(128) (no random signs, since the basis is "fixed"). It is symmetric,
      so H^T = H.
  R2  "absmax scale" with "cast * scale" dequant: s = absmax(x')/127, so the
      code range is the symmetric [-127, 127].
  R3  s is rounded to fp16 (round to nearest even) and the codes are computed
      with the stored fp16 s.  If absmax/127 overflows fp16, s saturates at
      65504 (the largest finite fp16); codes are clamped to [-127, 127].
  R4  codes = round-half-to-even(x'/s).
  R5  a row whose fp16 scale is 0 (all-zero row, or absmax/127 below half the
      smallest fp16 subnormal) has all codes 0.
  R6  softmax scale defaults to 1/sqrt(128); attention is non-causal and
      unmasked; output is fp32 (this oracle returns fp64).
  R8  the per-32-value variant (the write-up's roadmap: "a per-32-value
      scale variant of kvi8r (finer than per row)") splits each rotated row
      into 4 consecutive groups of 32 values and gives each group its own
      scale, defined as in R2-R5 over the group; dequantisation multiplies
      each code by its group's scale.
  R7  kv_block does not change the mathematical result: the blockwise
      log-sum-exp combine equals one full softmax.  ``attend`` uses one full
      softmax; ``attend_blockwise`` follows the blockwise description and is
      checked against it.
"""

from __future__ import annotations

import numpy as np

HEAD_DIM = 128
CODE_MAX = 127
FP16_MAX = 65504.0


# --------------------------------------------------------------------------
# inputs
# --------------------------------------------------------------------------
def as_f64(x) -> np.ndarray:
    """Exact fp64 copy of a NumPy array or a (CPU) torch tensor of any float
    dtype, bf16 included (every bf16/fp16/fp32 value is exact in fp64)."""
    if hasattr(x, "detach"):  # torch tensor, without importing torch here
        x = x.detach().to("cpu")
        if str(x.dtype) in ("torch.bfloat16", "torch.float16"):
            x = x.float()
        x = x.numpy()
    return np.asarray(x, dtype=np.float64)


# --------------------------------------------------------------------------
# A1: the fixed orthonormal 128-wide Hadamard basis   [P1 kv_store; P2 rotation]
# --------------------------------------------------------------------------
def hadamard(n: int = HEAD_DIM) -> np.ndarray:
    """Sylvester Hadamard matrix of order n, scaled by 1/sqrt(n) so that
    H @ H.T = I (reading R1)."""
    if n < 1 or n & (n - 1):
        raise ValueError("order must be a power of two")
    h = np.ones((1, 1))
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h / np.sqrt(n)


def rotate(x: np.ndarray) -> np.ndarray:
    """x' = x H applied to every head-dim row (last axis)."""
    x = as_f64(x)
    return x @ hadamard(x.shape[-1])


def unrotate(x: np.ndarray) -> np.ndarray:
    """x = x' H^T (the single un-rotation of the output)."""
    x = as_f64(x)
    return x @ hadamard(x.shape[-1]).T


# --------------------------------------------------------------------------
# A2: per-row absmax int8 with one fp16 scale        [P1 kv_store; P2 table]
# --------------------------------------------------------------------------
def fp16_round(x) -> np.ndarray:
    """Round fp64 values to the nearest fp16 value (ties to even), returned as
    fp64.  Overflow gives +-inf, as an fp16 cast does."""
    with np.errstate(over="ignore"):
        return np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)


def row_scales(xr: np.ndarray) -> np.ndarray:
    """s = fp16(absmax(x')/127) per row (readings R2, R3), saturated at 65504."""
    a = np.max(np.abs(xr), axis=-1)
    s = fp16_round(a / CODE_MAX)
    return np.minimum(s, FP16_MAX)


def quantize(xr: np.ndarray, s: np.ndarray) -> np.ndarray:
    """int8 codes = clamp(rne(x'/s), -127, 127) with the stored fp16 scale
    (readings R3-R5)."""
    s = np.asarray(s, dtype=np.float64)
    safe = np.where(s > 0, s, 1.0)[..., None]
    c = np.rint(xr / safe)  # np.rint rounds half to even
    c = np.clip(c, -CODE_MAX, CODE_MAX)
    c = np.where((s > 0)[..., None], c, 0.0)
    return c.astype(np.int8)


def encode_rows(x) -> tuple[np.ndarray, np.ndarray]:
    """Rotate then quantise rows of K or V: returns (codes int8, scales fp64
    holding fp16 values)."""
    xr = rotate(x)
    s = row_scales(xr)
    return quantize(xr, s), s


def build_store(K, V) -> dict:
    """The kvi8r store of K and V ([heads, seq, 128] each)."""
    kc, ks = encode_rows(K)
    vc, vs = encode_rows(V)
    return {"k_codes": kc, "k_scales": ks, "v_codes": vc, "v_scales": vs}


def dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """K^' = code * scale (the pages' int8->fp16 cast times the scale, here in
    exact fp64).  Per-row scales have one axis fewer than the codes; per-group
    scales (reading R8) have a last axis of 128/group, each covering that many
    consecutive values."""
    scales = np.asarray(scales, np.float64)
    if scales.ndim == codes.ndim:  # per-group scales
        group = codes.shape[-1] // scales.shape[-1]
        return codes.astype(np.float64) * np.repeat(scales, group, axis=-1)
    return codes.astype(np.float64) * scales[..., None]


# --------------------------------------------------------------------------
# per-32-value scale variant (reading R8)
# --------------------------------------------------------------------------
def group_scales(xr: np.ndarray, group: int = 32) -> np.ndarray:
    """One fp16 scale per `group` consecutive rotated values (R2, R3 per
    group): shape [..., 128/group]."""
    g = xr.reshape(*xr.shape[:-1], xr.shape[-1] // group, group)
    return row_scales(g)


def encode_rows_grouped(x, group: int = 32) -> tuple[np.ndarray, np.ndarray]:
    """Rotate, then quantise every group of `group` values with its own scale."""
    xr = rotate(x)
    s = group_scales(xr, group)
    g = xr.reshape(*xr.shape[:-1], xr.shape[-1] // group, group)
    codes = quantize(g, s).reshape(xr.shape)
    return codes, s


def build_store_grouped(K, V, group: int = 32) -> dict:
    kc, ks = encode_rows_grouped(K, group)
    vc, vs = encode_rows_grouped(V, group)
    return {"k_codes": kc, "k_scales": ks, "v_codes": vc, "v_scales": vs}


# --------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------
def default_scale(d: int = HEAD_DIM) -> float:
    return 1.0 / np.sqrt(d)


def softmax_attention(q, k, v, scale: float, row_block: int = 1024) -> np.ndarray:
    """Plain softmax attention for one head: softmax(q k^T * scale) v, with the
    full softmax over every key for each query row.  Query rows are evaluated
    ``row_block`` at a time only to bound memory; rows are independent."""
    q, k, v = as_f64(q), as_f64(k), as_f64(v)
    out = np.empty((q.shape[0], v.shape[1]))
    for r0 in range(0, q.shape[0], row_block):
        s = (q[r0:r0 + row_block] @ k.T) * scale
        s -= s.max(axis=1, keepdims=True)
        p = np.exp(s)
        out[r0:r0 + row_block] = (p @ v) / p.sum(axis=1, keepdims=True)
    return out


def attend(Q, store: dict, scale: float | None = None, heads=None) -> np.ndarray:
    """kvi8r attention: q' = Q H, S = q' K^'^T * scale over the dequantised
    rotated store, P = softmax(S), O = (P V^') H^T.  Q is [heads, q_seq, 128]
    (or a subset of heads given by ``heads``, an index list into the store)."""
    Q = as_f64(Q)
    scale = default_scale(Q.shape[-1]) if scale is None else scale
    hs = range(Q.shape[0]) if heads is None else heads
    out = np.empty(Q.shape)
    for i, h in enumerate(hs):
        kd = dequant(store["k_codes"][h], store["k_scales"][h])
        vd = dequant(store["v_codes"][h], store["v_scales"][h])
        o_rot = softmax_attention(rotate(Q[i]), kd, vd, scale)
        out[i] = unrotate(o_rot)
    return out


def attend_exact(Q, K, V, scale: float | None = None) -> np.ndarray:
    """The exact store: plain softmax attention on the given (bf16) values."""
    Q, K, V = as_f64(Q), as_f64(K), as_f64(V)
    scale = default_scale(Q.shape[-1]) if scale is None else scale
    return np.stack([softmax_attention(Q[h], K[h], V[h], scale) for h in range(Q.shape[0])])


def attend_blockwise(q, k, v, kv_block: int, scale: float) -> np.ndarray:
    """One head, following the blockwise description: for each K/V block b
    (in order) attend to get the block's un-normalised output O_b, its row
    max m_b and row sum l_b, then merge into the running (M, Lambda, O) by the
    log-sum-exp rule: M' = max(M, m_b); O <- O e^(M-M') + O_b e^(m_b-M');
    Lambda <- Lambda e^(M-M') + l_b e^(m_b-M').  Returns O / Lambda."""
    q, k, v = as_f64(q), as_f64(k), as_f64(v)
    M = np.full((q.shape[0], 1), -np.inf)
    lam = np.zeros((q.shape[0], 1))
    O = np.zeros((q.shape[0], v.shape[1]))
    for b0 in range(0, k.shape[0], kv_block):
        s = (q @ k[b0:b0 + kv_block].T) * scale
        m_b = s.max(axis=1, keepdims=True)
        p = np.exp(s - m_b)
        l_b = p.sum(axis=1, keepdims=True)
        o_b = p @ v[b0:b0 + kv_block]
        m_new = np.maximum(M, m_b)
        a = np.exp(M - m_new)
        bta = np.exp(m_b - m_new)
        O = O * a + o_b * bta
        lam = lam * a + l_b * bta
        M = m_new
    return O / lam


def rel_rms(a, b) -> float:
    """||a - b|| / ||b|| (the pages' quality number is of this kind)."""
    a, b = as_f64(a), as_f64(b)
    return float(np.sqrt(np.sum((a - b) ** 2) / np.sum(b ** 2)))
