"""Shared comparison helpers for the GPU parity tests (GPU path vs the oracle).

Tolerances (kvi8r pages give none; these are the build's stated bar):
  * int8 codes: identical except at most 1e-4 of the entries off by +-1 (the
    GPU rotates in fp32, the oracle in fp64, so a value at a rounding tie or a
    scale one fp16 ulp apart can land on the neighbouring code);
  * fp16 scales: within 1 fp16 ulp (bit patterns of positive values differ by
    at most 1);
  * attention output (fp32): max abs error <= 2e-2 and mean abs error <= 2e-3
    against the fp64 oracle on N(0, 1)-scale inputs.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

CODE_MISMATCH_FRAC = 1e-4
ATT_MAX_ABS = 2e-2
ATT_MEAN_ABS = 2e-3


def fp16_bits(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().cpu().contiguous().view(torch.int16).numpy().astype(np.int32) & 0xFFFF
    return np.asarray(t, dtype=np.float16).view(np.uint16).astype(np.int32)


def compare_store(gpu_codes, gpu_scales, ref_codes, ref_scales, what=""):
    """Assert the GPU store rows equal the oracle's within the stated bar and
    return (fraction of codes off by one, max scale ulp distance)."""
    gc = gpu_codes.detach().cpu().numpy().astype(np.int16)
    rc = np.asarray(ref_codes).astype(np.int16)
    assert gc.shape == rc.shape, what
    d = np.abs(gc - rc)
    assert d.max(initial=0) <= 1, f"{what}: code off by {d.max()}"
    frac = float((d != 0).mean()) if d.size else 0.0
    assert frac <= CODE_MISMATCH_FRAC, f"{what}: {frac:.2e} of codes differ"
    gs = fp16_bits(gpu_scales)
    rs = fp16_bits(np.asarray(ref_scales))
    ulp = int(np.abs(gs - rs).max(initial=0))
    assert ulp <= 1, f"{what}: scale off by {ulp} ulp"
    return frac, ulp


def compare_attention(gpu_out, ref_out, what=""):
    g = gpu_out.detach().cpu().double().numpy() if isinstance(gpu_out, torch.Tensor) else np.asarray(gpu_out)
    r = np.asarray(ref_out, dtype=np.float64)
    assert g.shape == r.shape, what
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - r)
    mx, mean = float(err.max()), float(err.mean())
    assert mx <= ATT_MAX_ABS and mean <= ATT_MEAN_ABS, f"{what}: max abs {mx:.3e} mean abs {mean:.3e}"
    return mx, mean


def oracle_store_heads(K, V, heads):
    """The oracle's store for the listed heads only (stacked in that order)."""
    parts = [oracle.build_store(K[h:h + 1], V[h:h + 1]) for h in heads]
    return {k: np.concatenate([p[k] for p in parts]) for k in parts[0]}


def store_to_numpy(store, heads=None):
    """GPU-built store (binding.Store) -> oracle-style dict of numpy arrays."""
    idx = slice(None) if heads is None else list(heads)
    return {
        "k_codes": store.k_codes[idx].cpu().numpy(),
        "v_codes": store.v_codes[idx].cpu().numpy(),
        "k_scales": store.k_scales[idx].cpu().double().numpy(),
        "v_scales": store.v_scales[idx].cpu().double().numpy(),
    }
