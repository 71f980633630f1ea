"""GPU parity of h3kv_build_store (through the C ABI) against the fp64 oracle.

The store is the kv_store row of the H3 Streamed Blocks Inputs table: rows
rotated by the fixed Hadamard basis, one fp16 absmax scale per (token, head),
int8 codes.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import compare_store, oracle_store_heads
from store_h3kv_build_gb300 import synth

pytestmark = pytest.mark.gpu


def _build(K, V):
    from store_h3kv_build_gb300 import binding as b
    st = b.build_store(K, V)
    b.sync_status()
    return st


def _check_all(st, K, V, heads=None, what=""):
    heads = list(range(K.shape[0])) if heads is None else heads
    ref = oracle_store_heads(K.cpu(), V.cpu(), heads)
    out = {}
    for name in ("k", "v"):
        out[name] = compare_store(getattr(st, f"{name}_codes")[heads], getattr(st, f"{name}_scales")[heads],
                                  ref[f"{name}_codes"], ref[f"{name}_scales"], f"{what} {name}")
    return out


def test_store_tiny(cuda):
    q, k, v = synth.make_qkv(1, 1024, seed=0)
    st = _build(k.to(cuda), v.to(cuda))
    _check_all(st, k, v, what="tiny")


@pytest.mark.parametrize("heads,seq", [(3, 1000), (1, 1), (2, 129), (5, 77)])
def test_store_ragged(cuda, heads, seq):
    q, k, v = synth.make_qkv(heads, seq, seed=4)
    st = _build(k.to(cuda), v.to(cuda))
    _check_all(st, k, v, what=f"{heads}x{seq}")


def test_store_special_rows(cuda):
    # zero row, rows whose scale underflows to 0, lands in the fp16 subnormal
    # range, saturates at 65504, single-channel rows (closed form: all codes
    # +-127), and outlier rows.
    k = synth.normal_f32((1, 300, 128), 9)
    k[0, 0] = 0
    k[0, 1] = 0
    k[0, 1, 7] = 1e-9
    k[0, 2] = 0
    k[0, 2, 3] = 5e-4
    k[0, 3] = 0
    k[0, 3, 5] = 1e12
    k[0, 4] = 0
    k[0, 4, 9] = -3.0
    k[0, 5:40, 11] *= 50
    kb = k.to(torch.bfloat16)
    vb = synth.normal_bf16((1, 300, 128), 10)
    st = _build(kb.to(cuda), vb.to(cuda))
    _check_all(st, kb, vb, what="special")
    kc = st.k_codes.cpu().numpy()
    ks = st.k_scales.cpu().double().numpy()
    assert ks[0, 0] == 0 and not kc[0, 0].any()
    assert ks[0, 1] == 0 and not kc[0, 1].any()
    assert ks[0, 3] == 65504.0
    assert np.all(np.abs(kc[0, 4]) == 127)


def test_store_outlier_config_h24_l32768(cuda):
    w = synth.WORKLOADS["h24_l32768_outlier"]
    q, k, v = synth.make_qkv(w["heads"], w["seq"], seed=0, k_outliers=True)
    st = _build(k.to(cuda), v.to(cuda))
    _check_all(st, k, v, what="h24 l32768 outlier")


@pytest.mark.slow
def test_store_full_size_h32_l217088(cuda):
    w = synth.WORKLOADS["h32_l217088_outlier"]
    q, k, v = synth.make_qkv(w["heads"], w["seq"], seed=0, k_outliers=True, device=cuda)
    del q
    st = _build(k, v)
    # every row: codes within range, the absmax entry reaches 127 where s > 0
    for name in ("k", "v"):
        codes = getattr(st, f"{name}_codes")
        assert int(codes.min()) >= -127 and int(codes.max()) <= 127
        amax = codes.abs().amax(dim=-1)
        nz = getattr(st, f"{name}_scales") > 0
        assert bool(((amax == 127) | ~nz).all())
    # sampled heads in full against the oracle
    _check_all(st, k.cpu(), v.cpu(), heads=[0, 31], what="h32 l217088")


def test_store_rotation_spreads_outliers(cuda):
    # The reason for the rotation: with 4 outlier channels x20, the per-row
    # quantisation error measured in the original basis is far below that of
    # quantising the raw rows.
    q, k, v = synth.make_qkv(1, 2048, seed=5, k_outliers=True)
    st = _build(k.to(cuda), v.to(cuda))
    deq = oracle.dequant(st.k_codes.cpu().numpy()[0], st.k_scales.cpu().double().numpy()[0])
    rot_err = np.abs(oracle.unrotate(deq) - oracle.as_f64(k[0]))
    raw = oracle.as_f64(k[0])
    s_raw = oracle.row_scales(raw)
    raw_err = np.abs(oracle.dequant(oracle.quantize(raw, s_raw), s_raw) - raw)
    assert rot_err.mean() < 0.5 * raw_err.mean()


@pytest.mark.parametrize("group", [0, 32])
def test_store_build_code_buffers_16_byte_aligned(cuda, group):
    # code buffers that are 16- but not 32-byte aligned take the 16-byte store
    # path; the store must be the same bit for bit as in aligned buffers
    from store_h3kv_build_gb300 import binding as b
    heads, seq = 3, 1337
    _, k, v = synth.make_qkv(heads, seq, seed=41, k_outliers=True, device=cuda)
    ref = b.build_store(k, v, scale_group=group)
    n = heads * seq * 128
    kbuf = torch.empty(n + 32, dtype=torch.int8, device=cuda)
    vbuf = torch.empty(n + 32, dtype=torch.int8, device=cuda)
    kc, vc = kbuf[16:16 + n].view(heads, seq, 128), vbuf[16:16 + n].view(heads, seq, 128)
    assert kc.data_ptr() % 32 == 16 and vc.data_ptr() % 32 == 16
    odd = b.Store(kc, vc, torch.empty_like(ref.k_scales), torch.empty_like(ref.v_scales))
    b.build_store(k, v, out=odd)
    b.sync_status()
    for name in ("k_codes", "v_codes", "k_scales", "v_scales"):
        assert torch.equal(getattr(odd, name), getattr(ref, name)), name
