"""Pins of the kvf8s oracle (fp8 e4m3 store in the kvi8s layout) against what
the pages and the mathematics fix, independent of the oracle's own code:
the e4m3 format's defining values, PyTorch's float8_e4m3fn cast, closed-form
special cases of attention, the softmax invariance that mean smoothing rests
on, and error bounds of round-to-nearest.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import kvf8s as f8
from store_h3kv_build_gb300 import synth


def test_e4m3_defining_values():
    # OCP E4M3: largest finite 448 = 1.75 * 2^8 (0x7e), 1.0 = 0x38, smallest
    # normal 2^-6 (0x08), smallest subnormal 2^-9 (0x01), 0x7f/0xff NaN
    v = f8.e4m3_values()
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0
    assert v[0x38] == 1.0 and v[0x08] == 2.0 ** -6 and v[0x01] == 2.0 ** -9
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    fin = v[np.isfinite(v)]
    assert len(fin) == 254 and np.count_nonzero(fin > 0) == 126
    assert np.all(np.diff(v[:0x7F]) > 0)  # codes 0..0x7e ascend


def test_e4m3_ties_and_saturation():
    # halfway cases go to the even mantissa; beyond 448 saturates
    assert f8.e4m3_encode(1.0625) == 0x38          # between 1 and 1.125 -> 1
    assert f8.e4m3_encode(1.1875) == 0x3A          # between 1.125 and 1.25 -> 1.25
    assert f8.e4m3_encode(2.0 ** -10) == 0x00      # half the smallest subnormal -> 0
    assert f8.e4m3_encode(1.5 * 2.0 ** -9) == 0x02
    assert f8.e4m3_encode(1000.0) == 0x7E and f8.e4m3_encode(-1e30) == 0xFE
    assert f8.e4m3_encode(-0.0) == 0x80 and f8.e4m3_encode(0.0) == 0x00


def test_e4m3_matches_torch_cast():
    # PyTorch's float8_e4m3fn cast (round to nearest even) on a dense grid of
    # fp32 values inside the range where it does not overflow to NaN
    g = torch.Generator().manual_seed(11)
    x = torch.cat([
        torch.linspace(-460, 460, 200001),
        torch.randn(100000, generator=g) * torch.exp2(torch.randint(-14, 9, (100000,), generator=g).float()),
        torch.tensor(f8.e4m3_values()[np.isfinite(f8.e4m3_values())], dtype=torch.float32),
    ]).float()
    x = x[x.abs() < 464]  # the cast gives NaN from 464 up; the encode saturates
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = f8.e4m3_encode(x.double().numpy())
    assert np.array_equal(got, ref)


def test_e4m3_round_trip_bound():
    # round to nearest: relative error <= 2^-4 in the normal range, absolute
    # <= 2^-10 (half the subnormal spacing) below it
    rng = np.random.default_rng(1)
    x = rng.standard_normal(200000) * np.exp2(rng.integers(-12, 8, 200000))
    x = x[np.abs(x) <= 448]
    err = np.abs(f8.e4m3_decode(f8.e4m3_encode(x)) - x)
    normal = np.abs(x) >= 2.0 ** -6
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(x[normal]))
    assert np.all(err[~normal] <= 2.0 ** -10)


def test_smoothing_leaves_softmax_unchanged():
    # reading R15: subtracting one vector from every key shifts a query row's
    # scores by a constant, which the softmax cancels
    rng = np.random.default_rng(2)
    q, k, v = rng.standard_normal((3, 40, 128))
    mu = rng.standard_normal(128) * 3
    a = oracle.softmax_attention(q, k, v, 0.1)
    b = oracle.softmax_attention(q, k - mu, v, 0.1)
    assert np.max(np.abs(a - b)) < 1e-12


def test_mean_of_rotated_is_rotated_mean():
    # the mean commutes with the (linear) rotation: mu = mean(k) H
    _, k, _ = synth.make_qkv(2, 300, seed=3)
    Kr = oracle.rotate(k)
    mu = f8.smooth_mean(Kr)
    ref = oracle.as_f64(k).mean(axis=1) @ oracle.hadamard()
    assert np.max(np.abs(mu - ref)) < 1e-12


def test_k_block_scale_maps_absmax_to_448():
    # R16: in every 64-token block the element of largest magnitude encodes to
    # +-448 (0x7e / 0xfe), and no code is NaN
    _, k, v = synth.make_qkv(2, 200, seed=4, k_outliers=True)
    st = f8.build_store_kvf8s(k, v)
    Ks = oracle.rotate(k) - st["k_mean"][:, None, :]
    for h in range(2):
        for b in range(4):
            blk = Ks[h, b * 64:(b + 1) * 64]
            c = st["k_codes"][h, b * 64:(b + 1) * 64]
            i = np.unravel_index(np.argmax(np.abs(blk)), blk.shape)
            assert c[i] & 0x7F == 0x7E
            assert np.all((c & 0x7F) != 0x7F)
            assert st["k_scales"][h, b] == np.float32(np.abs(blk).max() / 448.0)
    assert st["k_scales"].shape == (2, 4)  # 200 tokens: three full blocks and a tail of 8


def test_k_dequant_error_bound():
    # per element |k'' - dequant| <= max(2^-4 |k''|, 2^-10 s) + fp32 scale rounding
    _, k, v = synth.make_qkv(1, 256, seed=5, k_outliers=True)
    st = f8.build_store_kvf8s(k, v)
    Ks = (oracle.rotate(k) - st["k_mean"][:, None, :])[0]
    s = np.repeat(st["k_scales"][0], 64)[:, None]
    err = np.abs(f8.dequant_k(st, 0) - Ks)
    bound = np.maximum(2.0 ** -4 * np.abs(Ks), 2.0 ** -10 * s) + 448 * s * 2.0 ** -23
    assert np.all(err <= bound)


def test_v_channel_scale_and_codes():
    # R17: per channel the largest |v| encodes to +-448; the codes are the
    # fp32 product v * fp32(1/s) rounded to e4m3, which PyTorch's fp32
    # arithmetic and e4m3 cast reproduce
    _, _, v = synth.make_qkv(2, 100, seed=6)
    st = f8.encode_v(v)
    vv = v.float()
    s = vv.abs().amax(dim=1) / 448.0
    assert np.array_equal(st["v_scales"], s.double().numpy())
    ref = (vv * (1.0 / s)[:, None, :]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(st["v_codes"], ref)
    idx = vv.abs().argmax(dim=1)
    for h in range(2):
        for d in range(0, 128, 17):
            assert st["v_codes"][h, idx[h, d], d] & 0x7F == 0x7E


def test_zero_inputs_have_zero_codes():
    k = torch.zeros((1, 70, 128), dtype=torch.bfloat16)
    v = torch.zeros((1, 70, 128), dtype=torch.bfloat16)
    st = f8.build_store_kvf8s(k, v)
    assert not st["k_codes"].any() and not st["v_codes"].any()
    assert not st["k_scales"].any() and not st["v_scales"].any()


def test_attend_constant_v_is_exact():
    # every key carries the same value row c: any softmax returns c, in the
    # original basis (V is not rotated), up to the e4m3 encoding of c
    q, k, _ = synth.make_qkv(1, 130, seed=7)
    c = torch.linspace(-3, 3, 128).to(torch.bfloat16)
    v = c.expand(1, 130, 128).contiguous()
    st = f8.build_store_kvf8s(k, v)
    out = f8.attend_kvf8s(q, st)
    dc = f8.dequant_v(st, 0)[0]
    assert np.max(np.abs(out[0] - dc[None, :])) < 1e-12
    # and dequant(c) is c: each channel holds one value, its own absmax
    assert np.max(np.abs(dc - oracle.as_f64(c))) < 1e-6 * 3


def test_attend_zero_query_is_mean_of_v():
    # q = 0: every score is 0 and the softmax is uniform
    _, k, v = synth.make_qkv(1, 77, seed=8)
    q = torch.zeros((1, 5, 128), dtype=torch.bfloat16)
    st = f8.build_store_kvf8s(k, v)
    out = f8.attend_kvf8s(q, st)
    ref = f8.dequant_v(st, 0).mean(axis=0)
    assert np.max(np.abs(out[0] - ref[None, :])) < 1e-12


def test_attend_single_key():
    q, k, v = synth.make_qkv(1, 1, seed=9)
    st = f8.build_store_kvf8s(k, v)
    out = f8.attend_kvf8s(q, st)
    assert np.max(np.abs(out[0, 0] - f8.dequant_v(st, 0)[0])) < 1e-12


@pytest.mark.parametrize("outliers,bound", [(False, 0.06), (True, 0.15)])
def test_attend_close_to_exact(outliers, bound):
    # the encoding is lossy: against exact attention on the same bf16 inputs
    # the relative rms is a few percent (0.045 plain, 0.110 with the outlier
    # K, whose scores spread ~3.7x wider), dominated by the fp8 Q.K product;
    # it is coarser than kvi8r on the same inputs
    q, k, v = synth.make_qkv(1, 1024, seed=0, k_outliers=outliers)
    st = f8.build_store_kvf8s(k, v)
    ex = oracle.attend_exact(q, k, v)
    r = oracle.rel_rms(f8.attend_kvf8s(q, st), ex)
    r_i8 = oracle.rel_rms(oracle.attend(q, oracle.build_store(k, v)), ex)
    assert r_i8 < r < bound
