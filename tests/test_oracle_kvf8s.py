"""Pins of the kvf8s oracle (fp8 e4m3 store in the kvi8s layout) against what
the pages and the mathematics fix, independent of the oracle's own code:
the e4m3 format's defining values, PyTorch's float8_e4m3fn cast, the scaled
encode e4m3(x / s) against exact rational rounding and hand-worked ties,
closed-form special cases of attention (one of them analytic in the query's
scale), the softmax invariance that mean smoothing rests on, and error
bounds of round-to-nearest.
"""
from fractions import Fraction

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


def _e4m3_brute(x: Fraction) -> int:
    """The e4m3 code nearest to the exact rational x, ties to the even code,
    saturating at 448: a search over the format's values, from the bit
    fields, in exact rational arithmetic."""
    vals = []
    for c in range(0x7F):
        e, m = c >> 3, c & 7
        v = Fraction(m, 8) * Fraction(1, 64) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
        vals.append((v, c))
    a = min(abs(x), Fraction(448))
    best = min(vals, key=lambda vc: (abs(vc[0] - a), vc[1] & 1))
    return best[1] | (0x80 if x < 0 else 0)


def test_e4m3_div_matches_exact_rational_rounding():
    # brute force: the quotient of a bf16 or fp64 value by an fp32 scale,
    # rounded in exact rational arithmetic (no floating point anywhere)
    rng = np.random.default_rng(12)
    x = np.concatenate([
        rng.standard_normal(1500) * np.exp2(rng.integers(-10, 6, 1500)),
        synth.normal_f32((1, 1, 1500), 4).to(torch.bfloat16).double().numpy().ravel(),
    ])
    s = f8.fp32_round(np.abs(rng.standard_normal(x.size)) * np.exp2(rng.integers(-8, 2, x.size)) + 1e-3)
    got = f8.e4m3_div(x, s)
    ref = np.array([_e4m3_brute(Fraction(float(a)) / Fraction(float(b))) for a, b in zip(x, s)])
    assert np.array_equal(got, ref)


def test_e4m3_div_ties_that_a_reciprocal_product_misses():
    # scale 12.25 / 448 = 7/256, exact in fp32.  0.1708984375 / (7/256) = 6.25
    # exactly, the midpoint of 6 (0x4c) and 6.5 (0x4d): the tie goes to the
    # even code 0x4c.  The fp32 reciprocal 256/7 rounds up, so the fp32
    # product v * fp32(1/s) lands just above 6.25 and would give 0x4d.
    # Likewise 0.000347137451171875 / s = 6.5 * 2^-9, halfway between the
    # subnormals 6 * 2^-9 (0x06) and 7 * 2^-9 (0x07): 0x06.
    s = 7.0 / 256.0
    x = np.array([0.1708984375, 0.000347137451171875, -0.1708984375, 12.25, 1.0, 0.5, s, s / 2, 0.0])
    # hand-worked: 6.25 -> 0x4c; 6.5 * 2^-9 -> 0x06; sign bit; 448 -> 0x7e;
    # 36.57.. -> 36 (0x61); 18.29.. -> 18 (0x59); 1.0 -> 0x38; 0.5 -> 0x30; 0
    assert list(f8.e4m3_div(x, s)) == [0x4C, 0x06, 0xCC, 0x7E, 0x61, 0x59, 0x38, 0x30, 0x00]
    r = np.float32(1) / np.float32(s)
    assert f8.e4m3_encode(np.float64(np.float32(0.1708984375) * r)) == 0x4D  # the product's answer


def test_e4m3_div_by_powers_of_two_is_the_cast():
    # a power-of-two scale divides exactly, so the code is the (torch-pinned)
    # rounding of x * 2^-k itself
    rng = np.random.default_rng(13)
    x = rng.standard_normal(20000) * np.exp2(rng.integers(-12, 8, 20000))
    for k in (-6, 0, 3):
        assert np.array_equal(f8.e4m3_div(x, 2.0 ** k), f8.e4m3_encode(x / 2.0 ** k))


def test_v_channel_codes_hand_worked():
    # R17 on a channel whose absmax is 12.25: s_v = 12.25 / 448 = 7/256, and
    # the codes are the hand-worked quotients above; a second channel of
    # constant 3.5 has s_v = 1/128 and every code 448 (0x7e); a zero channel
    # has s_v = 0 and zero codes
    col = [12.25, 0.1708984375, 0.000347137451171875, -0.1708984375, 1.0, 0.5, 7.0 / 256.0, 7.0 / 512.0, 0.0]
    v = torch.zeros((1, len(col), 128), dtype=torch.float64)
    v[0, :, 0] = torch.tensor(col, dtype=torch.float64)
    v[0, :, 1] = 3.5
    st = f8.encode_v(v.to(torch.bfloat16))
    assert st["v_scales"][0, 0] == 7.0 / 256.0 and st["v_scales"][0, 1] == 1.0 / 128.0
    assert st["v_scales"][0, 2] == 0.0
    assert list(st["v_codes"][0, :, 0]) == [0x7E, 0x4C, 0x06, 0xCC, 0x61, 0x59, 0x38, 0x30, 0x00]
    assert np.all(st["v_codes"][0, :, 1] == 0x7E) and not st["v_codes"][0, :, 2:].any()


def test_v_scale_maps_channel_absmax_to_448():
    # per channel the largest |v| encodes to +-448 and no code is NaN
    _, _, v = synth.make_qkv(2, 100, seed=6)
    st = f8.encode_v(v)
    vv = v.float()
    assert np.array_equal(st["v_scales"], (vv.abs().amax(dim=1) / 448.0).double().numpy())
    assert np.all((st["v_codes"] & 0x7F) != 0x7F)
    idx = vv.abs().argmax(dim=1)
    for h in range(2):
        for d in range(0, 128, 17):
            assert st["v_codes"][h, idx[h, d], d] & 0x7F == 0x7E


def _rotated_one_hot(coeffs: dict) -> torch.Tensor:
    """A bf16 row q with q H = sqrt(128) * sum_c coeffs[c] e_c: row c of
    sqrt(128) H is a +-1 pattern, so q's entries are sums of +-coeffs."""
    Hs = np.sign(oracle.hadamard())  # +-1 Sylvester matrix
    q = sum(a * Hs[c] for c, a in coeffs.items())
    out = torch.tensor(q, dtype=torch.float64).to(torch.bfloat16)
    assert torch.equal(out.double(), torch.tensor(q))
    return out


def test_encode_q_codes_of_a_rotated_one_hot_row():
    # q' = sqrt(128) (0.25 e_5 + 0.125 e_40): s_q = fp32(0.25 sqrt(128) / 448),
    # the channel-5 value encodes to 448 (0x7e), channel 40 to 224 (0x76),
    # every other channel to (+-)0 -- codes that do not depend on s_q's
    # rounding (the fp64 rotation leaves values near 1e-17 off the two
    # channels, whose sign the zero code keeps)
    q = _rotated_one_hot({5: 0.25, 40: 0.125})[None, None, :]
    codes, s = f8.encode_q(q)
    assert codes[0, 0, 5] == 0x7E and codes[0, 0, 40] == 0x76
    assert not (np.delete(codes[0, 0], [5, 40]) & 0x7F).any()
    assert abs(s[0, 0] * 448.0 / (0.25 * np.sqrt(128.0)) - 1.0) < 2.0 ** -23


def test_attend_two_keys_closed_form_uses_the_query_scale():
    # query q' = a e_5, keys k1' = b e_5 and k2' = -b e_5 (a = b =
    # 0.25 sqrt(128); their mean is 0, so smoothing changes nothing), values
    # v1 = (7, 3.5, 0..), v2 = (-7, 3.5, 0..).  Every code is +-448 or 0, and
    # 7 / 448, 3.5 / 448 are powers of two, so dequantised V is exact.  With
    # scores +-a b * scale the softmax gives channel 0 = 7 tanh(a b scale) and
    # channel 1 = 3.5; a and b enter only through 448 * s_q and 448 * s_k,
    # each within 2^-24 of the exact value.  Dropping s_q (or a missing
    # rotation of q) moves channel 0 far from the closed form.
    a = b = 0.25 * np.sqrt(128.0)
    q = _rotated_one_hot({5: 0.25})[None, None, :]
    k1 = _rotated_one_hot({5: 0.25})
    k = torch.stack([k1, -k1])[None]
    v = torch.zeros((1, 2, 128), dtype=torch.float64)
    v[0, 0, :2] = torch.tensor([7.0, 3.5])
    v[0, 1, :2] = torch.tensor([-7.0, 3.5])
    st = f8.build_store_kvf8s(k, v.to(torch.bfloat16))
    scale = 1.0 / np.sqrt(128.0)
    out = f8.attend_kvf8s(q, st, scale=scale)[0, 0]
    assert abs(out[0] - 7.0 * np.tanh(a * b * scale)) < 7.0 * 4e-7
    assert abs(out[1] - 3.5) < 1e-12 and not out[2:].any()
    # a sharper softmax scale moves the closed form the same way
    out2 = f8.attend_kvf8s(q, st, scale=4 * scale)[0, 0]
    assert abs(out2[0] - 7.0 * np.tanh(4 * a * b * scale)) < 7.0 * 4e-7


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
