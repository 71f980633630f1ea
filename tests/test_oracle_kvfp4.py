"""Pins of the kvfp4 oracle (NVFP4 store: e2m1 values with one e4m3 scale per
16) against what the page and the mathematics fix, independent of the
oracle's own code: the e2m1 format written from its bit fields, nearest-value
rounding by brute force, the closed form of a one-channel key after the
rotation, exact reconstruction of values already on the grid (which reduces
the attention to the textbook one), and closed-form special cases.
"""
import numpy as np
import pytest

import oracle
from oracle import kvf8s as f8
from oracle import kvfp4 as f4
from store_h3kv_build_gb300 import synth


def _e2m1_from_bits(c: int) -> float:
    # 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit; exponent 0 is
    # subnormal: m * 2^-1
    sign = -1.0 if c & 8 else 1.0
    e, m = (c >> 1) & 3, c & 1
    return sign * (m * 0.5 if e == 0 else (1 + m / 2) * 2.0 ** (e - 1))


def test_e2m1_values_from_bit_fields():
    v = f4.e2m1_values()
    assert np.array_equal(v, [_e2m1_from_bits(c) for c in range(16)])
    assert v[7] == 6.0 and v[1] == 0.5 and v[2] == 1.0 and np.signbit(v[8])


def test_e2m1_encode_is_nearest_by_brute_force():
    # every finite input goes to a nearest value (saturating at +-6); on an
    # exact midpoint the even code (mantissa bit 0) wins
    vals = np.array([_e2m1_from_bits(c) for c in range(8)])
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.uniform(-8, 8, 20000), np.arange(-7, 7.01, 0.125)])
    got = f4.e2m1_encode(x)
    for xi, c in zip(x, got):
        a = min(abs(xi), 6.0)
        d = np.abs(vals - a)
        best = np.flatnonzero(d == d.min())
        want = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        assert c & 7 == want and bool(c & 8) == bool(np.signbit(xi))


def test_e2m1_midpoints():
    # midpoints between neighbours round to the value whose code is even
    assert list(f4.e2m1_decode(f4.e2m1_encode([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]))) == \
        [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]
    assert list(f4.e2m1_decode(f4.e2m1_encode([7.0, 1e9, -1e9]))) == [6.0, 6.0, -6.0]
    assert f4.e2m1_encode(-0.0) == 8 and f4.e2m1_encode(0.0) == 0


def test_pack_layout():
    # element 2i in the low nibble of byte i
    c = np.arange(16, dtype=np.uint8).repeat(8)[:128].reshape(1, 128)
    c[0, :4] = [1, 2, 3, 4]
    p = f4.pack_codes(c)
    assert p.shape == (1, 64) and p[0, 0] == 0x21 and p[0, 1] == 0x43
    assert np.array_equal(f4.unpack_codes(p), c)


def test_block_absmax_encodes_to_six():
    # s = e4m3(amax/6) lies within 2^-4 of amax/6, so amax/s is in
    # [5.65, 6.4]: past the 4|6 midpoint, the block maximum always encodes to +-6
    _, k, v = synth.make_qkv(2, 96, seed=1, k_outliers=True)
    for x in (oracle.rotate(k), oracle.as_f64(v)):
        codes, sc = f4.encode_blocks(x)
        g = x.reshape(2, 96, 8, 16)
        cg = codes.reshape(2, 96, 8, 16)
        i = np.argmax(np.abs(g), axis=-1)
        top = np.take_along_axis(cg, i[..., None], axis=-1)[..., 0]
        assert np.all(top & 7 == 7)
        assert np.array_equal(sc, f8.e4m3_encode(np.abs(g).max(axis=-1) / 6.0))


def test_dequant_error_bound():
    # round to nearest on the e2m1 grid times s: |x - q s| <= s (half the
    # widest gap, 4..6), including the saturated part above 6 s
    _, k, v = synth.make_qkv(1, 200, seed=2, k_outliers=True)
    for x in (oracle.rotate(k), oracle.as_f64(v)):
        codes, sc = f4.encode_blocks(x)
        s = np.repeat(f8.e4m3_decode(sc), 16, axis=-1)
        assert np.all(np.abs(f4.dequant(codes, sc) - x) <= s)


def test_one_channel_key_closed_form():
    # k = x e_c rotates to x/sqrt(128) times the signs of Hadamard row c
    # ((-1)^popcount(c & j)); every block then has amax |x|/sqrt(128), so
    # every element encodes to +-6 s with s = e4m3(|x| / (6 sqrt 128))
    x, c = 3.0, 37
    k = np.zeros((1, 1, 128))
    k[0, 0, c] = x
    codes, sc = f4.encode_blocks(oracle.rotate(k))
    s = f8.e4m3_decode(f8.e4m3_encode(x / (6 * np.sqrt(128))))
    sign = np.array([(-1.0) ** bin(c & j).count("1") for j in range(128)])
    assert np.all(f8.e4m3_decode(sc) == s)
    assert np.array_equal(f4.dequant(codes, sc)[0, 0], 6 * s * sign)


def _on_grid(rng, shape):
    # rows whose 16-value blocks are exact e2m1 multiples of an e4m3 scale,
    # with the block maximum at 6 s (so the encoder reproduces them exactly)
    s = f8.e4m3_decode(rng.integers(0x20, 0x50, size=shape[:-1] + (8,)).astype(np.uint8))
    vals = f4.e2m1_values()[rng.integers(0, 16, size=shape)]
    vals.reshape(*shape[:-1], 8, 16)[..., 0] = 6.0
    return vals * np.repeat(s, 16, axis=-1)


def test_grid_values_round_trip_exactly():
    rng = np.random.default_rng(3)
    y = _on_grid(rng, (2, 50, 128))
    codes, sc = f4.encode_blocks(y)
    assert np.array_equal(f4.dequant(codes, sc), y)


def test_attention_on_grid_store_is_textbook_attention():
    # K = Y H with Y on the grid: the store holds K H = Y exactly, so the
    # kvfp4 attention (rotated query against the rotated keys) must equal
    # softmax(Q K^T * scale) V; a query left unrotated, or keys rotated twice,
    # fails this
    rng = np.random.default_rng(4)
    y = _on_grid(rng, (2, 70, 128)) * 0.25
    K = y @ oracle.hadamard()                 # H is symmetric and H H = I
    V = _on_grid(rng, (2, 70, 128))
    Q = rng.standard_normal((2, 33, 128))
    st = f4.build_store_kvfp4(K, V)
    assert np.array_equal(f4.dequant(st["v_codes"], st["v_scales"]), V)
    got = f4.attend_kvfp4(Q, st)
    ref = np.stack([oracle.softmax_attention(Q[h], K[h], V[h], 1 / np.sqrt(128)) for h in range(2)])
    assert np.max(np.abs(got - ref)) < 1e-11


def test_attention_closed_forms():
    rng = np.random.default_rng(5)
    _, k, v = synth.make_qkv(1, 40, seed=6)
    st = f4.build_store_kvfp4(k, v)
    vd = f4.dequant(st["v_codes"], st["v_scales"])[0]
    # Q = 0: uniform weights, the mean of the dequantised V rows
    out = f4.attend_kvfp4(np.zeros((1, 3, 128)), st)
    assert np.max(np.abs(out[0] - vd.mean(axis=0))) < 1e-13
    # one key: every query returns that key's dequantised V row
    st1 = f4.build_store_kvfp4(k[:, :1], v[:, :1])
    out = f4.attend_kvfp4(rng.standard_normal((1, 5, 128)), st1)
    vd1 = f4.dequant(st1["v_codes"], st1["v_scales"])[0, 0]
    assert np.max(np.abs(out[0] - vd1)) < 1e-13


def test_zero_inputs_have_zero_codes():
    z = np.zeros((1, 9, 128))
    st = f4.build_store_kvfp4(z, z)
    assert not any(st[n].any() for n in ("k_codes", "k_scales", "v_codes", "v_scales"))


def test_quality_between_int8_and_page_figure():
    # 4-bit K/V is coarser than the per-row int8 of kvi8r; on gaussian inputs
    # (Q and P unquantised here) it is finer than the page's fully fp4
    # attention on gaussian inputs, rel-rms 0.192
    q, k, v = synth.make_qkv(2, 512, seed=7)
    ex = oracle.attend_exact(q, k, v)
    r4 = oracle.rel_rms(f4.attend_kvfp4(q, f4.build_store_kvfp4(k, v)), ex)
    r8 = oracle.rel_rms(oracle.attend(q, oracle.build_store(k, v)), ex)
    assert r8 < r4 < 0.192


def test_quality_with_key_outliers():
    # four key channels at 20x (the synthetic outlier inputs): the rotation
    # spreads them over every block, and the 4-bit keys carry most of the
    # error.  The page's outlier figure (0.293) is on a proxy it does not
    # define, so only the ordering against int8 and a loose ceiling are fixed
    q, k, v = synth.make_qkv(2, 512, seed=7, k_outliers=True)
    ex = oracle.attend_exact(q, k, v)
    r4 = oracle.rel_rms(f4.attend_kvfp4(q, f4.build_store_kvfp4(k, v)), ex)
    r8 = oracle.rel_rms(oracle.attend(q, oracle.build_store(k, v)), ex)
    assert 4 * r8 < r4 < 0.4
