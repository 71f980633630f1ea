"""Pins of the fp64 oracle against what the kvi8r pages and the mathematics fix.

Every check here compares the oracle with something other than itself: a
library routine (scipy's Hadamard, torch's fp16 cast), a closed form, an
invariant, or a brute-force evaluation written independently (pure-Python
loops with ``math.exp``).  Sources are the "H3 Streamed Blocks" node page
(Inputs table: kv_store, q_chunk and kv_block rows) and the "Low VRAM, low RAM"
write-up ("The K/V store options" table and its paragraph on the rotation).
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.linalg
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(12345)


def bf16_normal(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(torch.bfloat16)


# ---------------------------------------------------------------- Hadamard --
def test_hadamard_orthonormal_and_entries():
    H = oracle.hadamard()
    assert np.abs(H @ H.T - np.eye(128)).max() <= 1e-15
    assert np.allclose(np.abs(H), 1 / np.sqrt(128), rtol=0, atol=0)


def test_hadamard_is_scipy_sylvester():
    # scipy.linalg.hadamard builds the Sylvester-ordered matrix (textbook).
    for n in (1, 2, 4, 8, 128):
        assert np.array_equal(oracle.hadamard(n) * np.sqrt(n), scipy.linalg.hadamard(n))


def test_hadamard_h8_golden():
    # Sylvester H_8 written out by hand (rows: +/- patterns), golden fixture.
    rows = open(os.path.join(GOLDEN, "sylvester_h8.txt")).read().split()
    h8 = np.array([[1 if ch == "+" else -1 for ch in r] for r in rows])
    assert np.array_equal(oracle.hadamard(8) * np.sqrt(8), h8)


def test_hadamard_symmetric():
    H = oracle.hadamard()
    assert np.array_equal(H, H.T)


# ---------------------------------------------------------------- rotation --
def test_score_invariance_under_joint_rotation():
    # q.k = (qH).(kH)  (the pages' argument for rotating both sides)
    q = oracle.as_f64(bf16_normal((64, 128), 1))
    k = oracle.as_f64(bf16_normal((96, 128), 2))
    s0 = q @ k.T
    s1 = oracle.rotate(q) @ oracle.rotate(k).T
    assert np.abs(s0 - s1).max() <= 1e-12 * np.abs(s0).max()


def test_unrotate_inverts_rotate():
    x = RNG.standard_normal((5, 7, 128))
    assert np.abs(oracle.unrotate(oracle.rotate(x)) - x).max() <= 1e-13


def test_rotate_acts_on_last_axis_rows():
    # A transposed operand (H x instead of x H per row) fails this: the
    # rotated row of e_c is row c of H, i.e. column c as well (symmetric),
    # but for a non-basis row the product must match scipy's matrix per row.
    x = RNG.standard_normal((3, 128))
    ref = np.stack([scipy.linalg.hadamard(128).T @ r for r in x]) / np.sqrt(128)
    assert np.abs(oracle.rotate(x) - ref).max() <= 1e-13


# --------------------------------------------------------------- quantiser --
def test_fp16_round_matches_torch_cast():
    x = np.concatenate([RNG.standard_normal(10000) * 10.0 ** RNG.integers(-9, 5, 10000),
                        [1 + 2 ** -11, 1 + 3 * 2 ** -11, 65519.0, 65520.0, 2 ** -25, 3 * 2 ** -26]])
    ref = torch.tensor(x, dtype=torch.float64).to(torch.float16).to(torch.float64).numpy()
    got = oracle.fp16_round(x)
    assert np.array_equal(np.isinf(got), np.isinf(ref))
    assert np.array_equal(got[~np.isinf(got)], ref[~np.isinf(ref)])


def test_fp16_round_ties_to_even():
    assert oracle.fp16_round(1 + 2 ** -11) == 1.0
    assert oracle.fp16_round(1 + 3 * 2 ** -11) == 1 + 2 ** -9


def test_single_channel_row_closed_form():
    # x = v e_c: every rotated entry is v H[c, j] = +-|v|/sqrt(128), so the
    # absmax is |v|/sqrt(128), s = fp16(|v|/(127 sqrt 128)) and every code is
    # +-127 with the sign pattern of row c of the Hadamard matrix times sign(v).
    for c, v in [(0, 1.0), (5, -3.0), (77, 20.0), (127, 0.37)]:
        x = np.zeros((1, 128))
        x[0, c] = v
        codes, s = oracle.encode_rows(x)
        expect_s = float(torch.tensor(abs(v) / (127 * math.sqrt(128)), dtype=torch.float64)
                         .to(torch.float16).double())
        assert s[0] == expect_s
        signs = scipy.linalg.hadamard(128)[c] * np.sign(v)
        assert np.array_equal(codes[0], (127 * signs).astype(np.int8))


def test_outlier_spreading_lowers_error():
    # The reason for the rotation: a row with an outlier channel quantises
    # with far less error in the rotated basis than in the raw basis.
    x = RNG.standard_normal((256, 128))
    x[:, [3, 40, 99]] *= 20.0
    codes, s = oracle.encode_rows(x)
    err_rot = np.abs(oracle.unrotate(oracle.dequant(codes, s)) - x)
    s_raw = oracle.row_scales(x)
    err_raw = np.abs(oracle.dequant(oracle.quantize(x, s_raw), s_raw) - x)
    assert np.sqrt((err_rot ** 2).mean()) < 0.5 * np.sqrt((err_raw ** 2).mean())


def test_roundtrip_bound_and_code_range():
    # |c s - x'| <= s/2 for every element of every normal-range row; codes in
    # [-127, 127]; each nonzero row reaches |c| = 127 (the absmax entry).
    x = oracle.as_f64(bf16_normal((4, 300, 128), 7))
    x[0, :, 9] *= 20
    xr = oracle.rotate(x)
    codes, s = oracle.encode_rows(x)
    assert codes.dtype == np.int8
    assert codes.min() >= -127 and codes.max() <= 127
    err = np.abs(oracle.dequant(codes, s) - xr)
    assert np.all(err <= s[..., None] / 2 * (1 + 1e-12))
    assert np.all(np.abs(codes).max(axis=-1) == 127)


def test_scale_is_fp16_of_absmax_over_127():
    x = oracle.as_f64(bf16_normal((50, 128), 8))
    xr = oracle.rotate(x)
    _, s = oracle.encode_rows(x)
    a = np.abs(xr).max(axis=1)
    ref = torch.tensor(a / 127.0, dtype=torch.float64).to(torch.float16).double().numpy()
    assert np.array_equal(s, ref)


def test_code_ties_round_half_even():
    s = np.array([2.0 ** -4])
    xr = np.zeros((1, 128))
    xr[0, :6] = np.array([127, 2.5, 3.5, -2.5, -3.5, 0.5]) * s[0]
    codes = oracle.quantize(xr, s)
    assert codes[0, :6].tolist() == [127, 2, 4, -2, -4, 0]


def test_zero_tiny_and_huge_rows():
    x = np.zeros((3, 128))
    x[1, 4] = 1e-9           # absmax/127 far below the smallest fp16 subnormal
    x[2, 4] = 1e12           # absmax/127 overflows fp16: scale saturates
    codes, s = oracle.encode_rows(x)
    assert s[0] == 0 and not codes[0].any()
    assert s[1] == 0 and not codes[1].any()
    assert s[2] == 65504.0 and np.all(np.abs(codes[2]) == 127)


def test_subnormal_scale_clamps():
    # absmax/127 = 16.49 * 2^-24 lies in the fp16 subnormal range and rounds
    # down to 16 * 2^-24, so absmax/s = 127 * 16.49/16 = 130.9 and the clamp
    # must hold that code at 127 (reading: codes clamped to [-127, 127]).
    a = 127 * 16.49 * 2.0 ** -24
    xr = np.zeros((1, 128))
    xr[0, 0], xr[0, 1] = a, -a
    s = oracle.row_scales(xr)
    assert s[0] == 16 * 2.0 ** -24
    codes = oracle.quantize(xr, s)
    assert codes[0, 0] == 127 and codes[0, 1] == -127


# --------------------------------------------------------------- attention --
def brute_attention(q, k, v, scale):
    """Textbook softmax attention with Python loops and math.exp (a second,
    independent way of writing the plain definition)."""
    out = []
    for qi in q:
        scores = [scale * sum(float(a) * float(b) for a, b in zip(qi, kj)) for kj in k]
        mx = max(scores)
        w = [math.exp(t - mx) for t in scores]
        z = sum(w)
        out.append([sum(w[j] * float(v[j][c]) for j in range(len(k))) / z for c in range(len(v[0]))])
    return np.array(out)


def test_exact_path_equals_textbook_attention():
    q = oracle.as_f64(bf16_normal((1, 5, 128), 11))
    k = oracle.as_f64(bf16_normal((1, 9, 128), 12))
    v = oracle.as_f64(bf16_normal((1, 9, 128), 13))
    scale = 1 / math.sqrt(128)
    got = oracle.attend_exact(q, k, v)
    ref = brute_attention(q[0], k[0], v[0], scale)
    assert np.abs(got[0] - ref).max() <= 1e-12


def test_default_scale_is_inverse_sqrt_d():
    assert oracle.default_scale() == 1 / math.sqrt(128)


@pytest.mark.parametrize("L", [1, 2, 7, 16])
def test_blockwise_combine_equals_full_softmax(L):
    # Every kv_block partition of a tiny problem: the log-sum-exp combine of
    # per-block results equals one full softmax (brute force reference).
    q = RNG.standard_normal((3, 128)) * 2
    k = RNG.standard_normal((L, 128)) * 2
    v = RNG.standard_normal((L, 128))
    scale = 1 / math.sqrt(128)
    ref = brute_attention(q, k, v, scale)
    for kb in range(1, L + 1):
        got = oracle.attend_blockwise(q, k, v, kb, scale)
        assert np.abs(got - ref).max() <= 1e-12, kb


def test_blockwise_combine_with_dominant_late_block():
    # A later block whose max dominates (exercises the e^(M - M') rescale).
    q = np.ones((1, 128))
    k = np.zeros((6, 128))
    k[4] = 1.0
    v = np.eye(6, 128)
    scale = 1.0
    got = oracle.attend_blockwise(q, k, v, 2, scale)
    ref = brute_attention(q, k, v, scale)
    assert np.abs(got - ref).max() <= 1e-12


def test_two_key_worked_example_golden():
    # Hand-computed: q = sqrt(128) ln3 e_0, k1 = e_0, k2 = 0, v1 = 4 e_1,
    # v2 = 8 e_2, scale 1/sqrt(128): scores ln3 and 0, weights 3/4 and 1/4,
    # O = 3 e_1 + 2 e_2 (golden fixture).
    g = json.load(open(os.path.join(GOLDEN, "two_key_attention.json")))
    q = np.zeros((1, 1, 128)); q[0, 0, 0] = math.sqrt(128) * math.log(3)
    k = np.zeros((1, 2, 128)); k[0, 0, 0] = 1
    v = np.zeros((1, 2, 128)); v[0, 0, 1] = 4; v[0, 1, 2] = 8
    o = oracle.attend_exact(q, k, v)[0, 0]
    assert np.abs(o[:3] - np.array(g["o_first3"])).max() <= 1e-12
    assert np.abs(o[3:]).max() == 0


def _store_of(K, V):
    return oracle.build_store(K, V)


def test_kvi8r_zero_query_is_mean_of_dequantised_v():
    # Q = 0: uniform softmax, O = mean_j(V^'_j) H^T (closed form).
    K = bf16_normal((2, 33, 128), 21)
    V = bf16_normal((2, 33, 128), 22)
    st = _store_of(K, V)
    Q = np.zeros((2, 4, 128))
    got = oracle.attend(Q, st)
    for h in range(2):
        vd = st["v_codes"][h].astype(np.float64) * st["v_scales"][h][:, None]
        ref = vd.mean(axis=0) @ scipy.linalg.hadamard(128) / np.sqrt(128)
        assert np.abs(got[h] - ref[None]).max() <= 1e-13


def test_kvi8r_constant_v_rows():
    # Every V row equal to v: O = dequant(vH) H^T for every query, whatever Q
    # and K are (closed form).
    K = bf16_normal((1, 20, 128), 31)
    v = oracle.as_f64(bf16_normal((1, 1, 128), 32))
    V = np.repeat(v, 20, axis=1)
    st = _store_of(K, V)
    Q = bf16_normal((1, 3, 128), 33)
    got = oracle.attend(Q, st)
    c, s = oracle.encode_rows(v[0])
    ref = (c[0].astype(np.float64) * s[0]) @ scipy.linalg.hadamard(128) / np.sqrt(128)
    assert np.abs(got[0] - ref[None]).max() <= 1e-13


def test_kvi8r_unquantised_store_reduces_to_exact():
    # Replace the codes by the exact rotated values (scale 1): the kvi8r
    # arithmetic (rotate Q, attend in the rotated basis, un-rotate O) must
    # equal plain attention on the original K, V.
    Q = bf16_normal((2, 6, 128), 41)
    K = bf16_normal((2, 50, 128), 42)
    V = bf16_normal((2, 50, 128), 43)
    st = {"k_codes": oracle.rotate(K), "k_scales": np.ones((2, 50)),
          "v_codes": oracle.rotate(V), "v_scales": np.ones((2, 50))}
    got = oracle.attend(Q, st)
    ref = oracle.attend_exact(Q, K, V)
    assert np.abs(got - ref).max() <= 1e-12


def test_kvi8r_close_to_exact_on_gaussian_inputs():
    # Quality context (the pages quote rel-rms 1.3e-2 on an undefined proxy):
    # on N(0,1) inputs the kvi8r result stays within a few 1e-2 rel-rms.
    Q = bf16_normal((2, 64, 128), 51)
    K = bf16_normal((2, 256, 128), 52)
    V = bf16_normal((2, 256, 128), 53)
    st = _store_of(K, V)
    r = oracle.rel_rms(oracle.attend(Q, st), oracle.attend_exact(Q, K, V))
    assert 1e-4 < r < 3e-2


def test_attend_heads_subset_matches_full():
    Q = bf16_normal((3, 5, 128), 61)
    K = bf16_normal((3, 40, 128), 62)
    V = bf16_normal((3, 40, 128), 63)
    st = _store_of(K, V)
    full = oracle.attend(Q, st)
    part = oracle.attend(oracle.as_f64(Q)[[2, 0]], st, heads=[2, 0])
    assert np.array_equal(part, full[[2, 0]])


# ------------------------------------------------ per-32-value scales (R8) --
def test_grouped_scales_hand_example():
    # A rotated row whose 4 groups of 32 have maxima 127, 12.7, 1.27 and 0:
    # scales are fp16(1), fp16(0.1), fp16(0.01) and 0, and each group's
    # absmax entry quantises to +-127 with its own scale.
    xr = np.zeros((1, 128))
    xr[0, 5], xr[0, 40], xr[0, 70] = 127.0, -12.7, 1.27
    xr[0, 6] = 0.5
    s = oracle.group_scales(xr)
    assert s.shape == (1, 4)
    expect = torch.tensor([1.0, 0.1, 0.01], dtype=torch.float64).to(torch.float16).double().numpy()
    assert np.array_equal(s[0, :3], expect) and s[0, 3] == 0
    g = xr.reshape(1, 4, 32)
    codes = oracle.quantize(g, s).reshape(1, 128)
    assert codes[0, 5] == 127 and codes[0, 40] == -127 and codes[0, 70] == 127
    assert codes[0, 6] == 0  # 0.5 / fp16(1) = 0.5 -> ties to even -> 0
    assert not codes[0, 96:].any()


def test_grouped_roundtrip_bound_and_reach():
    x = oracle.as_f64(bf16_normal((3, 200, 128), 71))
    x[0, :, 17] *= 20
    codes, s = oracle.encode_rows_grouped(x)
    xr = oracle.rotate(x)
    assert s.shape == (3, 200, 4)
    err = np.abs(oracle.dequant(codes, s) - xr)
    assert np.all(err <= np.repeat(s, 32, axis=-1) / 2 * (1 + 1e-12))
    assert np.all(np.abs(codes.reshape(3, 200, 4, 32)).max(axis=-1) == 127)


def test_group_of_128_is_the_per_row_store():
    x = oracle.as_f64(bf16_normal((2, 50, 128), 72))
    c1, s1 = oracle.encode_rows(x)
    c2, s2 = oracle.encode_rows_grouped(x, group=128)
    assert np.array_equal(c1, c2) and np.array_equal(s1, s2[..., 0])


def test_grouped_scales_are_never_coarser():
    # each group's scale is at most the row's scale, so the error never grows
    x = oracle.as_f64(bf16_normal((1, 500, 128), 73))
    x[0, :, [3, 77]] *= 20
    _, s_row = oracle.encode_rows(x)
    cg, s_grp = oracle.encode_rows_grouped(x)
    assert np.all(s_grp <= s_row[..., None])
    cr, _ = oracle.encode_rows(x)
    xr = oracle.rotate(x)
    e_row = np.abs(oracle.dequant(cr, s_row) - xr).mean()
    e_grp = np.abs(oracle.dequant(cg, s_grp) - xr).mean()
    assert e_grp < e_row


def test_grouped_attention_closer_to_exact():
    Q = bf16_normal((2, 64, 128), 74)
    K = bf16_normal((2, 512, 128), 75)
    V = bf16_normal((2, 512, 128), 76)
    ex = oracle.attend_exact(Q, K, V)
    r_row = oracle.rel_rms(oracle.attend(Q, oracle.build_store(K, V)), ex)
    r_grp = oracle.rel_rms(oracle.attend(Q, oracle.build_store_grouped(K, V)), ex)
    assert r_grp < r_row


# ------------------------------------------------------------------ rel_rms --
def test_rel_rms_closed_forms():
    # rel_rms is the kind of relative error the kv_store row quotes for the
    # lower store rungs; pinned by values fixed without its formula
    b = oracle.as_f64(bf16_normal((3, 40, 128), 80))
    assert oracle.rel_rms(b, b) == 0.0
    assert oracle.rel_rms(np.zeros_like(b), b) == pytest.approx(1.0, rel=1e-15)
    # a uniform relative error eps gives exactly |eps|, of either sign
    for eps in (1e-3, -0.25, 2.0):
        assert oracle.rel_rms(b * (1 + eps), b) == pytest.approx(abs(eps), rel=1e-12)
    # joint scaling leaves it unchanged; it is not symmetric in its arguments
    a = b + oracle.as_f64(bf16_normal((3, 40, 128), 81)) * 0.1
    assert oracle.rel_rms(7.5 * a, 7.5 * b) == pytest.approx(oracle.rel_rms(a, b), rel=1e-12)
    assert oracle.rel_rms(2 * b, b) == pytest.approx(1.0) and oracle.rel_rms(b, 2 * b) == pytest.approx(0.5)


def test_rel_rms_hand_worked():
    # a = (1, 2), b = (1, 1): the difference is (0, 1), so the error's norm is
    # 1 against the reference's sqrt(2): 1/sqrt(2)
    assert oracle.rel_rms(np.array([1.0, 2.0]), np.array([1.0, 1.0])) == pytest.approx(2 ** -0.5, rel=1e-15)
    # a = (3, 0, 4), b = (0, 0, 5): difference (3, 0, -1), norm sqrt(10) against 5
    assert oracle.rel_rms(np.array([3.0, 0.0, 4.0]), np.array([0.0, 0.0, 5.0])) == pytest.approx(10 ** 0.5 / 5,
                                                                                                   rel=1e-15)
