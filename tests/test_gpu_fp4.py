"""GPU parity of the kvfp4 store build and attention (h3kv_build_store_fp4,
h3kv_attend_fp4) against the fp64 oracle (``oracle.kvfp4``).

The store is kvfp4s of the kv_store row (H3 Streamed Blocks, Inputs table):
NVFP4 K/V -- e2m1 values with one e4m3 scale per 16 -- with K rotated into
the Hadamard basis and V not.

Bars:
  * V codes and V scales: bit-exact.  Both sides round max|v| / 6 and v / s to
    nearest even from bf16 values; such a quotient is either exact (then both
    sides see the midpoint itself) or at least 2^-8 (relative) away from any
    midpoint, far beyond fp32 rounding;
  * K scales: identical except at most 1e-3 of the blocks, each one e4m3
    step apart; K codes in the blocks whose scales agree: identical except at
    most 1e-3 of them, each on a neighbouring e2m1 value (the GPU rotates in
    fp32, the oracle in fp64);
  * attention: the kvi8r bar (max abs 2e-2, mean abs 2e-3), both against the
    oracle's attention over the GPU-built store (the store's values are exact
    in fp16, so only the fp16 query and fp16 softmax weights round) and end
    to end against the oracle's attention over its own store (tiny, 24 x
    32768 on four heads, 32 x 217088 on eight heads).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import kvf8s as f8
from oracle import kvfp4 as f4
from store_h3kv_build_gb300 import synth
from parity import compare_attention

pytestmark = pytest.mark.gpu

K_MISMATCH_FRAC = 1e-3


def _b():
    from store_h3kv_build_gb300 import binding as b
    return b


def _build(K, V):
    b = _b()
    st = b.build_store_fp4(K, V)
    b.sync_status()
    return st


def gpu_store_numpy(st, heads=None):
    """GPU kvfp4 store -> the oracle's dict layout (codes unpacked)."""
    idx = list(range(st.heads)) if heads is None else list(heads)
    return {
        "k_codes": f4.unpack_codes(st.k_codes[idx].cpu().numpy()),
        "k_scales": st.k_scales[idx].cpu().numpy(),
        "v_codes": f4.unpack_codes(st.v_codes[idx].cpu().numpy()),
        "v_scales": st.v_scales[idx].cpu().numpy(),
    }


def check_store(st, K, V, heads=None, what=""):
    heads = list(range(K.shape[0])) if heads is None else heads
    g_packed_v = st.v_codes[heads].cpu().numpy()
    g = gpu_store_numpy(st, heads)
    ref = f4.build_store_kvfp4(K[heads], V[heads])
    # V: bit-exact, packed bytes included
    assert np.array_equal(g["v_scales"], ref["v_scales"]), f"{what}: V scales"
    assert np.array_equal(g_packed_v, f4.pack_codes(ref["v_codes"])), f"{what}: V codes"
    # K scales: rare neighbours
    gs, rs = g["k_scales"].astype(np.int16), ref["k_scales"].astype(np.int16)
    sbad = gs != rs
    assert float(sbad.mean()) <= K_MISMATCH_FRAC, f"{what}: {sbad.mean():.2e} of K scales differ"
    assert np.all(np.abs(gs[sbad] - rs[sbad]) == 1), f"{what}: K scale off by more than one step"
    # K codes where the scales agree
    same = np.repeat(~sbad, 16, axis=-1)
    gc, rc = g["k_codes"][same].astype(np.int16), ref["k_codes"][same].astype(np.int16)
    bad = gc != rc
    assert float(bad.mean()) <= K_MISMATCH_FRAC, f"{what}: {bad.mean():.2e} of K codes differ"
    if bad.any():
        gv, rv = f4.e2m1_decode(gc[bad]), f4.e2m1_decode(rc[bad])
        assert np.all(np.abs((gc[bad] & 7) - (rc[bad] & 7)) <= 1), f"{what}: K code off by more than one step"
        assert np.all((np.sign(gv) == np.sign(rv)) | (gv == 0) | (rv == 0)), f"{what}: sign flip"
    return float(bad.mean()), float(sbad.mean())


def compare_fp4_attention(out, Q, store, what="", scale=None):
    """GPU output vs the oracle's attention over the same (GPU-built) store."""
    ref = f4.attend_kvfp4(Q, store, scale=scale)
    return compare_attention(out, ref, what)


def oracle_store_heads(K, V, heads):
    """The oracle's own kvfp4 store of the listed heads (stacked in order)."""
    parts = [f4.build_store_kvfp4(K[h:h + 1], V[h:h + 1]) for h in heads]
    return {k: np.concatenate([p[k] for p in parts]) for k in parts[0]}


# ------------------------------------------------------------------ store --
def test_store_fp4_tiny(cuda):
    _, k, v = synth.make_qkv(1, 1024, seed=0)
    st = _build(k.to(cuda), v.to(cuda))
    check_store(st, k, v, what="tiny")


@pytest.mark.parametrize("heads,seq", [(3, 1000), (1, 1), (2, 129), (5, 77), (2, 64), (1, 8192)])
def test_store_fp4_ragged(cuda, heads, seq):
    _, k, v = synth.make_qkv(heads, seq, seed=4, k_outliers=True)
    st = _build(k.to(cuda), v.to(cuda))
    check_store(st, k, v, what=f"{heads}x{seq}")


def test_store_fp4_special_rows(cuda):
    # V rows built to hit the encoder's edge cases, every one exact in bf16:
    #   row 0: block maximum 6 (scale 1) with the seven e2m1 midpoints
    #          0.25 .. 5 (each a tie, to the even code) and their negatives;
    #   row 1: midpoints under a scale of 1.125 (0x39), whose reciprocal is
    #          not exact in fp32;
    #   row 2: -0.0 everywhere but one value (zeros keep their sign);
    #   row 3: values past 448 * 6 (the scale saturates at 448, codes at 6);
    #   row 4: a block below half the smallest scale (scale 0, codes 0);
    #   row 5: all zero.  K: a zero row and a one-channel row.
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    v = torch.zeros((1, 6, 128), dtype=torch.float32)
    for blk in range(8):
        v[0, 0, blk * 16] = 6.0
        v[0, 0, blk * 16 + 1:blk * 16 + 8] = torch.tensor(mids)
        v[0, 0, blk * 16 + 8:blk * 16 + 15] = -torch.tensor(mids)
        v[0, 1, blk * 16] = 6.0 * 1.125
        v[0, 1, blk * 16 + 1:blk * 16 + 8] = torch.tensor(mids) * 1.125
    v[0, 2] = -0.0
    v[0, 2, 3] = 1.0
    v[0, 3] = 3000.0
    v[0, 3, ::2] = -5000.0
    v[0, 4, :16] = 0.005
    v[0, 4, 16:] = 1.0
    vb = v.to(torch.bfloat16)
    assert torch.equal(vb.float()[0, :3], v[0, :3])  # the tie rows are exact in bf16
    k = synth.normal_f32((1, 6, 128), 30)
    k[0, 0] = 0.0
    k[0, 1] = 0.0
    k[0, 1, 37] = 3.0
    kb = k.to(torch.bfloat16)
    st = _build(kb.to(cuda), vb.to(cuda))
    check_store(st, kb, vb, what="special")
    g = gpu_store_numpy(st)
    # the ties went to the even codes: 0.25 -> 0, 0.75 -> 1, 1.25 -> 1, 1.75 -> 2, 2.5 -> 2, 3.5 -> 4, 5 -> 4
    assert np.array_equal(f4.e2m1_decode(g["v_codes"][0, 0, 1:8]), [0, 1, 1, 2, 2, 4, 4])
    # -0 keeps its sign where the block has a scale; blocks of zeros have none
    assert np.all(g["v_codes"][0, 2, [0, 1, 2] + list(range(4, 16))] == 8) and g["v_codes"][0, 2, 3] != 8
    assert not g["v_codes"][0, 2, 16:].any() and not g["v_scales"][0, 2, 1:].any()
    assert np.all(g["v_scales"][0, 3] == 0x7E) and np.all(g["v_codes"][0, 3] & 7 == 7)
    assert g["v_scales"][0, 4, 0] == 0 and not g["v_codes"][0, 4, :16].any()
    assert not g["v_codes"][0, 5].any() and not g["v_scales"][0, 5].any()
    assert not g["k_codes"][0, 0].any() and not g["k_scales"][0, 0].any()


def test_store_fp4_deterministic(cuda):
    _, k, v = synth.make_qkv(4, 5000, seed=12, k_outliers=True, device=cuda)
    a, b2 = _build(k, v), _build(k, v)
    for name in ("k_codes", "v_codes", "k_scales", "v_scales"):
        assert torch.equal(getattr(a, name), getattr(b2, name)), name


def test_store_fp4_h24_l32768_outlier(cuda):
    w = synth.WORKLOADS["h24_l32768_outlier"]
    _, k, v = synth.make_qkv(w["heads"], w["seq"], seed=0, k_outliers=True)
    st = _build(k.to(cuda), v.to(cuda))
    check_store(st, k, v, heads=[0, 7, 23], what="h24 l32768")


# -------------------------------------------------------------- attention --
@pytest.mark.parametrize("q_chunk,kv_block", [(256, 512), (1024, 0), (100, 128), (1, 256)])
def test_attend_fp4_tiny(cuda, q_chunk, kv_block):
    b = _b()
    q, k, v = synth.make_qkv(1, 1024, seed=0)
    st = _build(k.to(cuda), v.to(cuda))
    out = b.attend_fp4(q.to(cuda), st, q_chunk=q_chunk, kv_block=kv_block)
    b.sync_status()
    compare_fp4_attention(out, q, gpu_store_numpy(st), f"tiny q_chunk={q_chunk} kv_block={kv_block}")


@pytest.mark.parametrize("heads,q_seq,kv_seq,q_chunk,kv_block",
                         [(2, 1000, 1337, 300, 512), (1, 1, 1, 1, 0), (3, 129, 5, 64, 128),
                          (1, 700, 4000, 700, 1024), (2, 257, 300, 257, 0), (1, 300, 65, 128, 0)])
def test_attend_fp4_ragged(cuda, heads, q_seq, kv_seq, q_chunk, kv_block):
    b = _b()
    q, k, v = synth.make_qkv(heads, kv_seq, seed=7, q_seq=q_seq, k_outliers=True)
    st = _build(k.to(cuda), v.to(cuda))
    out = b.attend_fp4(q.to(cuda), st, q_chunk=q_chunk, kv_block=kv_block)
    b.sync_status()
    compare_fp4_attention(out, q, gpu_store_numpy(st), f"{heads}x{q_seq}x{kv_seq}")


def test_attend_fp4_against_oracle_store(cuda):
    # end to end: GPU store + GPU attention against the oracle's own store
    b = _b()
    q, k, v = synth.make_qkv(2, 3000, seed=5, k_outliers=True)
    st = _build(k.to(cuda), v.to(cuda))
    out = b.attend_fp4(q.to(cuda), st, q_chunk=1024, kv_block=1024)
    b.sync_status()
    compare_fp4_attention(out, q, f4.build_store_kvfp4(k, v), "against the oracle store")


def test_attend_fp4_end_to_end_tiny(cuda):
    b = _b()
    q, k, v = synth.make_qkv(1, 1024, seed=0)
    st = _build(k.to(cuda), v.to(cuda))
    out = b.attend_fp4(q.to(cuda), st, q_chunk=256, kv_block=512)
    b.sync_status()
    mx, mean = compare_fp4_attention(out, q, f4.build_store_kvfp4(k, v), "tiny, oracle store")
    print(f"kvfp4 end to end tiny: max abs {mx:.3e} mean abs {mean:.3e}")


def test_attend_fp4_end_to_end_h24_l32768_outlier(cuda):
    # end to end on the outlier workload in its launch configuration: four
    # heads, 256 sampled query rows each, against the oracle's store of those
    # heads over all 32768 keys
    b = _b()
    w = synth.WORKLOADS["h24_l32768_outlier"]
    q, k, v = synth.make_qkv(w["heads"], w["seq"], seed=0, k_outliers=True)
    st = _build(k.to(cuda), v.to(cuda))
    out = b.attend_fp4(q.to(cuda), st, q_chunk=w["q_chunk"], kv_block=w["kv_block"])
    b.sync_status()
    heads = [0, 7, 13, 23]
    rows = torch.randperm(w["seq"], generator=torch.Generator().manual_seed(2))[:256].sort().values
    mx, mean = compare_fp4_attention(out[heads][:, rows.to(cuda)], q[heads][:, rows],
                                     oracle_store_heads(k, v, heads), "h24 l32768 outlier, oracle store")
    print(f"kvfp4 end to end h24 l32768: max abs {mx:.3e} mean abs {mean:.3e}")


def test_attend_fp4_q_chunk_invariance(cuda):
    b = _b()
    q, k, v = synth.make_qkv(2, 3000, seed=3, k_outliers=True, device=cuda)
    st = _build(k, v)
    outs = [b.attend_fp4(q, st, q_chunk=c, kv_block=1024) for c in (3000, 1024, 700, 256)]
    b.sync_status()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


def test_attend_fp4_zero_queries_average_v(cuda):
    # q = 0: every weight is exactly 1, so O is the mean of the dequantised V
    # rows (exact fp16 values), up to fp32 accumulation
    b = _b()
    _, k, v = synth.make_qkv(1, 777, seed=8)
    q = torch.zeros((1, 40, 128), dtype=torch.bfloat16)
    st = _build(k.to(cuda), v.to(cuda))
    out = b.attend_fp4(q.to(cuda), st)
    b.sync_status()
    g = gpu_store_numpy(st)
    ref = f4.dequant(g["v_codes"][0], g["v_scales"][0]).mean(axis=0)
    assert np.max(np.abs(out[0].cpu().double().numpy() - ref[None, :])) < 1e-4


@pytest.mark.parametrize("softmax_scale", [0.02, 0.3])
def test_attend_fp4_softmax_scale(cuda, softmax_scale):
    b = _b()
    q, k, v = synth.make_qkv(2, 1500, seed=21, k_outliers=True)
    st = _build(k.to(cuda), v.to(cuda))
    out = b.attend_fp4(q.to(cuda), st, q_chunk=512, kv_block=512, softmax_scale=softmax_scale)
    b.sync_status()
    compare_fp4_attention(out, q, gpu_store_numpy(st), f"softmax_scale={softmax_scale}", scale=softmax_scale)


def test_attend_fp4_h24_l32768_sampled(cuda):
    # the q_chunk=16384, kv_block=16384 launch configuration on the outlier
    # workload; sampled rows of two heads against the full key set
    b = _b()
    w = synth.WORKLOADS["h24_l32768_outlier"]
    q, k, v = synth.make_qkv(w["heads"], w["seq"], seed=0, k_outliers=True, device=cuda)
    st = _build(k, v)
    out = b.attend_fp4(q, st, q_chunk=16384, kv_block=16384)
    b.sync_status()
    heads = [0, 11]
    rows = torch.arange(0, w["seq"], 97)
    compare_fp4_attention(out[heads][:, rows], q[heads][:, rows].cpu(), gpu_store_numpy(st, heads),
                          "h24 l32768 sampled")


@pytest.mark.slow
def test_fp4_full_size_h32_l217088(cuda):
    # the full-size workload in the launch configuration the bench times:
    # store heads 0 and 31 in full; attention on 64 sampled rows x 8 heads,
    # over the GPU store and end to end over the oracle's own store
    b = _b()
    w = synth.WORKLOADS["h32_l217088_outlier"]
    q, k, v = synth.make_qkv(w["heads"], w["seq"], seed=0, k_outliers=True, device=cuda)
    st = _build(k, v)
    kc, vc = k.cpu(), v.cpu()
    for h in (0, 31):
        check_store(st, kc, vc, heads=[h], what=f"h{h}")
    out = b.attend_fp4(q, st, q_chunk=16384, kv_block=16384)
    b.sync_status()
    heads = [0, 5, 9, 13, 17, 21, 26, 31]
    rows = torch.linspace(0, w["seq"] - 1, 64).long()
    qs = q[heads][:, rows].cpu()
    compare_fp4_attention(out[heads][:, rows], qs, gpu_store_numpy(st, heads), "h32 l217088 sampled")
    # end to end against the oracle's own store of the eight heads
    mx, mean = compare_fp4_attention(out[heads][:, rows], qs, oracle_store_heads(kc, vc, heads),
                                     "h32 l217088, oracle store")
    print(f"kvfp4 end to end h32 l217088: max abs {mx:.3e} mean abs {mean:.3e}")


def test_attend_fp4_calls_on_one_output_stay_in_stream_order(cuda):
    # chained launches inside a call may overlap, but each call's first
    # launch waits for the previous call on the same output
    b = _b()
    q, k, v = synth.make_qkv(2, 2500, seed=42, k_outliers=True, device=cuda)
    st1 = b.build_store_fp4(k, v)
    st2 = b.build_store_fp4(v, k)
    ref2 = b.attend_fp4(q, st2, q_chunk=2500, kv_block=1024)
    o = torch.empty_like(ref2)
    for _ in range(3):
        b.attend_fp4(q, st1, q_chunk=256, kv_block=1024, out=o)
        b.attend_fp4(q, st2, q_chunk=600, kv_block=1024, out=o)
    b.sync_status()
    assert torch.equal(o, ref2)


def test_fp4_scale_codes_are_e4m3(cuda):
    # every stored scale decodes to a finite, non-negative e4m3 value
    _, k, v = synth.make_qkv(2, 500, seed=9, k_outliers=True)
    st = _build(k.to(cuda), v.to(cuda))
    for s in (st.k_scales, st.v_scales):
        d = f8.e4m3_decode(s.cpu().numpy())
        assert np.isfinite(d).all() and (d >= 0).all()


def test_attend_fp4_query_outliers_and_zero_keys(cuda):
    # query rows 100x larger than the rest (a much sharper softmax), and a
    # second head whose keys are all zero: every score is 0, so the output
    # is the mean of the dequantised V rows.  With scores of order 100 the
    # kernel's fp16 query (its stated precision step, 2^-11 relative) moves
    # logits by tenths, so the reference takes the rotated query rounded to
    # fp16 as well; the rest (fp16 weights, fp32 sums) stays within the bar
    b = _b()
    q, k, v = synth.make_qkv(2, 900, seed=22)
    q = q.float()
    q[:, ::7] *= 100
    q = q.to(torch.bfloat16)
    k = k.clone()
    k[1] = 0
    st = _build(k.to(cuda), v.to(cuda))
    out = b.attend_fp4(q.to(cuda), st, q_chunk=300, kv_block=256)
    b.sync_status()
    g = gpu_store_numpy(st)
    assert not g["k_scales"][1].any()
    q16 = oracle.fp16_round(oracle.rotate(q))
    ref = np.stack([oracle.softmax_attention(q16[h], f4.dequant(g["k_codes"][h], g["k_scales"][h]),
                                             f4.dequant(g["v_codes"][h], g["v_scales"][h]), 1 / np.sqrt(128))
                    for h in range(2)])
    compare_attention(out, ref, "q outliers / zero keys")
    mean_v = f4.dequant(g["v_codes"][1], g["v_scales"][1]).mean(axis=0)
    assert np.max(np.abs(out[1].cpu().double().numpy() - mean_v[None, :])) < 1e-4


def test_attend_fp4_every_kv_block(cuda):
    # the log-sum-exp combine over every kv_block from one tile to one block
    b = _b()
    q, k, v = synth.make_qkv(1, 1000, seed=24, q_seq=300, k_outliers=True)
    st = _build(k.to(cuda), v.to(cuda))
    g = gpu_store_numpy(st)
    for kvb in (128, 256, 384, 512, 1024, 0):
        out = b.attend_fp4(q.to(cuda), st, q_chunk=128, kv_block=kvb)
        b.sync_status()
        compare_fp4_attention(out, q, g, f"kv_block={kvb}")


def test_store_fp4_code_buffers_16_byte_aligned(cuda):
    # 16- but not 32-byte aligned code buffers take the 16-byte store path
    b = _b()
    heads, seq = 2, 999
    _, k, v = synth.make_qkv(heads, seq, seed=43, k_outliers=True, device=cuda)
    ref = _build(k, v)
    n = heads * seq * 64
    kbuf = torch.empty(n + 32, dtype=torch.uint8, device=cuda)
    vbuf = torch.empty(n + 32, dtype=torch.uint8, device=cuda)
    kc, vc = kbuf[16:16 + n].view(heads, seq, 64), vbuf[16:16 + n].view(heads, seq, 64)
    assert kc.data_ptr() % 32 == 16
    odd = b.StoreFp4(kc, vc, torch.empty_like(ref.k_scales), torch.empty_like(ref.v_scales))
    b.build_store_fp4(k, v, out=odd)
    b.sync_status()
    for name in ("k_codes", "v_codes", "k_scales", "v_scales"):
        assert torch.equal(getattr(odd, name), getattr(ref, name)), name
