"""The GPU paths at the largest sizes the C ABI takes, each against the fp64
oracle on sampled heads or rows, or against a closed form:

  * 65535 heads (the most an attention grid holds, one grid row per head),
    three tokens each: every store build and attention path;
  * one head of 2^24 + 84 tokens, so that row offsets into the bf16 inputs
    and the stores pass 2^31 bytes: the kvi8r and kvfp4 stores on sampled
    rows (rows are independent), and attention with Q = 0, whose every output
    row is the mean of the attended V rows -- for kvi8r the dequantised
    rotated rows, rotated back -- computed here in fp64 in chunks.

The Q = 0 bound: blocks of 16384 keys, each summed on the tensor cores
(about 10^3 accumulate steps into fp32 of magnitude up to a few hundred,
truncated rather than rounded), then merged in IEEE fp32; at most about
one ulp of 512 per step and block, times 1024 blocks, over 2^24 keys: 4e-6
in the worst case, far less with signs that vary; 2e-6 is the bar.  (One
block of all 2^24 keys accumulates ~10^6 steps into sums near 4096 and
measured 7.7e-6 on the exact path.)
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import kvfp4 as f4
from parity import compare_attention, fp16_bits, oracle_store_heads, store_to_numpy
from store_h3kv_build_gb300 import synth
from test_gpu_f8 import compare_f8_attention
from test_gpu_f8 import gpu_store_numpy as f8_store_numpy
from test_gpu_fp4 import gpu_store_numpy as fp4_store_numpy

pytestmark = pytest.mark.gpu

MAX_HEADS = 65535
SAMPLE_HEADS = [0, 1, 32767, 65534]


def _b():
    from store_h3kv_build_gb300 import binding as b
    return b


def _store_rows_close(codes, scales, ref_codes, ref_scales, what):
    """kvi8r rows on a small sample: codes off by at most one, and on at most
    0.1 % of the entries (at least 2: a handful of sampled rows cannot carry
    the full-size 1e-4 bar); fp16 scales within one ulp."""
    d = np.abs(codes.cpu().numpy().astype(np.int16) - np.asarray(ref_codes).astype(np.int16))
    assert d.max(initial=0) <= 1, f"{what}: code off by {d.max()}"
    assert int((d != 0).sum()) <= max(2, int(1e-3 * d.size)), f"{what}: {int((d != 0).sum())} codes differ"
    ulp = int(np.abs(fp16_bits(scales) - fp16_bits(np.asarray(ref_scales))).max(initial=0))
    assert ulp <= 1, f"{what}: scale off by {ulp} ulp"


def test_max_heads_every_path(cuda):
    b = _b()
    hs = SAMPLE_HEADS
    q, k, v = synth.make_qkv(MAX_HEADS, 3, seed=77, q_seq=2, k_outliers=True)
    qd, kd, vd = q.to(cuda), k.to(cuda), v.to(cuda)

    st = b.build_store(kd, vd)
    o = b.attend(qd, st, q_chunk=2, kv_block=0)
    b.sync_status()
    ref = oracle_store_heads(k, v, hs)
    _store_rows_close(st.k_codes[hs], st.k_scales[hs], ref["k_codes"], ref["k_scales"], "K, 65535 heads")
    _store_rows_close(st.v_codes[hs], st.v_scales[hs], ref["v_codes"], ref["v_scales"], "V, 65535 heads")
    compare_attention(o[hs], oracle.attend(q[hs], store_to_numpy(st, hs)), "kvi8r, 65535 heads")

    o = b.attend_exact(qd, kd, vd, q_chunk=2, kv_block=0)
    b.sync_status()
    compare_attention(o[hs], oracle.attend_exact(q[hs], k[hs], v[hs]), "exact, 65535 heads")

    st4 = b.build_store_fp4(kd, vd)
    o = b.attend_fp4(qd, st4, q_chunk=2, kv_block=0)
    b.sync_status()
    # V is not rotated: its codes and scales are bit-exact (K is covered by the attention bar)
    ref4 = f4.build_store_kvfp4(k[hs], v[hs])
    assert np.array_equal(st4.v_scales[hs].cpu().numpy(), ref4["v_scales"]), "kvfp4 V scales, 65535 heads"
    assert np.array_equal(st4.v_codes[hs].cpu().numpy(), f4.pack_codes(ref4["v_codes"])), "kvfp4 V codes, 65535 heads"
    compare_attention(o[hs], f4.attend_kvfp4(q[hs], fp4_store_numpy(st4, hs)), "kvfp4, 65535 heads")

    st8 = b.build_store_f8(kd, vd)
    o = b.attend_f8(qd, st8, q_chunk=2, kv_block=0)
    b.sync_status()
    compare_f8_attention(o[hs], q[hs], f8_store_numpy(st8, hs), "kvf8s, 65535 heads")


def _mean_dequant_rows(codes, scales, chunk=1 << 18):
    """Mean over all rows of codes * scales (oracle.dequant), in fp64, chunked."""
    n = codes.shape[0]
    acc = np.zeros(codes.shape[1])
    for c0 in range(0, n, chunk):
        acc += oracle.dequant(codes[c0:c0 + chunk].cpu().numpy(), scales[c0:c0 + chunk].cpu().double().numpy()).sum(
            axis=0)
    return acc / n


def test_rows_past_2_31_bytes(cuda):
    b = _b()
    L = (1 << 24) + 84  # row offsets of the int8 codes reach 2^31 + 10752 bytes
    g = torch.Generator(device=cuda).manual_seed(78)
    k = torch.randn((1, L, 128), generator=g, device=cuda).to(torch.bfloat16)
    v = torch.randn((1, L, 128), generator=g, device=cuda).to(torch.bfloat16)
    rows = [0, 1, (1 << 24) - 1, 1 << 24, L - 2, L - 1]

    st = b.build_store(k, v)
    b.sync_status()
    ref = oracle.build_store(k[:, rows].cpu(), v[:, rows].cpu())
    _store_rows_close(st.k_codes[:, rows], st.k_scales[:, rows], ref["k_codes"], ref["k_scales"], "K rows past 2^31 B")
    _store_rows_close(st.v_codes[:, rows], st.v_scales[:, rows], ref["v_codes"], ref["v_scales"], "V rows past 2^31 B")

    # Q = 0: every score is 0, every weight 1, so each output row is the mean
    # of the attended V rows (for kvi8r: dequantised, rotated, then rotated back)
    q = torch.zeros((1, 2, 128), dtype=torch.bfloat16, device=cuda)
    o = b.attend(q, st, q_chunk=2, kv_block=16384)
    b.sync_status()
    mean = oracle.unrotate(_mean_dequant_rows(st.v_codes[0], st.v_scales[0])[None, :])[0]
    err = np.abs(o[0].cpu().double().numpy() - mean[None, :]).max()
    assert err <= 2e-6, f"kvi8r, Q = 0 over {L} keys: max abs error {err:.3e} (mean magnitude ~{np.abs(mean).mean():.1e})"

    o = b.attend_exact(q, k, v, q_chunk=2, kv_block=16384)
    b.sync_status()
    vmean = np.zeros(128)
    for c0 in range(0, L, 1 << 18):
        vmean += v[0, c0:c0 + (1 << 18)].cpu().double().numpy().sum(axis=0)
    vmean /= L
    err = np.abs(o[0].cpu().double().numpy() - vmean[None, :]).max()
    assert err <= 2e-6, f"exact, Q = 0 over {L} keys: max abs error {err:.3e}"
    del st

    st4 = b.build_store_fp4(k, v)
    b.sync_status()
    ref4 = f4.build_store_kvfp4(k[:, rows].cpu(), v[:, rows].cpu())
    assert np.array_equal(st4.v_scales[:, rows].cpu().numpy(), ref4["v_scales"]), "kvfp4 V scales past 2^31 B"
    assert np.array_equal(st4.v_codes[:, rows].cpu().numpy(), f4.pack_codes(ref4["v_codes"])), \
        "kvfp4 V codes past 2^31 B"
