"""GPU parity of h3kv_attend (kvi8r) and h3kv_attend_exact against the oracle.

kvi8r attention (kv_store row of the H3 Streamed Blocks Inputs table): rotate
the query chunk, attend over the dequantised rotated store blockwise with a
log-sum-exp combine over kv_block, un-rotate once.  The q_chunk row states the
result is exact at any q_chunk: the GPU output must be bit-identical across
q_chunk values.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import compare_attention, oracle_store_heads, store_to_numpy
from store_h3kv_build_gb300 import synth

pytestmark = pytest.mark.gpu


def _b():
    from store_h3kv_build_gb300 import binding as b
    return b


def _kvi8r(Q, K, V, q_chunk, kv_block):
    b = _b()
    st = b.build_store(K, V)
    out = b.attend(Q, st, q_chunk=q_chunk, kv_block=kv_block)
    b.sync_status()
    return out, st


def _exact(Q, K, V, q_chunk, kv_block):
    b = _b()
    out = b.attend_exact(Q, K, V, q_chunk=q_chunk, kv_block=kv_block)
    b.sync_status()
    return out


# ------------------------------------------------------------------ kvi8r --
@pytest.mark.parametrize("q_chunk,kv_block", [(256, 512), (1024, 0), (100, 128), (1, 256)])
def test_kvi8r_tiny(cuda, q_chunk, kv_block):
    w = synth.WORKLOADS["tiny_1x1024"]
    q, k, v = synth.make_qkv(w["heads"], w["seq"], seed=0)
    out, st = _kvi8r(q.to(cuda), k.to(cuda), v.to(cuda), q_chunk, kv_block)
    ref = oracle.attend(q, oracle.build_store(k, v))
    compare_attention(out, ref, f"tiny q_chunk={q_chunk} kv_block={kv_block}")
    # attention error alone: the oracle's attention over the GPU-built store
    ref_gpu_store = oracle.attend(q, store_to_numpy(st))
    compare_attention(out, ref_gpu_store, "tiny on gpu store")


@pytest.mark.parametrize("heads,q_seq,kv_seq,q_chunk,kv_block",
                         [(2, 1000, 1337, 300, 512), (1, 1, 1, 1, 0), (3, 129, 5, 64, 128),
                          (1, 700, 4000, 700, 1024), (2, 257, 300, 257, 0)])
def test_kvi8r_ragged(cuda, heads, q_seq, kv_seq, q_chunk, kv_block):
    q, k, v = synth.make_qkv(heads, kv_seq, seed=7, q_seq=q_seq, k_outliers=True)
    out, st = _kvi8r(q.to(cuda), k.to(cuda), v.to(cuda), q_chunk, kv_block)
    ref = oracle.attend(q, oracle.build_store(k, v))
    compare_attention(out, ref, f"{heads}x{q_seq}x{kv_seq}")


def test_kvi8r_bit_identical_across_q_chunk_small(cuda):
    q, k, v = synth.make_qkv(3, 3000, seed=11)
    q, k, v = q.to(cuda), k.to(cuda), v.to(cuda)
    b = _b()
    st = b.build_store(k, v)
    outs = [b.attend(q, st, q_chunk=c, kv_block=1024) for c in (3000, 1, 7, 128, 300, 1999)]
    b.sync_status()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


def test_kvi8r_h8_l16384_sampled(cuda):
    w = synth.WORKLOADS["h8_l16384"]
    q, k, v = synth.make_qkv(w["heads"], w["seq"], seed=0)
    out, st = _kvi8r(q.to(cuda), k.to(cuda), v.to(cuda), w["q_chunk"], w["kv_block"])
    rows = torch.randperm(w["seq"], generator=torch.Generator().manual_seed(1))[:256].sort().values
    heads = list(range(w["heads"]))
    ref_store = oracle_store_heads(k, v, heads)
    ref = oracle.attend(q[:, rows], ref_store)
    compare_attention(out[:, rows.to(cuda)], ref, "h8 l16384")


def test_kvi8r_outlier_h24_l32768_sampled(cuda):
    w = synth.WORKLOADS["h24_l32768_outlier"]
    q, k, v = synth.make_qkv(w["heads"], w["seq"], seed=0, k_outliers=True)
    out, st = _kvi8r(q.to(cuda), k.to(cuda), v.to(cuda), w["q_chunk"], w["kv_block"])
    heads = [0, 7, 13, 23]
    rows = torch.randperm(w["seq"], generator=torch.Generator().manual_seed(2))[:256].sort().values
    ref = oracle.attend(q[heads][:, rows], oracle_store_heads(k, v, heads), heads=list(range(len(heads))))
    compare_attention(out[heads][:, rows.to(cuda)], ref, "h24 l32768 outlier")


@pytest.mark.slow
def test_kvi8r_full_size_h32_l217088_sampled(cuda):
    w = synth.WORKLOADS["h32_l217088_outlier"]
    q, k, v = synth.make_qkv(w["heads"], w["seq"], seed=0, k_outliers=True, device=cuda)
    out, st = _kvi8r(q, k, v, w["q_chunk"], w["kv_block"])
    heads = [0, 5, 9, 14, 18, 22, 27, 31]
    rows = torch.randperm(w["seq"], generator=torch.Generator().manual_seed(3))[:64].sort().values
    kc, vc = k[heads].cpu(), v[heads].cpu()
    ref_store = oracle_store_heads(kc, vc, list(range(len(heads))))
    ref = oracle.attend(q[heads][:, rows.to(cuda)].cpu(), ref_store)
    compare_attention(out[heads][:, rows.to(cuda)], ref, "h32 l217088")


@pytest.mark.slow
def test_kvi8r_sweep_h32_l65536_bit_identical(cuda):
    w = synth.WORKLOADS["h32_l65536_sweep"]
    q, k, v = synth.make_qkv(w["heads"], w["seq"], seed=0, device=cuda)
    b = _b()
    st = b.build_store(k, v)
    rows = torch.randperm(w["seq"], generator=torch.Generator().manual_seed(4))[:32].sort().values.to(cuda)
    heads = [1, 30]
    ref = oracle.attend(q[heads][:, rows].cpu(), oracle_store_heads(k[heads].cpu(), v[heads].cpu(), [0, 1]))
    for kv_block in (4096, 16384):
        base = b.attend(q, st, q_chunk=65536, kv_block=kv_block)
        for qc in (1024, 4096, 16384):
            o = b.attend(q, st, q_chunk=qc, kv_block=kv_block)
            b.sync_status()
            assert torch.equal(o, base), (qc, kv_block)
            del o
        compare_attention(base[heads][:, rows], ref, f"sweep kv_block={kv_block}")
        del base


def test_launch_orders_bit_identical(cuda):
    # 131072 keys: 4500-row (18 CTAs) and 4096-row (16 CTAs) chunks launch head
    # by head, 3840-row chunks (15 CTAs) one launch per chunk over all heads;
    # a row's arithmetic is the same in every launch, on all four paths
    H, L, QS = 3, 131072, 4500
    b = _b()
    n = b.h3kv_attend_launch_count
    assert (n(QS, L, H, 4500), n(QS, L, H, 4096), n(QS, L, H, 3840)) == (3, 6, 2)
    q, k, v = synth.make_qkv(H, L, seed=13, q_seq=QS, k_outliers=True, device=cuda)
    st, st8, st4 = b.build_store(k, v), b.build_store_f8(k, v), b.build_store_fp4(k, v)
    calls = {
        "kvi8r": lambda c: b.attend(q, st, q_chunk=c, kv_block=16384),
        "exact": lambda c: b.attend_exact(q, k, v, q_chunk=c, kv_block=16384),
        "kvf8s": lambda c: b.attend_f8(q, st8, q_chunk=c, kv_block=16384),
        "kvfp4": lambda c: b.attend_fp4(q, st4, q_chunk=c, kv_block=16384),
    }
    for name, call in calls.items():
        outs = [call(c) for c in (4500, 4096, 3840)]
        b.sync_status()
        for o in outs[1:]:
            assert torch.equal(o, outs[0]), name
    # and the head-major kvi8r result against the oracle on sampled rows of one head
    rows = torch.randperm(QS, generator=torch.Generator().manual_seed(5))[:16].sort().values.to(cuda)
    out = b.attend(q, st, q_chunk=4096, kv_block=16384)
    b.sync_status()
    ref = oracle.attend(q[[1]][:, rows].cpu(), oracle_store_heads(k[[1]].cpu(), v[[1]].cpu(), [0]))
    compare_attention(out[[1]][:, rows], ref, "head-major 3x4500x131072")


# ------------------------------------------------------------------ exact --
@pytest.mark.parametrize("q_chunk,kv_block", [(256, 0), (1024, 512), (1, 128)])
def test_exact_tiny(cuda, q_chunk, kv_block):
    q, k, v = synth.make_qkv(1, 1024, seed=0)
    out = _exact(q.to(cuda), k.to(cuda), v.to(cuda), q_chunk, kv_block)
    compare_attention(out, oracle.attend_exact(q, k, v), f"exact tiny {q_chunk} {kv_block}")


@pytest.mark.parametrize("heads,q_seq,kv_seq,q_chunk,kv_block",
                         [(2, 1000, 1337, 300, 512), (1, 1, 1, 1, 0), (3, 129, 5, 64, 0)])
def test_exact_ragged(cuda, heads, q_seq, kv_seq, q_chunk, kv_block):
    q, k, v = synth.make_qkv(heads, kv_seq, seed=8, q_seq=q_seq)
    out = _exact(q.to(cuda), k.to(cuda), v.to(cuda), q_chunk, kv_block)
    compare_attention(out, oracle.attend_exact(q, k, v), f"exact {heads}x{q_seq}x{kv_seq}")


def test_exact_bit_identical_across_q_chunk(cuda):
    q, k, v = synth.make_qkv(2, 2500, seed=12)
    q, k, v = q.to(cuda), k.to(cuda), v.to(cuda)
    b = _b()
    outs = [b.attend_exact(q, k, v, q_chunk=c, kv_block=0) for c in (2500, 1, 256, 999)]
    b.sync_status()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


def test_exact_h8_l16384_sampled(cuda):
    w = synth.WORKLOADS["h8_l16384"]
    q, k, v = synth.make_qkv(w["heads"], w["seq"], seed=0)
    out = _exact(q.to(cuda), k.to(cuda), v.to(cuda), w["q_chunk"], 0)
    rows = torch.randperm(w["seq"], generator=torch.Generator().manual_seed(5))[:256].sort().values
    ref = oracle.attend_exact(q[:, rows], k, v)
    compare_attention(out[:, rows.to(cuda)], ref, "exact h8 l16384")


def test_kvi8r_close_to_exact(cuda):
    # the pages' quality number is a rel-rms against the exact path on an
    # undefined proxy (parity unpinned); here: both GPU paths on N(0,1) inputs
    q, k, v = synth.make_qkv(2, 4096, seed=13, k_outliers=True)
    q, k, v = q.to(cuda), k.to(cuda), v.to(cuda)
    o1, _ = _kvi8r(q, k, v, 4096, 0)
    o2 = _exact(q, k, v, 4096, 0)
    assert oracle.rel_rms(o1.cpu(), o2.cpu()) < 5e-2


def test_calls_on_one_output_stay_in_stream_order(cuda):
    # Launches 2..n of one call overlap the previous launch's tail; the first
    # launch of every call must still wait for everything before it.  Calls
    # that write the same O back to back (different stores, q_chunks and
    # paths) must leave exactly the last call's result.
    b = _b()
    q, k, v = synth.make_qkv(2, 3000, seed=41, k_outliers=True, device=cuda)
    st1 = b.build_store(k, v)
    st2 = b.build_store(v, k)
    ref1 = b.attend(q, st1, q_chunk=3000, kv_block=1024)
    ref2 = b.attend(q, st2, q_chunk=3000, kv_block=1024)
    ref_x = b.attend_exact(q, k, v, q_chunk=3000, kv_block=0)
    o = torch.empty_like(ref1)
    for _ in range(3):
        b.attend(q, st1, q_chunk=256, kv_block=1024, out=o)
        b.attend(q, st2, q_chunk=700, kv_block=1024, out=o)
    b.sync_status()
    assert torch.equal(o, ref2)
    b.attend(q, st2, q_chunk=300, kv_block=1024, out=o)
    b.attend_exact(q, k, v, q_chunk=256, kv_block=0, out=o)
    b.sync_status()
    assert torch.equal(o, ref_x)
    b.attend_exact(q, k, v, q_chunk=512, kv_block=0, out=o)
    b.attend(q, st1, q_chunk=1000, kv_block=1024, out=o)
    b.sync_status()
    assert torch.equal(o, ref1)
