"""Seeded random shapes through every attention path, each against the fp64
oracle at its stated bar: kvi8r and kvfp4 (over the GPU-built store) and the
exact store within the kvi8r bar, kvf8s within the e4m3 bound.  The draws
cover ragged query and key lengths, q_chunk values that do not divide the
query count, every kv_block granularity and softmax scales on both sides of
the default."""
import numpy as np
import pytest
import torch

import oracle
from oracle import kvfp4 as f4
from parity import compare_attention, store_to_numpy
from store_h3kv_build_gb300 import synth
from test_gpu_f8 import compare_f8_attention
from test_gpu_f8 import gpu_store_numpy as f8_store_numpy
from test_gpu_fp4 import gpu_store_numpy as fp4_store_numpy

pytestmark = pytest.mark.gpu


def _configs(n=12, seed=2026):
    rng = np.random.RandomState(seed)
    out = []
    for _ in range(n):
        heads = int(rng.randint(1, 4))
        kv_seq = int(rng.choice([1, 7, 64, 129, 383, 700, 1024, 1999, 2500]))
        q_seq = int(rng.choice([1, 5, 128, 257, 600, 1300]))
        q_chunk = int(rng.choice([1, 3, 100, 256, 1000, 4096]))
        kv_block = int(rng.choice([0, 128, 256, 640, 1024]))
        scale = float(rng.choice([0.0, 0.05, 0.2]))
        outliers = bool(rng.randint(0, 2))
        out.append((heads, q_seq, kv_seq, q_chunk, kv_block, scale, outliers))
    return out


@pytest.mark.parametrize("heads,q_seq,kv_seq,q_chunk,kv_block,scale,outliers", _configs())
def test_random_shape_every_path(cuda, heads, q_seq, kv_seq, q_chunk, kv_block, scale, outliers):
    from store_h3kv_build_gb300 import binding as b
    q, k, v = synth.make_qkv(heads, kv_seq, seed=heads * 1000 + q_seq + kv_seq, q_seq=q_seq, k_outliers=outliers)
    qd, kd, vd = q.to(cuda), k.to(cuda), v.to(cuda)
    sc = None if scale == 0.0 else scale
    what = f"H{heads} q{q_seq} kv{kv_seq} qc{q_chunk} kvb{kv_block} s{scale}"

    st = b.build_store(kd, vd)
    o = b.attend(qd, st, q_chunk=q_chunk, kv_block=kv_block, softmax_scale=scale)
    b.sync_status()
    compare_attention(o, oracle.attend(q, store_to_numpy(st), scale=sc), "kvi8r " + what)

    o = b.attend_exact(qd, kd, vd, q_chunk=q_chunk, kv_block=kv_block, softmax_scale=scale)
    b.sync_status()
    compare_attention(o, oracle.attend_exact(q, k, v, scale=sc), "exact " + what)

    st4 = b.build_store_fp4(kd, vd)
    o = b.attend_fp4(qd, st4, q_chunk=q_chunk, kv_block=kv_block, softmax_scale=scale)
    b.sync_status()
    compare_attention(o, f4.attend_kvfp4(q, fp4_store_numpy(st4), scale=sc), "kvfp4 " + what)

    if sc is None:
        # the kvf8s bound helper takes the default softmax scale
        st8 = b.build_store_f8(kd, vd)
        o = b.attend_f8(qd, st8, q_chunk=q_chunk, kv_block=kv_block)
        b.sync_status()
        compare_f8_attention(o, q, f8_store_numpy(st8), "kvf8s " + what)


def test_four_paths_on_four_streams_at_once(cuda):
    # kvi8r, exact, kvfp4 and kvf8s attention in flight together on four
    # streams, each a chain of query-chunk launches (programmatic dependent
    # launch within each stream): every output bit-identical to the same
    # call run alone
    from store_h3kv_build_gb300 import binding as b
    heads, seq, q_chunk, kvb = 3, 2500, 512, 1024
    q, k, v = synth.make_qkv(heads, seq, seed=61, k_outliers=True)
    qd, kd, vd = q.to(cuda), k.to(cuda), v.to(cuda)
    st, st4, st8 = b.build_store(kd, vd), b.build_store_fp4(kd, vd), b.build_store_f8(kd, vd)
    calls = [
        lambda s: b.attend(qd, st, q_chunk=q_chunk, kv_block=kvb, stream=s),
        lambda s: b.attend_exact(qd, kd, vd, q_chunk=q_chunk, kv_block=kvb, stream=s),
        lambda s: b.attend_fp4(qd, st4, q_chunk=q_chunk, kv_block=kvb, stream=s),
        lambda s: b.attend_f8(qd, st8, q_chunk=q_chunk, kv_block=kvb, stream=s),
    ]
    refs = [c(None) for c in calls]
    b.sync_status()
    streams = [torch.cuda.Stream() for _ in calls]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    outs = [c(s) for c, s in zip(calls, streams)]
    for s in streams:
        b.sync_status(s)
    for name, o, r in zip(("kvi8r", "exact", "kvfp4", "kvf8s"), outs, refs):
        assert torch.equal(o, r), name
