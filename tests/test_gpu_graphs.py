"""The device entry points under CUDA graph capture: the store builds and the
attention paths (chains of query-chunk launches with programmatic dependent
launch) are captured once into a graph, the graph is replayed on new inputs
copied into the captured tensors, and every output must be bit-identical to
the same calls run eagerly."""
import pytest
import torch

from store_h3kv_build_gb300 import synth

pytestmark = pytest.mark.gpu


def _b():
    from store_h3kv_build_gb300 import binding as b
    return b


def test_build_and_attend_replay_from_a_graph(cuda):
    b = _b()
    heads, seq, q_chunk, kvb = 2, 1500, 512, 512
    q, k, v = synth.make_qkv(heads, seq, seed=71, k_outliers=True)
    qs, ks, vs = q.to(cuda), k.to(cuda), v.to(cuda)  # the captured (static) inputs
    st, st4, st8 = b.Store.empty(heads, seq, cuda), b.StoreFp4.empty(heads, seq, cuda), b.StoreF8.empty(heads, seq, cuda)
    outs = [torch.empty((heads, seq, 128), dtype=torch.float32, device=cuda) for _ in range(4)]

    def step(stream=None):
        b.build_store(ks, vs, out=st, stream=stream)
        b.attend(qs, st, q_chunk=q_chunk, kv_block=kvb, out=outs[0], stream=stream)
        b.attend_exact(qs, ks, vs, q_chunk=q_chunk, kv_block=kvb, out=outs[1], stream=stream)
        b.build_store_fp4(ks, vs, out=st4, stream=stream)
        b.attend_fp4(qs, st4, q_chunk=q_chunk, kv_block=kvb, out=outs[2], stream=stream)
        b.build_store_f8(ks, vs, out=st8, stream=stream)
        b.attend_f8(qs, st8, q_chunk=q_chunk, kv_block=kvb, out=outs[3], stream=stream)

    # eager warm-up on a side stream (the library's one-time set-up happens here)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(side)
    b.sync_status(side)
    torch.cuda.current_stream().wait_stream(side)

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(torch.cuda.current_stream())

    for seed in (72, 73):
        q2, k2, v2 = synth.make_qkv(heads, seq, seed=seed, k_outliers=True)
        qs.copy_(q2)
        ks.copy_(k2)
        vs.copy_(v2)
        g.replay()
        b.sync_status()
        got = [o.clone() for o in outs]
        step()  # the same calls, eagerly
        b.sync_status()
        for name, x, y in zip(("kvi8r", "exact", "kvfp4", "kvf8s"), got, outs):
            assert torch.equal(x, y), f"{name}, inputs seed {seed}"
