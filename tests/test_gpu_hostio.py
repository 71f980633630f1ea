"""h3kv_attend_hostio: kvi8r attention with Q and O in pinned host memory,
streamed through HBM one query chunk at a time (the q_chunk input bounds the
device transient), with the copies of other chunks overlapping the attention
of the current one.  Every chunk runs the same kernel with the same per-row
arithmetic as h3kv_attend, so the outputs must be bit-identical.  Launches
after the first wait inside the kernel for their buffer's ready word; the
cases include many chunks (20, and 1100 one-row chunks, more than the ready
values before they repeat)."""
import pytest
import torch

from store_h3kv_build_gb300 import synth

pytestmark = pytest.mark.gpu


def _b():
    from store_h3kv_build_gb300 import binding as b
    return b


@pytest.mark.parametrize("heads,q_seq,kv_seq,q_chunk,kv_block",
                         [(1, 1024, 1024, 256, 512), (2, 1000, 1337, 300, 512), (3, 700, 900, 4096, 0),
                          (1, 5, 300, 1, 128), (3, 4096, 2000, 1000, 1024), (2, 4100, 513, 2048, 256),
                          (2, 5000, 2000, 256, 512), (1, 1100, 300, 1, 128), (2, 3000, 700, 2048, 256),
                          # device attention launches these head by head (131072 keys, 16 CTAs per chunk)
                          (2, 4500, 131072, 4096, 16384)])
def test_hostio_bit_identical_to_device_attend(cuda, heads, q_seq, kv_seq, q_chunk, kv_block):
    b = _b()
    q, k, v = synth.make_qkv(heads, kv_seq, seed=31, q_seq=q_seq, k_outliers=True)
    st = b.build_store(k.to(cuda), v.to(cuda))
    ref = b.attend(q.to(cuda), st, q_chunk=q_chunk, kv_block=kv_block)
    hq = q.contiguous().pin_memory()
    out = b.attend_hostio(hq, st, q_chunk=q_chunk, kv_block=kv_block)
    b.sync_status()
    assert out.is_pinned() and out.device.type == "cpu"
    assert torch.equal(out, ref.cpu())


def test_hostio_reuses_scratch_and_orders_on_stream(cuda):
    # two calls on a side stream sharing one scratch buffer, then a device
    # read of the second output: every copy is ordered on the stream
    b = _b()
    q, k, v = synth.make_qkv(2, 2048, seed=32)
    st = b.build_store(k.to(cuda), v.to(cuda))
    ref = b.attend(q.to(cuda), st, q_chunk=512, kv_block=1024).cpu()
    hq = q.contiguous().pin_memory()
    scratch = torch.empty(int(b.h3kv_hostio_scratch_bytes(2, 512)), dtype=torch.uint8, device=cuda)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        o1 = b.attend_hostio(hq, st, q_chunk=512, kv_block=1024, scratch=scratch, stream=side)
        o2 = b.attend_hostio(hq, st, q_chunk=512, kv_block=1024, scratch=scratch, stream=side)
    b.sync_status(side)
    assert torch.equal(o1, ref) and torch.equal(o2, ref)


def test_hostio_calls_on_two_streams_at_once(cuda):
    # two calls in flight together, each with its own scratch (the pinned
    # value table behind the ready words is shared and read-only), many
    # chunks each: both outputs bit-identical to device attention
    b = _b()
    heads, q_seq, kv_seq, q_chunk = 2, 3000, 1500, 256
    q1, k, v = synth.make_qkv(heads, kv_seq, seed=51, q_seq=q_seq, k_outliers=True)
    q2 = synth.normal_bf16((heads, q_seq, 128), 52)
    st = b.build_store(k.to(cuda), v.to(cuda))
    ref1 = b.attend(q1.to(cuda), st, q_chunk=q_chunk, kv_block=512).cpu()
    ref2 = b.attend(q2.to(cuda), st, q_chunk=q_chunk, kv_block=512).cpu()
    h1, h2 = q1.contiguous().pin_memory(), q2.contiguous().pin_memory()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    s1.wait_stream(torch.cuda.current_stream())
    s2.wait_stream(torch.cuda.current_stream())
    o1 = b.attend_hostio(h1, st, q_chunk=q_chunk, kv_block=512, stream=s1)
    o2 = b.attend_hostio(h2, st, q_chunk=q_chunk, kv_block=512, stream=s2)
    b.sync_status(s1)
    b.sync_status(s2)
    assert torch.equal(o1, ref1) and torch.equal(o2, ref2)
