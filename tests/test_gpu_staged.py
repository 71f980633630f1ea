"""kvi8r attention over a store held outside HBM, staged one kv_block at a time.

The kv_block row of the H3 Streamed Blocks Inputs table keeps the blockwise
log-sum-exp combine "for the host-staged K/V design to come".
h3kv_attend_staged copies each block of the store (here in pinned Grace
memory) into an HBM staging buffer, attends every query chunk over it, and
carries the combine across blocks in a per-row (max, sum) state.  Its output
must be bit-identical to h3kv_attend over the same store with the same
q_chunk and kv_block, and match the oracle.
"""
import pytest
import torch

import oracle
from parity import compare_attention
from store_h3kv_build_gb300 import synth

pytestmark = pytest.mark.gpu


def _b():
    from store_h3kv_build_gb300 import binding as b
    return b


@pytest.mark.parametrize("heads,q_seq,kv_seq,q_chunk,kv_block", [
    (1, 1024, 1024, 256, 512),      # two blocks
    (2, 1000, 1337, 300, 256),      # six blocks, ragged last block and query chunks
    (3, 129, 5, 64, 128),           # one block shorter than a tile
    (1, 4096, 4096, 4096, 0),       # kv_block 16384 > sequence: one block
    (2, 700, 3000, 256, 1024),      # three blocks, last one ragged
    (2, 2100, 5000, 512, 512),      # ten blocks of five query chunks each
])
@pytest.mark.parametrize("buffers", [1, 2])
def test_staged_bit_identical_to_resident(cuda, heads, q_seq, kv_seq, q_chunk, kv_block, buffers):
    # buffers 1: each block copied on the caller's stream between the blocks'
    # launches; 2: the next block copied on a second stream meanwhile
    b = _b()
    q, k, v = synth.make_qkv(heads, kv_seq, seed=31, q_seq=q_seq, k_outliers=True)
    qd = q.to(cuda)
    dev = b.build_store(k.to(cuda), v.to(cuda))
    host = b.build_store(k.to(cuda), v.to(cuda), out=b.Store.empty(heads, kv_seq, host=True))
    ref = b.attend(qd, dev, q_chunk=q_chunk, kv_block=kv_block)
    nbytes = b.h3kv_staging_bytes(heads, kv_block) if buffers == 1 else b.staging_bytes_double(heads, kv_block)
    staging = torch.empty(nbytes, dtype=torch.uint8, device=cuda)
    staged_host = b.attend_staged(qd, host, q_chunk=q_chunk, kv_block=kv_block, staging=staging)
    staged_dev = b.attend_staged(qd, dev, q_chunk=q_chunk, kv_block=kv_block, staging=staging)
    b.sync_status()
    assert torch.equal(staged_host, ref)
    assert torch.equal(staged_dev, ref)
    compare_attention(staged_host, oracle.attend(q, oracle.build_store(k, v)), f"staged {heads}x{q_seq}x{kv_seq}")


def test_staged_bit_identical_to_head_major_resident(cuda):
    # at 131072 keys with 4096-row chunks the resident call launches head by
    # head; the staged call runs block by block over all heads
    b = _b()
    heads, q_seq, kv_seq, q_chunk, kv_block = 2, 4500, 131072, 4096, 16384
    assert b.h3kv_attend_launch_count(q_seq, kv_seq, heads, q_chunk) == heads * 2
    q, k, v = synth.make_qkv(heads, kv_seq, seed=33, q_seq=q_seq, k_outliers=True, device=cuda)
    dev = b.build_store(k, v)
    host = b.build_store(k, v, out=b.Store.empty(heads, kv_seq, host=True))
    ref = b.attend(q, dev, q_chunk=q_chunk, kv_block=kv_block)
    staging = torch.empty(b.staging_bytes_double(heads, kv_block), dtype=torch.uint8, device=cuda)
    out = b.attend_staged(q, host, q_chunk=q_chunk, kv_block=kv_block, staging=staging)
    b.sync_status()
    assert torch.equal(out, ref)


def test_staged_reuses_scratch_across_calls(cuda):
    # the same staging buffer and state serve consecutive calls; nothing of a
    # previous call may leak into the next
    b = _b()
    heads, seq, kvb = 2, 2000, 512
    staging = torch.empty(b.h3kv_staging_bytes(heads, kvb), dtype=torch.uint8, device=cuda)
    state = torch.full((heads, seq, 2), float("nan"), dtype=torch.float32, device=cuda)
    outs = []
    for seed in (41, 42, 41):
        q, k, v = synth.make_qkv(heads, seq, seed=seed)
        host = b.build_store(k.to(cuda), v.to(cuda), out=b.Store.empty(heads, seq, host=True))
        outs.append(b.attend_staged(q.to(cuda), host, q_chunk=700, kv_block=kvb, staging=staging, state=state))
    b.sync_status()
    assert torch.equal(outs[0], outs[2])
    assert not torch.equal(outs[0], outs[1])


def test_staged_double_buffer_on_a_side_stream(cuda):
    # two calls on a side stream sharing one two-block staging buffer, with the
    # store written on that stream just before: the copies stream is ordered
    # after earlier work on the stream, and later work sees every output row
    b = _b()
    heads, seq, kvb = 2, 3000, 256
    q, k, v = synth.make_qkv(heads, seq, seed=43, k_outliers=True)
    qd, kd, vd = q.to(cuda), k.to(cuda), v.to(cuda)
    ref = b.attend(qd, b.build_store(kd, vd), q_chunk=1000, kv_block=kvb)
    host = b.Store.empty(heads, seq, host=True)
    staging = torch.empty(b.staging_bytes_double(heads, kvb), dtype=torch.uint8, device=cuda)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        b.build_store(kd, vd, out=host, stream=side)
        o1 = b.attend_staged(qd, host, q_chunk=1000, kv_block=kvb, staging=staging, stream=side)
        o2 = b.attend_staged(qd, host, q_chunk=1000, kv_block=kvb, staging=staging, stream=side)
        s1, s2 = o1.sum(), o2.sum()
    b.sync_status(side)
    assert torch.equal(o1, ref) and torch.equal(o2, ref)
    assert float(s1) == float(s2)


def test_staged_calls_on_two_streams_at_once(cuda):
    # two calls in flight together over one store in Grace memory, each with
    # the staging and state the binding creates for it (two staging blocks,
    # a copy stream per call): both outputs bit-identical to the resident path
    b = _b()
    heads, seq, kvb = 2, 3000, 256
    q1, k, v = synth.make_qkv(heads, seq, seed=44, k_outliers=True)
    q2 = synth.normal_bf16((heads, seq, 128), 45)
    kd, vd = k.to(cuda), v.to(cuda)
    dev = b.build_store(kd, vd)
    host = b.build_store(kd, vd, out=b.Store.empty(heads, seq, host=True))
    ref1 = b.attend(q1.to(cuda), dev, q_chunk=1000, kv_block=kvb)
    ref2 = b.attend(q2.to(cuda), dev, q_chunk=1000, kv_block=kvb)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    s1.wait_stream(torch.cuda.current_stream())
    s2.wait_stream(torch.cuda.current_stream())
    qa, qb = q1.to(cuda), q2.to(cuda)
    s1.wait_stream(torch.cuda.current_stream())
    s2.wait_stream(torch.cuda.current_stream())
    o1 = b.attend_staged(qa, host, q_chunk=1000, kv_block=kvb, stream=s1)
    o2 = b.attend_staged(qb, host, q_chunk=1000, kv_block=kvb, stream=s2)
    b.sync_status(s1)
    b.sync_status(s2)
    assert torch.equal(o1, ref1) and torch.equal(o2, ref2)


def test_host_store_buffers_are_all_pinned(cuda):
    # the staged copies are stream-ordered only from pinned memory; every
    # buffer of a host store must be page-locked, not only the first of each
    # kind (an empty_like of a pinned tensor is pageable)
    b = _b()
    for sg in (0, 32):
        st = b.Store.empty(2, 300, host=True, scale_group=sg)
        assert all(t.is_pinned() for t in (st.k_codes, st.v_codes, st.k_scales, st.v_scales))


def test_staged_refuses_a_pageable_store(cuda):
    # a store buffer in pageable host memory is refused before any copy:
    # copies from it would take its bytes when issued, not in stream order
    b = _b()
    heads, seq = 1, 300
    q, k, v = synth.make_qkv(heads, seq, seed=61)
    st = b.Store.empty(heads, seq, host=True)
    st.v_codes = torch.empty((heads, seq, 128), dtype=torch.int8)  # pageable
    with pytest.raises(b.H3kvError) as e:
        b.attend_staged(q.to(cuda), st, q_chunk=256, kv_block=128)
    assert e.value.status == b.H3KV_ERR_INVALID_ARG


@pytest.mark.parametrize("buffers", [1, 2])
def test_staged_reads_a_host_store_built_just_before(cuda, buffers):
    # the store is built into host memory behind a long queue of GPU work and
    # attended at once, with no synchronisation: the block copies must read
    # it in stream order, after the build (a pageable buffer was read before
    # the build ran, and every output row was wrong)
    b = _b()
    heads, seq, kvb = 1, 300, 128
    q, k, v = synth.make_qkv(heads, seq, seed=62, q_seq=200000, device=cuda)
    ref = b.attend(q, b.build_store(k, v), q_chunk=1 << 16, kv_block=kvb)
    b.sync_status()
    x = torch.randn((8192, 8192), device=cuda)
    for _ in range(40):  # tens of milliseconds of queued work before the build
        x = (x @ x) * 1e-3
    host = b.build_store(k, v, out=b.Store.empty(heads, seq, host=True))
    nbytes = b.h3kv_staging_bytes(heads, kvb) if buffers == 1 else b.staging_bytes_double(heads, kvb)
    out = b.attend_staged(q, host, q_chunk=1 << 16, kv_block=kvb,
                          staging=torch.empty(nbytes, dtype=torch.uint8, device=cuda))
    b.sync_status()
    assert torch.equal(out, ref)
