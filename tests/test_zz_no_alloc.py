"""h3kv_attend_staged_static: staged kvi8r attention for callers that cannot
allocate device memory (for example a plugin whose host application owns all
device memory, or code where a cudaMalloc -- which can synchronise the device
-- is not allowed).  Its scratch is a fixed array inside the library.

Kept in a file that pytest collects last, so that a run stopping at the first
failure has already run every other test.
"""
import ctypes

import pytest
import torch

import oracle
from parity import compare_attention
from store_h3kv_build_gb300 import binding as b
from store_h3kv_build_gb300 import synth

LIMIT = b.H3KV_STATIC_SCRATCH_BYTES


def _static(q, store, q_chunk, kv_block, out):
    st = store.c_struct()
    stream = torch.cuda.current_stream().cuda_stream
    return b.h3kv_attend_staged_static(q.data_ptr(), q.shape[1], ctypes.byref(st), q_chunk, kv_block, 0.0,
                                       out.data_ptr(), stream)


@pytest.mark.gpu
def test_static_scratch_matches_staged_on_two_calls(cuda):
    # Two calls in a row share (and reuse) the fixed scratch.  The staged
    # path is deterministic and its result does not depend on where the
    # store lives or how many staging blocks it uses, so the output must equal
    # h3kv_attend_staged's (two staging blocks, here) and h3kv_attend's on a
    # device-resident store bit for bit; it must also meet the oracle bar.
    heads, seq, q_chunk, kv_block = 2, 1500, 512, 512
    for seed in (51, 52):
        q, k, v = synth.make_qkv(heads, seq, seed=seed, k_outliers=True)
        qd = q.to(cuda)
        dev = b.build_store(k.to(cuda), v.to(cuda))
        host = b.build_store(k.to(cuda), v.to(cuda), out=b.Store.empty(heads, seq, host=True))
        ref_staged = b.attend_staged(qd, host, q_chunk=q_chunk, kv_block=kv_block)
        ref_resident = b.attend(qd, dev, q_chunk=q_chunk, kv_block=kv_block)
        out = torch.empty(qd.shape, dtype=torch.float32, device=cuda)
        assert _static(qd, host, q_chunk, kv_block, out) == b.H3KV_OK
        b.sync_status()
        assert torch.equal(out, ref_staged)
        assert torch.equal(out, ref_resident)
        compare_attention(out, oracle.attend(q, oracle.build_store(k, v)), f"static scratch, seed {seed}")


@pytest.mark.gpu
def test_static_scratch_call_at_its_limit(cuda):
    # one head, 128-key blocks: the staging block takes 33280 bytes and the
    # rest of the fixed scratch holds the row state of exactly this many
    # query rows; one more row is refused
    staging = 2 * 1 * 128 * 130
    q_seq = (LIMIT - staging) // 8
    q, k, v = synth.make_qkv(1, 300, seed=53, q_seq=q_seq, device=cuda)
    dev = b.build_store(k, v)
    host = b.build_store(k, v, out=b.Store.empty(1, 300, host=True))
    out = torch.empty(q.shape, dtype=torch.float32, device=cuda)
    assert _static(q, host, 1 << 20, 128, out) == b.H3KV_OK
    ref = b.attend(q, dev, q_chunk=1 << 20, kv_block=128)
    b.sync_status()
    assert torch.equal(out, ref)
    st = host.c_struct()
    assert b.h3kv_attend_staged_static(q.data_ptr(), q_seq + 1, ctypes.byref(st), 1 << 20, 128, 0.0,
                                       out.data_ptr(), None) == b.H3KV_ERR_INVALID_ARG


def _fake_store(heads, seq, head_dim=128, scale_group=0):
    return b.h3kv_store(4096, 4096, 4096, 4096, heads, seq, head_dim, scale_group)


def _call(store, q_seq, q_chunk=16384, kv_block=16384):
    return b.h3kv_attend_staged_static(4096, q_seq, ctypes.byref(store), q_chunk, kv_block, 0.0, 4096, None)


def test_static_scratch_rejects_staging_beyond_its_limit():
    # 32 heads x 16384-key blocks need 136 MB of staging: more than the fixed
    # scratch holds, so the call is refused before any device work
    assert _call(_fake_store(32, 217088), 217088) == b.H3KV_ERR_INVALID_ARG


def test_static_scratch_rejects_row_state_beyond_its_limit():
    # one head and 128-key blocks: the 33280-byte staging block fits, and the
    # row state of one query row more than the rest of the scratch holds does
    # not; an absurd q_seq is refused without any size product wrapping
    staging = 2 * 1 * 128 * 130
    st = _fake_store(1, 300)
    assert _call(st, (LIMIT - staging) // 8 + 1, kv_block=128) == b.H3KV_ERR_INVALID_ARG
    assert _call(st, 2 ** 62, kv_block=128) == b.H3KV_ERR_INVALID_ARG
    assert _call(_fake_store(65535, 300), 2 ** 62, kv_block=128) == b.H3KV_ERR_INVALID_ARG


def test_static_scratch_rejects_stores_as_the_staged_path_does():
    # the same status as h3kv_attend_staged, whatever the size: head_dim other
    # than 128 and per-32-value scales are unsupported, a bad scale group or
    # chunk is an invalid argument
    for q_seq in (10, 2 ** 40):
        assert _call(_fake_store(4, 300, head_dim=64), q_seq) == b.H3KV_ERR_UNSUPPORTED
        assert _call(_fake_store(4, 300, scale_group=32), q_seq) == b.H3KV_ERR_UNSUPPORTED
        assert _call(_fake_store(4, 300, scale_group=7), q_seq) == b.H3KV_ERR_INVALID_ARG
        assert _call(_fake_store(4, 300), q_seq, q_chunk=0) == b.H3KV_ERR_INVALID_ARG
        assert _call(_fake_store(4, 300), q_seq, kv_block=100) == b.H3KV_ERR_INVALID_ARG
