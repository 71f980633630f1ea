"""Failure detection on the GPU without faulting it.

Every wait in the kernels is bounded.  These tests make waits run out on
purpose -- one on a barrier that nothing ever arrives on, and in the real
attention kernels a "P ready" arrival that the softmax warps withhold -- and
check that the host reads H3KV_ERR_DEVICE_TIMEOUT, that the error word
clears, and that the context still computes correct results afterwards.  The
real kernels also run under a wait limit far below their normal waits: a
suspended barrier poll can outlast such a limit, so there they may finish
cleanly, and then their output must be right.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import compare_attention
from store_h3kv_build_gb300 import synth

pytestmark = pytest.mark.gpu


def _b():
    from store_h3kv_build_gb300 import binding as b
    return b


def _tiny_check(cuda):
    b = _b()
    q, k, v = synth.make_qkv(1, 1024, seed=0)
    st = b.build_store(k.to(cuda), v.to(cuda))
    out = b.attend(q.to(cuda), st, q_chunk=256, kv_block=512)
    b.sync_status()
    compare_attention(out, oracle.attend(q, oracle.build_store(k, v)), "after timeout")


def test_selftest_wait_runs_out_and_context_survives(cuda):
    b = _b()
    s = torch.cuda.current_stream().cuda_stream
    assert b.h3kv_sync_status(s) == b.H3KV_OK
    assert b.h3kv_selftest_wait_timeout(2_000_000, s) == b.H3KV_OK  # 2 ms limit
    assert b.h3kv_sync_status(s) == b.H3KV_ERR_DEVICE_TIMEOUT
    assert b.h3kv_sync_status(s) == b.H3KV_OK  # cleared
    _tiny_check(cuda)


def _run(b, path, q, k, v, st, st8, st4, hq):
    if path == "store":
        return b.build_store(k, v, out=st)
    if path == "kvi8r":
        return b.attend(q, st, q_chunk=4096, kv_block=0)
    if path == "exact":
        return b.attend_exact(q, k, v, q_chunk=4096, kv_block=0)
    if path == "store_f8":
        return b.build_store_f8(k, v, out=st8)
    if path == "store_fp4":
        return b.build_store_fp4(k, v, out=st4)
    if path == "kvfp4":
        return b.attend_fp4(q, st4, q_chunk=4096, kv_block=0)
    if path == "hostio":
        # four chunks: the chained launches' ready-word waits run under the limit too
        return b.attend_hostio(hq, st, q_chunk=1024, kv_block=0)
    if path == "staged":
        # four blocks through two staging buffers: the blocks' ready-word waits too
        return b.attend_staged(q, st, q_chunk=2048, kv_block=1024)
    assert path == "kvf8s"
    return b.attend_f8(q, st8, q_chunk=4096, kv_block=0)


def _inputs(cuda):
    b = _b()
    q, k, v = synth.make_qkv(2, 4096, seed=3)
    q, k, v = q.to(cuda), k.to(cuda), v.to(cuda)
    st = b.build_store(k, v)
    st8 = b.build_store_f8(k, v)
    st4 = b.build_store_fp4(k, v)
    hq = q.cpu().contiguous().pin_memory()
    return q, k, v, st, st8, st4, hq


ATTENTION_PATHS = ["kvi8r", "exact", "kvf8s", "kvfp4", "hostio", "staged"]


@pytest.mark.parametrize("path", ATTENTION_PATHS)
def test_withheld_arrival_runs_out_and_context_survives(cuda, path):
    b = _b()
    s = torch.cuda.current_stream().cuda_stream
    q, k, v, st, st8, st4, hq = _inputs(cuda)
    assert b.h3kv_sync_status(s) == b.H3KV_OK
    # the softmax warps never report P of tile 1 ready; a 2 ms limit
    b.check(b.h3kv_set_wait_timeout_ns(2_000_000))
    b.check(b.h3kv_debug_withhold_p(1))
    try:
        _run(b, path, q, k, v, st, st8, st4, hq)
        status = b.h3kv_sync_status(s)
    finally:
        b.check(b.h3kv_debug_withhold_p(-1))
        b.check(b.h3kv_set_wait_timeout_ns(0))
    assert status == b.H3KV_ERR_DEVICE_TIMEOUT
    assert b.h3kv_sync_status(s) == b.H3KV_OK
    _tiny_check(cuda)


@pytest.mark.parametrize("path", ["store", "store_f8", "store_fp4"] + ATTENTION_PATHS)
def test_kernels_under_tiny_wait_limit(cuda, path):
    b = _b()
    s = torch.cuda.current_stream().cuda_stream
    q, k, v, st, st8, st4, hq = _inputs(cuda)
    assert b.h3kv_sync_status(s) == b.H3KV_OK
    b.check(b.h3kv_set_wait_timeout_ns(1))
    try:
        out = _run(b, path, q, k, v, st, st8, st4, hq)
        status = b.h3kv_sync_status(s)
    finally:
        b.check(b.h3kv_set_wait_timeout_ns(0))
    # a wait whose phase completes inside its first suspended poll never runs
    # out, so any kernel may finish cleanly: then its output must be right
    assert status in (b.H3KV_OK, b.H3KV_ERR_DEVICE_TIMEOUT)
    if status == b.H3KV_OK and path in ("kvi8r", "exact"):
        rows = torch.arange(0, q.shape[1], 61)
        if path == "exact":
            ref = oracle.attend_exact(q[:, rows].cpu(), k.cpu(), v.cpu())
        else:
            ref = oracle.attend(q[:, rows].cpu(), oracle.build_store(k.cpu(), v.cpu()))
        compare_attention(out[:, rows], ref, f"{path} under a tiny limit")
    assert b.h3kv_sync_status(s) == b.H3KV_OK
    _tiny_check(cuda)
