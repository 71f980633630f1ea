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

from parity import ATT_MAX_ABS, ATT_MEAN_ABS
from store_h3kv_build_gb300 import binding as b
from store_h3kv_build_gb300 import synth


@pytest.mark.gpu
def test_static_scratch_matches_staged_on_two_calls(cuda):
    heads, seq, q_chunk, kv_block = 2, 1500, 512, 512
    stream = torch.cuda.current_stream().cuda_stream
    for seed in (51, 52):  # two calls in a row share (and reuse) the fixed scratch
        q, k, v = synth.make_qkv(heads, seq, seed=seed, k_outliers=True)
        q = q.to(cuda)
        host = b.build_store(k.to(cuda), v.to(cuda), out=b.Store.empty(heads, seq, host=True))
        ref = b.attend_staged(q, host, q_chunk=q_chunk, kv_block=kv_block)
        out = torch.empty(q.shape, dtype=torch.float32, device=cuda)
        st = host.c_struct()
        rc = b.h3kv_attend_staged_static(q.data_ptr(), seq, ctypes.byref(st), q_chunk, kv_block, 0.0,
                                         out.data_ptr(), stream)
        assert rc == b.H3KV_OK
        b.sync_status()
        err = (out.double() - ref.double()).abs()
        assert torch.isfinite(out).all()
        assert err.max().item() <= ATT_MAX_ABS and err.mean().item() <= ATT_MEAN_ABS


def test_static_scratch_rejects_sizes_beyond_its_limit():
    # 32 heads x 217088 query rows need 55.6 MB of row state: more than the
    # fixed scratch holds, so the call is refused before any device work
    st = b.h3kv_store(4096, 4096, 4096, 4096, 32, 217088, 128)
    rc = b.h3kv_attend_staged_static(4096, 217088, ctypes.byref(st), 16384, 16384, 0.0, 4096, None)
    assert rc == b.H3KV_ERR_INVALID_ARG
