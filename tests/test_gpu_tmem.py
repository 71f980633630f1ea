"""The reducing tensor-memory load (tcgen05.ld.red, sm_103a) that every
attention path uses for the row maximum of a full key tile.  The library's
self-test stores known values into tensor memory and checks each reduced
maximum and every reloaded value; the attention parity tests then check the
kernels that rely on it against the oracle."""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


def test_reducing_tmem_load_returns_group_maxima(cuda):
    from store_h3kv_build_gb300 import binding as b
    s = torch.cuda.current_stream().cuda_stream
    count = ctypes.c_int32(-1)
    assert b.h3kv_selftest_tmem_ld_max(ctypes.byref(count), s) == b.H3KV_OK
    assert count.value == 0
    assert b.h3kv_sync_status(s) == b.H3KV_OK
