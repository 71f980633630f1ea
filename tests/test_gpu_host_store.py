"""kvi8r store resident in Grace memory, read over NVLink-C2C.

The kv_block row of the H3 Streamed Blocks Inputs table keeps the blockwise
design "for the host-staged K/V design to come".  On a Grace-Blackwell node the
GPU addresses pinned host memory directly, so the store (int8 codes and fp16
scales) can live in host memory while the same kernels build it and attend
over it.  The results must be bit-identical to the HBM-resident store.
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


@pytest.mark.parametrize("heads,seq,q_chunk,kv_block", [(1, 1024, 256, 512), (3, 1337, 300, 256),
                                                        (2, 4096, 4096, 0)])
def test_host_store_matches_device_store(cuda, heads, seq, q_chunk, kv_block):
    b = _b()
    q, k, v = synth.make_qkv(heads, seq, seed=21, k_outliers=True)
    qd, kd, vd = q.to(cuda), k.to(cuda), v.to(cuda)
    dev = b.build_store(kd, vd)
    host = b.build_store(kd, vd, out=b.Store.empty(heads, seq, host=True))
    b.sync_status()
    assert host.in_host_memory
    for name in ("k_codes", "v_codes", "k_scales", "v_scales"):
        assert torch.equal(getattr(host, name), getattr(dev, name).cpu()), name
    o_dev = b.attend(qd, dev, q_chunk=q_chunk, kv_block=kv_block)
    o_host = b.attend(qd, host, q_chunk=q_chunk, kv_block=kv_block)
    b.sync_status()
    assert torch.equal(o_dev, o_host)
    compare_attention(o_host, oracle.attend(q, oracle.build_store(k, v)), f"host store {heads}x{seq}")


@pytest.mark.parametrize("heads,seq,group", [(2, 3000, 0), (1, 129, 0), (3, 1000, 32)])
def test_store_built_from_host_inputs(cuda, heads, seq, group):
    # bf16 K and V left in pinned host memory: the build kernel reads them
    # over NVLink-C2C and writes the same store as from HBM copies
    b = _b()
    _, k, v = synth.make_qkv(heads, seq, seed=23, k_outliers=True)
    hk, hv = k.pin_memory(), v.pin_memory()
    dev = b.build_store(k.to(cuda), v.to(cuda), scale_group=group)
    from_host = b.build_store(hk, hv, out=b.Store.empty(heads, seq, cuda, scale_group=group))
    b.sync_status()
    for name in ("k_codes", "v_codes", "k_scales", "v_scales"):
        assert torch.equal(getattr(from_host, name), getattr(dev, name)), name
