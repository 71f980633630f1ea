"""Checkpoint and resume of a kvi8r store.

The store is four plain buffers (h3kv_store_bytes gives their total size), so
a caller can save it and attend over the restored copy later.  Attention over
a store that went through a file must equal attention over the original.
"""
import pytest
import torch

from store_h3kv_build_gb300 import synth

pytestmark = pytest.mark.gpu


def test_store_survives_save_and_restore(cuda, tmp_path):
    from store_h3kv_build_gb300 import binding as b
    q, k, v = synth.make_qkv(2, 3000, seed=81, k_outliers=True)
    q = q.to(cuda)
    st = b.build_store(k.to(cuda), v.to(cuda))
    ref = b.attend(q, st, q_chunk=1000, kv_block=1024)
    b.sync_status()
    path = tmp_path / "store.pt"
    torch.save({n: getattr(st, n).cpu() for n in ("k_codes", "v_codes", "k_scales", "v_scales")}, path)
    assert sum(getattr(st, n).numel() * getattr(st, n).element_size()
               for n in ("k_codes", "v_codes", "k_scales", "v_scales")) == st.nbytes()
    saved = torch.load(path)
    restored = b.Store(*(saved[n].to(cuda) for n in ("k_codes", "v_codes", "k_scales", "v_scales")))
    out = b.attend(q, restored, q_chunk=1000, kv_block=1024)
    b.sync_status()
    assert torch.equal(out, ref)
