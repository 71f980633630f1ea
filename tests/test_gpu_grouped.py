"""GPU parity of the per-32-value scale variant of kvi8r (the Low VRAM
write-up's roadmap: "a per-32-value scale variant of kvi8r (finer than per
row)"): every row's 4 groups of 32 rotated values get their own fp16 scale.
Build and attention through the C ABI against the oracle's grouped store."""
import numpy as np
import pytest
import torch

import oracle
from parity import compare_attention, compare_store
from store_h3kv_build_gb300 import synth

pytestmark = pytest.mark.gpu


def _b():
    from store_h3kv_build_gb300 import binding as b
    return b


def _check_store(st, k, v, what):
    ref = oracle.build_store_grouped(k.cpu(), v.cpu())
    for name in ("k", "v"):
        compare_store(getattr(st, f"{name}_codes"), getattr(st, f"{name}_scales"), ref[f"{name}_codes"],
                      ref[f"{name}_scales"], f"{what} {name}")


@pytest.mark.parametrize("heads,seq", [(1, 1024), (3, 1000), (2, 129), (4, 4096)])
def test_grouped_store_matches_oracle(cuda, heads, seq):
    b = _b()
    q, k, v = synth.make_qkv(heads, seq, seed=61, k_outliers=True)
    st = b.build_store(k.to(cuda), v.to(cuda), scale_group=32)
    b.sync_status()
    assert tuple(st.k_scales.shape) == (heads, seq, 4)
    _check_store(st, k, v, f"g32 {heads}x{seq}")


def test_grouped_store_special_rows(cuda):
    # a zero row; a row whose signal lives in one rotated group only is not
    # constructible from K directly, so use rows spanning 5 orders of magnitude
    k = synth.normal_f32((1, 300, 128), 62)
    k[0, 0] = 0
    k[0, 1] *= 1e-6
    k[0, 2] *= 1e4
    k[0, 3:40, 9] *= 50
    kb = k.to(torch.bfloat16)
    vb = synth.normal_bf16((1, 300, 128), 63)
    b = _b()
    st = b.build_store(kb.to(cuda), vb.to(cuda), scale_group=32)
    b.sync_status()
    _check_store(st, kb, vb, "g32 special")
    assert not st.k_codes[0, 0].any() and not st.k_scales[0, 0].any()


@pytest.mark.parametrize("heads,q_seq,kv_seq,q_chunk,kv_block", [(1, 1024, 1024, 256, 512),
                                                                 (2, 1000, 1337, 300, 512),
                                                                 (3, 129, 5, 64, 0)])
def test_grouped_attend_matches_oracle(cuda, heads, q_seq, kv_seq, q_chunk, kv_block):
    b = _b()
    q, k, v = synth.make_qkv(heads, kv_seq, seed=64, q_seq=q_seq, k_outliers=True)
    st = b.build_store(k.to(cuda), v.to(cuda), scale_group=32)
    out = b.attend(q.to(cuda), st, q_chunk=q_chunk, kv_block=kv_block)
    b.sync_status()
    compare_attention(out, oracle.attend(q, oracle.build_store_grouped(k, v)), f"g32 {heads}x{q_seq}x{kv_seq}")


def test_grouped_attend_bit_identical_across_q_chunk(cuda):
    b = _b()
    q, k, v = synth.make_qkv(2, 2500, seed=65)
    q = q.to(cuda)
    st = b.build_store(k.to(cuda), v.to(cuda), scale_group=32)
    outs = [b.attend(q, st, q_chunk=c, kv_block=1024) for c in (2500, 1, 300, 1024)]
    b.sync_status()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


def test_grouped_closer_to_exact_than_per_row(cuda):
    b = _b()
    q, k, v = synth.make_qkv(4, 4096, seed=66, k_outliers=True)
    q, k, v = q.to(cuda), k.to(cuda), v.to(cuda)
    exact = b.attend_exact(q, k, v, q_chunk=4096)
    o_row = b.attend(q, b.build_store(k, v), q_chunk=4096)
    o_grp = b.attend(q, b.build_store(k, v, scale_group=32), q_chunk=4096)
    b.sync_status()
    r_row = oracle.rel_rms(o_row.cpu(), exact.cpu())
    r_grp = oracle.rel_rms(o_grp.cpu(), exact.cpu())
    assert r_grp < r_row
