"""The binding's argument checks, on the CPU: the library reads and writes raw
contiguous buffers of the sizes its arguments imply, so the binding refuses
strided views, other dtypes and buffers of other shapes before any call
(otherwise they would be read as garbage or written past their end)."""
import pytest
import torch

from store_h3kv_build_gb300 import binding as b

H, L = 2, 64


def _qkv(dtype=torch.bfloat16):
    return (torch.zeros((H, L, 128), dtype=dtype), torch.zeros((H, L, 128), dtype=dtype),
            torch.zeros((H, L, 128), dtype=dtype))


def _store():
    return b.Store(torch.zeros((H, L, 128), dtype=torch.int8), torch.zeros((H, L, 128), dtype=torch.int8),
                   torch.zeros((H, L), dtype=torch.float16), torch.zeros((H, L), dtype=torch.float16))


def test_inputs_must_be_bf16_contiguous_with_head_dim_128():
    q, k, v = _qkv()
    with pytest.raises(TypeError, match="dtype"):
        b.build_store(k.float(), v)
    with pytest.raises(ValueError, match="contiguous"):
        b.build_store(k.transpose(0, 1), v)
    with pytest.raises(ValueError, match="heads, rows, 128"):
        b.build_store(k[..., :64].contiguous(), v[..., :64].contiguous())
    with pytest.raises(ValueError, match="K has"):
        b.build_store(k, v[:, :32].contiguous())
    with pytest.raises(ValueError, match="contiguous"):
        b.attend_exact(q[:, ::2], k, v)


def test_query_heads_must_match_the_store():
    q, _, _ = _qkv()
    with pytest.raises(ValueError, match="heads"):
        b.attend(q[:1].contiguous(), _store())
    with pytest.raises(ValueError, match="heads"):
        b.attend_hostio(q[:1].contiguous(), _store())


def test_store_buffers_must_match_heads_and_seq():
    st = _store()
    st.v_codes = torch.zeros((H, L - 1, 128), dtype=torch.int8)  # one row short: a write past its end
    with pytest.raises(ValueError, match="store.v_codes"):
        st.c_struct()
    st = _store()
    st.k_scales = torch.zeros((H, L), dtype=torch.float32)
    with pytest.raises(TypeError, match="store.k_scales"):
        st.c_struct()
    s8 = b.StoreF8(torch.zeros((H, L, 128), dtype=torch.uint8), torch.zeros((H, 128, L), dtype=torch.uint8),
                   torch.zeros((H, 1), dtype=torch.float32), torch.zeros((H, 128), dtype=torch.float32),
                   torch.zeros((H, 128), dtype=torch.float32), L)
    s8.c_struct()  # L = 64 is a multiple of 16, one K block: the right sizes
    s8.k_scales = torch.zeros((H, 2), dtype=torch.float32)
    with pytest.raises(ValueError, match="store.k_scales"):
        s8.c_struct()
    s4 = b.StoreFp4(*(torch.zeros((H, L, n), dtype=torch.uint8) for n in (64, 64, 8, 8)))
    s4.c_struct()
    s4.v_scales = torch.zeros((H, L, 4), dtype=torch.uint8)
    with pytest.raises(ValueError, match="store.v_scales"):
        s4.c_struct()


def test_outputs_and_scratch_must_have_the_implied_shape():
    q, _, _ = _qkv()
    with pytest.raises(ValueError, match="out"):
        b.attend(q, _store(), out=torch.zeros((H, L, 64), dtype=torch.float32))
    with pytest.raises(TypeError, match="out"):
        b.attend(q, _store(), out=torch.zeros((H, L, 128), dtype=torch.float16))
    with pytest.raises(ValueError, match="state"):
        b.attend_staged(q, _store(), staging=torch.zeros(16, dtype=torch.uint8),
                        state=torch.zeros((H, L, 3), dtype=torch.float32))
    with pytest.raises(TypeError, match="scratch"):
        b.attend_hostio(q, _store(), out=torch.zeros((H, L, 128), dtype=torch.float32),
                        scratch=torch.zeros(16, dtype=torch.float32))
