"""CPU-side checks of the C-ABI library: it loads, exports every entry point
that include/h3kv.h declares, and rejects bad arguments on the host before any
launch (no GPU is needed for any of these)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "h3kv.h")

from store_h3kv_build_gb300 import binding as b  # noqa: E402  (built by conftest if missing)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(h3kv_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert len(names) == 24
    assert {"h3kv_attend_f8", "h3kv_build_store_f8", "h3kv_f8_v_stride", "h3kv_store_f8_bytes"} <= set(names)
    assert {"h3kv_attend_fp4", "h3kv_build_store_fp4", "h3kv_store_fp4_bytes"} <= set(names)
    lib = ctypes.CDLL(b.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(b.EXPORTED)


def test_abi_version_and_strings():
    assert b.h3kv_abi_version() == 9
    for st in range(5):
        assert b.h3kv_strerror(st)
    assert b.h3kv_strerror(99) == b"unknown status"


def test_store_bytes():
    assert b.h3kv_store_bytes(32, 217088, 128) == 2 * 32 * 217088 * 130
    assert b.h3kv_store_bytes(1, 0, 128) == 0
    assert b.h3kv_store_bytes(1, 10, 64) == 0
    assert b.h3kv_store_bytes(-1, 10, 128) == 0


def _store(heads=1, seq=256, ptr=4096, head_dim=128):
    return b.h3kv_store(ptr, ptr, ptr, ptr, heads, seq, head_dim)


def test_build_store_rejects_bad_arguments():
    st = _store()
    bs = b.h3kv_build_store
    assert bs(4096, 4096, 1, 256, 128, None, None) == b.H3KV_ERR_INVALID_ARG          # no store
    assert bs(4096, 4096, 1, 256, 64, ctypes.byref(st), None) == b.H3KV_ERR_UNSUPPORTED  # head_dim
    assert bs(4096, 4096, 2, 256, 128, ctypes.byref(st), None) == b.H3KV_ERR_INVALID_ARG  # shape mismatch
    assert bs(0, 4096, 1, 256, 128, ctypes.byref(st), None) == b.H3KV_ERR_INVALID_ARG     # null K
    assert bs(4097, 4096, 1, 256, 128, ctypes.byref(st), None) == b.H3KV_ERR_INVALID_ARG  # misaligned
    assert bs(4096, 4096, -1, 256, 128, ctypes.byref(_store(heads=-1)), None) == b.H3KV_ERR_INVALID_ARG
    assert bs(0, 0, 0, 0, 128, ctypes.byref(_store(heads=0, seq=0, ptr=0)), None) == b.H3KV_OK  # empty


def test_attend_rejects_bad_arguments():
    st = _store()
    at = b.h3kv_attend
    assert at(4096, 256, None, 256, 0, 0.0, 4096, None) == b.H3KV_ERR_INVALID_ARG
    assert at(4096, 256, ctypes.byref(st), 0, 0, 0.0, 4096, None) == b.H3KV_ERR_INVALID_ARG     # q_chunk 0
    assert at(4096, 256, ctypes.byref(st), 64, 100, 0.0, 4096, None) == b.H3KV_ERR_INVALID_ARG  # kv_block % 128
    assert at(4096, 256, ctypes.byref(st), 64, -128, 0.0, 4096, None) == b.H3KV_ERR_INVALID_ARG
    assert at(4096, 256, ctypes.byref(_store(head_dim=64)), 64, 0, 0.0, 4096, None) == b.H3KV_ERR_UNSUPPORTED
    assert at(4104, 256, ctypes.byref(st), 64, 0, 0.0, 4096, None) == b.H3KV_ERR_INVALID_ARG    # misaligned Q
    assert at(4096, 256, ctypes.byref(st), 64, 0, 0.0, 0, None) == b.H3KV_ERR_INVALID_ARG       # null O
    assert at(4096, 256, ctypes.byref(_store(seq=0)), 64, 0, 0.0, 4096, None) == b.H3KV_ERR_INVALID_ARG
    assert at(4096, 0, ctypes.byref(st), 64, 0, 0.0, 4096, None) == b.H3KV_OK                  # empty queries


def test_attend_exact_rejects_bad_arguments():
    ae = b.h3kv_attend_exact
    assert ae(4096, 256, 4096, 4096, 1, 256, 96, 64, 0, 0.0, 4096, None) == b.H3KV_ERR_UNSUPPORTED
    assert ae(4096, 256, 4096, 4096, 1, 256, 128, 0, 0, 0.0, 4096, None) == b.H3KV_ERR_INVALID_ARG
    assert ae(4096, 256, 4096, 4096, 1, 256, 128, 64, 64, 0.0, 4096, None) == b.H3KV_ERR_INVALID_ARG
    assert ae(4096, 256, 0, 4096, 1, 256, 128, 64, 0, 0.0, 4096, None) == b.H3KV_ERR_INVALID_ARG
    assert ae(4096, 256, 4096, 4096, 1, 0, 128, 64, 0, 0.0, 4096, None) == b.H3KV_ERR_INVALID_ARG
    assert ae(4096, 256, 4096, 4104, 1, 256, 128, 64, 0, 0.0, 4096, None) == b.H3KV_ERR_INVALID_ARG
    assert ae(4096, 256, 4096, 4096, 0, 256, 128, 64, 0, 0.0, 4096, None) == b.H3KV_OK


def test_binding_raises_on_error_status():
    with pytest.raises(b.H3kvError) as e:
        b.check(b.H3KV_ERR_INVALID_ARG, "x")
    assert e.value.status == b.H3KV_ERR_INVALID_ARG


def test_wait_timeout_setter_needs_no_device():
    assert b.h3kv_set_wait_timeout_ns(5000) == b.H3KV_OK
    assert b.h3kv_set_wait_timeout_ns(0) == b.H3KV_OK


def test_withhold_p_setter_needs_no_device():
    assert b.h3kv_debug_withhold_p(0) == b.H3KV_OK
    assert b.h3kv_debug_withhold_p(-1) == b.H3KV_OK
    assert b.h3kv_debug_withhold_p(-2) == b.H3KV_ERR_INVALID_ARG


def test_staging_bytes():
    assert b.h3kv_staging_bytes(32, 16384) == 2 * 32 * 16384 * 130
    assert b.h3kv_staging_bytes(2, 0) == 2 * 2 * 16384 * 130
    assert b.h3kv_staging_bytes(2, 100) == 0
    assert b.h3kv_staging_bytes(-1, 128) == 0


def test_attend_staged_rejects_bad_arguments():
    st = _store()
    at = b.h3kv_attend_staged
    big = b.h3kv_staging_bytes(1, 256)
    assert at(4096, 256, None, 256, 256, 0.0, 4096, 4096, big, 4096, None) == b.H3KV_ERR_INVALID_ARG
    assert at(4096, 256, ctypes.byref(st), 0, 256, 0.0, 4096, 4096, big, 4096, None) == b.H3KV_ERR_INVALID_ARG
    assert at(4096, 256, ctypes.byref(st), 64, 200, 0.0, 4096, 4096, big, 4096, None) == b.H3KV_ERR_INVALID_ARG
    assert at(4096, 256, ctypes.byref(st), 64, 256, 0.0, 4096, 0, big, 4096, None) == b.H3KV_ERR_INVALID_ARG
    assert at(4096, 256, ctypes.byref(st), 64, 256, 0.0, 4096, 4096, big, 0, None) == b.H3KV_ERR_INVALID_ARG
    assert at(4096, 256, ctypes.byref(st), 64, 256, 0.0, 4096, 4096, big - 1, 4096, None) == b.H3KV_ERR_INVALID_ARG
    assert at(4096, 256, ctypes.byref(st), 64, 256, 0.0, 4096, 4104, big, 4096, None) == b.H3KV_ERR_INVALID_ARG
    assert at(4096, 256, ctypes.byref(_store(head_dim=64)), 64, 256, 0.0, 4096, 4096, big, 4096,
              None) == b.H3KV_ERR_UNSUPPORTED
    assert at(4096, 0, ctypes.byref(st), 64, 256, 0.0, 4096, 4096, big, 4096, None) == b.H3KV_OK


def test_scale_group_validation():
    bad = b.h3kv_store(4096, 4096, 4096, 4096, 1, 256, 128, 64)
    assert b.h3kv_build_store(4096, 4096, 1, 256, 128, ctypes.byref(bad), None) == b.H3KV_ERR_INVALID_ARG
    assert b.h3kv_attend(4096, 256, ctypes.byref(bad), 64, 0, 0.0, 4096, None) == b.H3KV_ERR_INVALID_ARG
    g32 = b.h3kv_store(4096, 4096, 4096, 4096, 1, 256, 128, 32)
    big = b.h3kv_staging_bytes(1, 256)
    assert b.h3kv_attend_staged(4096, 256, ctypes.byref(g32), 64, 256, 0.0, 4096, 4096, big, 4096,
                                None) == b.H3KV_ERR_UNSUPPORTED


def test_store_f8_sizes():
    assert b.h3kv_f8_v_stride(0) == 0 and b.h3kv_f8_v_stride(1) == 16 and b.h3kv_f8_v_stride(217088) == 217088
    assert b.h3kv_f8_v_stride(77) == 80 and b.h3kv_f8_v_stride(-5) == 0
    H, L = 32, 217088
    assert b.h3kv_store_f8_bytes(H, L, 128) == H * L * 128 * 2 + H * (L // 64) * 4 + 2 * H * 128 * 4
    assert b.h3kv_store_f8_bytes(1, 77, 128) == 77 * 128 + 128 * 80 + 2 * 4 + 2 * 128 * 4
    assert b.h3kv_store_f8_bytes(1, 10, 64) == 0 and b.h3kv_store_f8_bytes(-1, 10, 128) == 0


def _store_f8(heads=1, seq=256, ptr=4096, head_dim=128):
    return b.h3kv_store_f8(ptr, ptr, ptr, ptr, ptr, heads, seq, head_dim)


def test_build_store_f8_rejects_bad_arguments():
    st = _store_f8()
    bs = b.h3kv_build_store_f8
    assert bs(4096, 4096, 1, 256, 128, None, None) == b.H3KV_ERR_INVALID_ARG
    assert bs(4096, 4096, 1, 256, 64, ctypes.byref(st), None) == b.H3KV_ERR_UNSUPPORTED
    assert bs(4096, 4096, 2, 256, 128, ctypes.byref(st), None) == b.H3KV_ERR_INVALID_ARG   # shape mismatch
    assert bs(0, 4096, 1, 256, 128, ctypes.byref(st), None) == b.H3KV_ERR_INVALID_ARG      # null K
    assert bs(4100, 4096, 1, 256, 128, ctypes.byref(st), None) == b.H3KV_ERR_INVALID_ARG   # misaligned
    assert bs(4096, 4096, 1, 256, 128, ctypes.byref(_store_f8(ptr=0)), None) == b.H3KV_ERR_INVALID_ARG
    big = _store_f8(heads=70000, seq=1)
    assert bs(4096, 4096, 70000, 1, 128, ctypes.byref(big), None) == b.H3KV_ERR_INVALID_ARG  # grid limit
    assert bs(0, 0, 0, 0, 128, ctypes.byref(_store_f8(heads=0, seq=0, ptr=0)), None) == b.H3KV_OK


def test_attend_f8_rejects_bad_arguments():
    st = _store_f8()
    at = b.h3kv_attend_f8
    assert at(4096, 256, None, 256, 0, 0.0, 4096, None) == b.H3KV_ERR_INVALID_ARG
    assert at(4096, 256, ctypes.byref(st), 0, 0, 0.0, 4096, None) == b.H3KV_ERR_INVALID_ARG      # q_chunk 0
    assert at(4096, 256, ctypes.byref(st), 64, 100, 0.0, 4096, None) == b.H3KV_ERR_INVALID_ARG   # kv_block % 128
    assert at(4096, 256, ctypes.byref(_store_f8(head_dim=64)), 64, 0, 0.0, 4096, None) == b.H3KV_ERR_UNSUPPORTED
    assert at(4104, 256, ctypes.byref(st), 64, 0, 0.0, 4096, None) == b.H3KV_ERR_INVALID_ARG     # misaligned Q
    assert at(4096, 256, ctypes.byref(st), 64, 0, 0.0, 0, None) == b.H3KV_ERR_INVALID_ARG        # null O
    assert at(4096, 256, ctypes.byref(_store_f8(seq=0)), 64, 0, 0.0, 4096, None) == b.H3KV_ERR_INVALID_ARG
    assert at(4096, 0, ctypes.byref(st), 64, 0, 0.0, 4096, None) == b.H3KV_OK


def test_hostio_checks():
    assert b.h3kv_hostio_scratch_bytes(32, 16384) == 2 * 32 * 16384 * 128 * 6 + 256
    assert b.h3kv_hostio_scratch_bytes(1, 0) == 0 and b.h3kv_hostio_scratch_bytes(-1, 10) == 0
    st = _store()
    hi = b.h3kv_attend_hostio
    need = b.h3kv_hostio_scratch_bytes(1, 64)
    assert hi(4096, 256, ctypes.byref(st), 64, 0, 0.0, 4096, 4096, need - 1, None) == b.H3KV_ERR_INVALID_ARG
    assert hi(4096, 256, ctypes.byref(st), 64, 0, 0.0, 4096, 0, need, None) == b.H3KV_ERR_INVALID_ARG
    assert hi(4096, 256, ctypes.byref(st), 64, 0, 0.0, 4096, 4100, need, None) == b.H3KV_ERR_INVALID_ARG
    assert hi(0, 256, ctypes.byref(st), 64, 0, 0.0, 4096, 4096, need, None) == b.H3KV_ERR_INVALID_ARG
    assert hi(4096, 256, ctypes.byref(st), 0, 0, 0.0, 4096, 4096, need, None) == b.H3KV_ERR_INVALID_ARG
    assert hi(4096, 0, ctypes.byref(st), 64, 0, 0.0, 4096, 4096, need, None) == b.H3KV_OK


def test_store_fp4_sizes():
    # 0.5625 byte per element: 64 code bytes and 8 scale bytes per 128 values
    assert b.h3kv_store_fp4_bytes(32, 217088, 128) == 2 * 32 * 217088 * 72
    assert b.h3kv_store_fp4_bytes(1, 77, 128) == 2 * 77 * 72
    assert b.h3kv_store_fp4_bytes(1, 10, 64) == 0 and b.h3kv_store_fp4_bytes(-1, 10, 128) == 0


def _store_fp4(heads=1, seq=256, ptr=4096, head_dim=128):
    return b.h3kv_store_fp4(ptr, ptr, ptr, ptr, heads, seq, head_dim)


def test_build_store_fp4_rejects_bad_arguments():
    st = _store_fp4()
    bs = b.h3kv_build_store_fp4
    assert bs(4096, 4096, 1, 256, 128, None, None) == b.H3KV_ERR_INVALID_ARG
    assert bs(4096, 4096, 1, 256, 64, ctypes.byref(st), None) == b.H3KV_ERR_UNSUPPORTED
    assert bs(4096, 4096, 2, 256, 128, ctypes.byref(st), None) == b.H3KV_ERR_INVALID_ARG   # shape mismatch
    assert bs(0, 4096, 1, 256, 128, ctypes.byref(st), None) == b.H3KV_ERR_INVALID_ARG      # null K
    assert bs(4096, 4100, 1, 256, 128, ctypes.byref(st), None) == b.H3KV_ERR_INVALID_ARG   # misaligned V
    assert bs(4096, 4096, 1, 256, 128, ctypes.byref(_store_fp4(ptr=0)), None) == b.H3KV_ERR_INVALID_ARG
    big = _store_fp4(heads=1 << 20, seq=1 << 12)
    assert bs(4096, 4096, 1 << 20, 1 << 12, 128, ctypes.byref(big), None) == b.H3KV_ERR_INVALID_ARG  # rows
    assert bs(0, 0, 0, 0, 128, ctypes.byref(_store_fp4(heads=0, seq=0, ptr=0)), None) == b.H3KV_OK


def test_attend_fp4_rejects_bad_arguments():
    st = _store_fp4()
    at = b.h3kv_attend_fp4
    assert at(4096, 256, None, 256, 0, 0.0, 4096, None) == b.H3KV_ERR_INVALID_ARG
    assert at(4096, 256, ctypes.byref(st), 0, 0, 0.0, 4096, None) == b.H3KV_ERR_INVALID_ARG      # q_chunk 0
    assert at(4096, 256, ctypes.byref(st), 64, 100, 0.0, 4096, None) == b.H3KV_ERR_INVALID_ARG   # kv_block % 128
    assert at(4096, 256, ctypes.byref(_store_fp4(head_dim=64)), 64, 0, 0.0, 4096, None) == b.H3KV_ERR_UNSUPPORTED
    assert at(4104, 256, ctypes.byref(st), 64, 0, 0.0, 4096, None) == b.H3KV_ERR_INVALID_ARG     # misaligned Q
    assert at(4096, 256, ctypes.byref(st), 64, 0, 0.0, 0, None) == b.H3KV_ERR_INVALID_ARG        # null O
    assert at(4096, 256, ctypes.byref(_store_fp4(seq=0)), 64, 0, 0.0, 4096, None) == b.H3KV_ERR_INVALID_ARG
    assert at(4096, 0, ctypes.byref(st), 64, 0, 0.0, 4096, None) == b.H3KV_OK


def test_attention_rejects_more_than_65535_heads():
    # one grid row per head: more heads than a grid dimension holds is an
    # argument error on the host, not a failed launch
    H = 65536
    st = b.h3kv_store(4096, 4096, 4096, 4096, H, 16, 128, 0)
    assert b.h3kv_attend(4096, 16, ctypes.byref(st), 16, 0, 0.0, 4096, None) == b.H3KV_ERR_INVALID_ARG
    assert b.h3kv_attend_exact(4096, 16, 4096, 4096, H, 16, 128, 16, 0, 0.0, 4096, None) == b.H3KV_ERR_INVALID_ARG
    big = b.h3kv_staging_bytes(H, 128)
    assert b.h3kv_attend_staged(4096, 16, ctypes.byref(st), 16, 128, 0.0, 4096, 4096, big, 4096,
                                None) == b.H3KV_ERR_INVALID_ARG
    need = b.h3kv_hostio_scratch_bytes(H, 16)
    assert b.h3kv_attend_hostio(4096, 16, ctypes.byref(st), 16, 0, 0.0, 4096, 4096, need,
                                None) == b.H3KV_ERR_INVALID_ARG
    st4 = b.h3kv_store_fp4(4096, 4096, 4096, 4096, H, 16, 128)
    assert b.h3kv_attend_fp4(4096, 16, ctypes.byref(st4), 16, 0, 0.0, 4096, None) == b.H3KV_ERR_INVALID_ARG
    st8 = b.h3kv_store_f8(4096, 4096, 4096, 4096, 4096, H, 16, 128)
    assert b.h3kv_attend_f8(4096, 16, ctypes.byref(st8), 16, 0, 0.0, 4096, None) == b.H3KV_ERR_INVALID_ARG


def test_tmem_selftest_rejects_null_before_device_work():
    # the argument check comes before the device query, so no GPU is needed
    assert b.h3kv_selftest_tmem_ld_max(None, None) == b.H3KV_ERR_INVALID_ARG


def test_attend_launch_count():
    # head by head (heads x chunks launches) with more than one head, at least
    # 131072 keys and at least 16 CTAs (256 rows each) per head and chunk;
    # otherwise one launch per chunk over all heads
    n = b.h3kv_attend_launch_count
    assert n(217088, 217088, 32, 16384) == 32 * 14
    assert n(217088, 217088, 32, 4096) == 32 * 53
    assert n(217088, 217088, 32, 3841) == 32 * 57   # 16 CTAs per chunk
    assert n(217088, 217088, 32, 3840) == 57        # 15 CTAs per chunk
    assert n(217088, 131072, 32, 16384) == 32 * 14  # the shortest head-major key count
    assert n(217088, 131071, 32, 16384) == 14
    assert n(65536, 65536, 32, 16384) == 4          # shorter sequences: chunk by chunk
    assert n(3000, 300000, 1, 256) == 12            # one head: chunk by chunk
    assert n(0, 217088, 8, 256) == 0
    assert n(100, 217088, 8, 0) == 0
