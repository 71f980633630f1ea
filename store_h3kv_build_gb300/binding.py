"""Thin Python binding over ``libh3kv.so`` (the C ABI in ``include/h3kv.h``).

Argument marshalling only: torch tensors are used for device memory and the
current CUDA stream, their pointers and sizes go through ctypes, and every
step of the computation runs in the library's CUDA kernels.  Importing this
module loads the library and raises ImportError if it has not been built
(``python -m store_h3kv_build_gb300.build_lib``); there is no fallback.
"""
from __future__ import annotations

import contextlib
import ctypes
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libh3kv.so")
if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python -m store_h3kv_build_gb300.build_lib`")
_lib = ctypes.CDLL(LIB_PATH)

HEAD_DIM = 128
DEFAULT_KV_BLOCK = 16384
KV_TILE = 128
H3KV_STATIC_SCRATCH_BYTES = 32 * 1024 * 1024  # the fixed scratch of h3kv_attend_staged_static

H3KV_OK = 0
H3KV_ERR_INVALID_ARG = 1
H3KV_ERR_UNSUPPORTED = 2
H3KV_ERR_CUDA = 3
H3KV_ERR_DEVICE_TIMEOUT = 4


class h3kv_store(ctypes.Structure):  # noqa: N801 - mirrors the C struct name
    _fields_ = [
        ("k_codes", ctypes.c_void_p),
        ("v_codes", ctypes.c_void_p),
        ("k_scales", ctypes.c_void_p),
        ("v_scales", ctypes.c_void_p),
        ("heads", ctypes.c_int32),
        ("seq", ctypes.c_int64),
        ("head_dim", ctypes.c_int32),
        ("scale_group", ctypes.c_int32),
    ]


class h3kv_store_f8(ctypes.Structure):  # noqa: N801 - mirrors the C struct name
    _fields_ = [
        ("k_codes", ctypes.c_void_p),
        ("v_codes_t", ctypes.c_void_p),
        ("k_scales", ctypes.c_void_p),
        ("v_scales", ctypes.c_void_p),
        ("k_mean", ctypes.c_void_p),
        ("heads", ctypes.c_int32),
        ("seq", ctypes.c_int64),
        ("head_dim", ctypes.c_int32),
    ]


class h3kv_store_fp4(ctypes.Structure):  # noqa: N801 - mirrors the C struct name
    _fields_ = [
        ("k_codes", ctypes.c_void_p),
        ("v_codes", ctypes.c_void_p),
        ("k_scales", ctypes.c_void_p),
        ("v_scales", ctypes.c_void_p),
        ("heads", ctypes.c_int32),
        ("seq", ctypes.c_int64),
        ("head_dim", ctypes.c_int32),
    ]


_vp, _i32, _i64, _f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
_SIGS = {
    "h3kv_abi_version": (ctypes.c_uint32, []),
    "h3kv_store_bytes": (ctypes.c_size_t, [_i32, _i64, _i32]),
    "h3kv_build_store": (ctypes.c_int, [_vp, _vp, _i32, _i64, _i32, ctypes.POINTER(h3kv_store), _vp]),
    "h3kv_attend": (ctypes.c_int, [_vp, _i64, ctypes.POINTER(h3kv_store), _i32, _i32, _f32, _vp, _vp]),
    "h3kv_attend_exact": (ctypes.c_int, [_vp, _i64, _vp, _vp, _i32, _i64, _i32, _i32, _i32, _f32, _vp, _vp]),
    "h3kv_sync_status": (ctypes.c_int, [_vp]),
    "h3kv_staging_bytes": (ctypes.c_size_t, [_i32, _i32]),
    "h3kv_attend_staged_static": (ctypes.c_int, [_vp, _i64, ctypes.POINTER(h3kv_store), _i32, _i32, _f32, _vp,
                                                 _vp]),
    "h3kv_attend_staged": (ctypes.c_int, [_vp, _i64, ctypes.POINTER(h3kv_store), _i32, _i32, _f32, _vp, _vp,
                                          ctypes.c_size_t, _vp, _vp]),
    "h3kv_hostio_scratch_bytes": (ctypes.c_size_t, [_i32, _i32]),
    "h3kv_attend_hostio": (ctypes.c_int, [_vp, _i64, ctypes.POINTER(h3kv_store), _i32, _i32, _f32, _vp, _vp,
                                          ctypes.c_size_t, _vp]),
    "h3kv_f8_v_stride": (ctypes.c_int64, [_i64]),
    "h3kv_store_f8_bytes": (ctypes.c_size_t, [_i32, _i64, _i32]),
    "h3kv_build_store_f8": (ctypes.c_int, [_vp, _vp, _i32, _i64, _i32, ctypes.POINTER(h3kv_store_f8), _vp]),
    "h3kv_attend_f8": (ctypes.c_int, [_vp, _i64, ctypes.POINTER(h3kv_store_f8), _i32, _i32, _f32, _vp, _vp]),
    "h3kv_store_fp4_bytes": (ctypes.c_size_t, [_i32, _i64, _i32]),
    "h3kv_build_store_fp4": (ctypes.c_int, [_vp, _vp, _i32, _i64, _i32, ctypes.POINTER(h3kv_store_fp4), _vp]),
    "h3kv_attend_fp4": (ctypes.c_int, [_vp, _i64, ctypes.POINTER(h3kv_store_fp4), _i32, _i32, _f32, _vp, _vp]),
    "h3kv_set_wait_timeout_ns": (ctypes.c_int, [ctypes.c_uint64]),
    "h3kv_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_uint64, _vp]),
    "h3kv_selftest_tmem_ld_max": (ctypes.c_int, [ctypes.POINTER(ctypes.c_int32), _vp]),
    "h3kv_attend_launch_count": (ctypes.c_int64, [ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32]),
    "h3kv_debug_withhold_p": (ctypes.c_int, [ctypes.c_int32]),
    "h3kv_strerror": (ctypes.c_char_p, [ctypes.c_int]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args
    globals()[_name] = _fn

EXPORTED = tuple(_SIGS)


class H3kvError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {h3kv_strerror(status).decode()} (status {status})")


def check(status: int, where: str = "h3kv") -> None:
    if status != H3KV_OK:
        raise H3kvError(status, where)


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def _need(t, name: str, dtype, shape=None) -> None:
    """Argument check: the library reads and writes raw contiguous buffers of
    the sizes its arguments imply, so a strided view, another dtype or a
    buffer of another shape would be read as garbage or written past its end."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(int(x) for x in shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(int(x) for x in shape)}")


def _need_rows(t, name: str, heads: int | None = None) -> None:
    """bf16 [heads, rows, 128] input (Q, K or V)."""
    _need(t, name, torch.bfloat16)
    if t.dim() != 3 or t.shape[2] != HEAD_DIM:
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected [heads, rows, {HEAD_DIM}]")
    if heads is not None and t.shape[0] != heads:
        raise ValueError(f"{name}: {t.shape[0]} heads, the store has {heads}")


def _need_out(out, Q) -> None:
    _need(out, "out", torch.float32, Q.shape)


def _stream(stream=None) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _on(stream=None):
    """Context for the device tensors the binding allocates for a call
    (outputs, stores, scratch): the call's stream, so that PyTorch's caching
    allocator hands a freed block to new work only after that stream's work
    on it -- a scratch dropped when the call returns is still in use there."""
    return torch.cuda.stream(stream) if stream is not None else contextlib.nullcontext()


class Store:
    """A kvi8r store held in torch tensors: int8 codes [heads, seq, 128] and
    fp16 scales [heads, seq] for K and for V."""

    def __init__(self, k_codes, v_codes, k_scales, v_scales):
        self.k_codes, self.v_codes = k_codes, v_codes
        self.k_scales, self.v_scales = k_scales, v_scales
        self.heads, self.seq = int(k_codes.shape[0]), int(k_codes.shape[1])
        # [heads, seq] scales: one per row; [heads, seq, 4]: one per 32 values
        self.scale_group = 32 if k_scales.dim() == 3 else 0

    @classmethod
    def empty(cls, heads: int, seq: int, device="cuda", host: bool = False, scale_group: int = 0) -> "Store":
        """Uninitialised store buffers.  ``host=True`` places them in pinned
        host memory: on a Grace-Blackwell node the kernels read (and the
        store build writes) them directly over NVLink-C2C, so the whole
        sequence's K/V need not occupy HBM."""
        if host:
            kw = dict(pin_memory=True)
        else:
            kw = dict(device=device)
        # every buffer allocated with its own pin_memory request: empty_like
        # of a pinned tensor is pageable, and h3kv_attend_staged refuses a
        # store with pageable buffers
        sshape = (heads, seq, HEAD_DIM // 32) if scale_group == 32 else (heads, seq)
        kc, vc = (torch.empty((heads, seq, HEAD_DIM), dtype=torch.int8, **kw) for _ in range(2))
        ks, vs = (torch.empty(sshape, dtype=torch.float16, **kw) for _ in range(2))
        return cls(kc, vc, ks, vs)

    @property
    def in_host_memory(self) -> bool:
        return not self.k_codes.is_cuda

    def c_struct(self) -> h3kv_store:
        H, L = self.heads, self.seq
        _need(self.k_codes, "store.k_codes", torch.int8, (H, L, HEAD_DIM))
        _need(self.v_codes, "store.v_codes", torch.int8, (H, L, HEAD_DIM))
        sshape = (H, L, HEAD_DIM // 32) if self.scale_group == 32 else (H, L)
        _need(self.k_scales, "store.k_scales", torch.float16, sshape)
        _need(self.v_scales, "store.v_scales", torch.float16, sshape)
        return h3kv_store(_ptr(self.k_codes), _ptr(self.v_codes), _ptr(self.k_scales), _ptr(self.v_scales),
                          self.heads, self.seq, HEAD_DIM, self.scale_group)

    def nbytes(self) -> int:
        return int(h3kv_store_bytes(self.heads, self.seq, HEAD_DIM))


def build_store(K: torch.Tensor, V: torch.Tensor, out: Store | None = None, stream=None,
                scale_group: int = 0) -> Store:
    """h3kv_build_store on bf16 K, V [heads, seq, 128] (CUDA, contiguous);
    scale_group 32 gives one scale per 32 rotated values."""
    _need_rows(K, "K")
    _need_rows(V, "V")
    if V.shape != K.shape:
        raise ValueError(f"V: shape {tuple(V.shape)}, K has {tuple(K.shape)}")
    heads, seq = int(K.shape[0]), int(K.shape[1])
    with _on(stream):
        out = Store.empty(heads, seq, K.device, scale_group=scale_group) if out is None else out
    st = out.c_struct()
    check(h3kv_build_store(_ptr(K), _ptr(V), heads, seq, int(K.shape[2]), ctypes.byref(st), _stream(stream)),
          "h3kv_build_store")
    return out


def attend(Q: torch.Tensor, store: Store, q_chunk: int = 16384, kv_block: int = 0, softmax_scale: float = 0.0,
           out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """h3kv_attend: kvi8r attention of bf16 Q [heads, q_seq, 128] over `store`
    -> fp32 [heads, q_seq, 128]."""
    _need_rows(Q, "Q", store.heads)
    q_seq = int(Q.shape[1])
    with _on(stream):
        out = torch.empty(Q.shape, dtype=torch.float32, device=Q.device) if out is None else out
    _need_out(out, Q)
    st = store.c_struct()
    check(h3kv_attend(_ptr(Q), q_seq, ctypes.byref(st), int(q_chunk), int(kv_block), float(softmax_scale),
                      _ptr(out), _stream(stream)), "h3kv_attend")
    return out


def staging_bytes_double(heads: int, kv_block: int) -> int:
    """Staging bytes with room for two kv_blocks (h3kv_attend_staged then
    copies the next block while attending the current one)."""
    need = int(h3kv_staging_bytes(int(heads), int(kv_block)))
    return (need + 255) // 256 * 256 + need


def attend_staged(Q: torch.Tensor, store: Store, q_chunk: int = 16384, kv_block: int = 0,
                  softmax_scale: float = 0.0, out: torch.Tensor | None = None, staging: torch.Tensor | None = None,
                  state: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """h3kv_attend_staged: kvi8r attention over a store held outside HBM (e.g.
    ``Store.empty(..., host=True)``), staged through HBM one kv_block at a
    time.  ``staging`` (uint8, >= h3kv_staging_bytes; with
    ``staging_bytes_double`` bytes two blocks are staged and the next block's
    copy overlaps the current block's attention) and ``state`` (fp32 [heads,
    q_seq, 2]) are device scratch; they are created here if not given (the
    staging with room for two blocks)."""
    _need_rows(Q, "Q", store.heads)
    dev = Q.device
    heads, q_seq = int(Q.shape[0]), int(Q.shape[1])
    with _on(stream):
        out = torch.empty(Q.shape, dtype=torch.float32, device=dev) if out is None else out
        if staging is None:
            staging = torch.empty(max(staging_bytes_double(store.heads, int(kv_block)), 16), dtype=torch.uint8,
                                  device=dev)
        if state is None:
            state = torch.empty((heads, q_seq, 2), dtype=torch.float32, device=dev)
    _need_out(out, Q)
    _need(staging, "staging", torch.uint8)
    _need(state, "state", torch.float32, (int(Q.shape[0]), int(Q.shape[1]), 2))
    st = store.c_struct()
    check(h3kv_attend_staged(_ptr(Q), q_seq, ctypes.byref(st), int(q_chunk), int(kv_block), float(softmax_scale),
                             _ptr(out), _ptr(staging), staging.numel() * staging.element_size(), _ptr(state),
                             _stream(stream)), "h3kv_attend_staged")
    return out


def attend_hostio(Q_host: torch.Tensor, store: Store, q_chunk: int = 16384, kv_block: int = 0,
                  softmax_scale: float = 0.0, out: torch.Tensor | None = None, scratch: torch.Tensor | None = None,
                  stream=None) -> torch.Tensor:
    """h3kv_attend_hostio: kvi8r attention of bf16 Q in (pinned) host memory
    over a device store, streamed through HBM per query chunk; the fp32
    output lands in host memory (``out``, pinned, created here if not
    given).  ``scratch`` (uint8 device, >= h3kv_hostio_scratch_bytes) is
    created here if not given."""
    _need_rows(Q_host, "Q_host", store.heads)
    heads, q_seq = int(Q_host.shape[0]), int(Q_host.shape[1])
    if out is None:
        out = torch.empty(Q_host.shape, dtype=torch.float32, pin_memory=True)
    if scratch is None:
        dev = store.k_codes.device
        with _on(stream):
            scratch = torch.empty(max(int(h3kv_hostio_scratch_bytes(heads, int(q_chunk))), 16), dtype=torch.uint8,
                                  device=dev)
    _need_out(out, Q_host)
    _need(scratch, "scratch", torch.uint8)
    st = store.c_struct()
    check(h3kv_attend_hostio(_ptr(Q_host), q_seq, ctypes.byref(st), int(q_chunk), int(kv_block),
                             float(softmax_scale), _ptr(out), _ptr(scratch), scratch.numel(), _stream(stream)),
          "h3kv_attend_hostio")
    return out


def attend_exact(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, q_chunk: int = 16384, kv_block: int = 0,
                 softmax_scale: float = 0.0, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """h3kv_attend_exact: softmax attention on bf16 Q, K, V -> fp32."""
    _need_rows(K, "K")
    _need_rows(V, "V")
    if V.shape != K.shape:
        raise ValueError(f"V: shape {tuple(V.shape)}, K has {tuple(K.shape)}")
    _need_rows(Q, "Q", int(K.shape[0]))
    with _on(stream):
        out = torch.empty(Q.shape, dtype=torch.float32, device=Q.device) if out is None else out
    _need_out(out, Q)
    check(h3kv_attend_exact(_ptr(Q), int(Q.shape[1]), _ptr(K), _ptr(V), int(K.shape[0]), int(K.shape[1]),
                            int(K.shape[2]), int(q_chunk), int(kv_block), float(softmax_scale), _ptr(out),
                            _stream(stream)), "h3kv_attend_exact")
    return out


K_BLOCK_F8 = 64


class StoreF8:
    """A kvf8s store held in torch tensors: e4m3 K codes [heads, seq, 128]
    (uint8), channel-major e4m3 V codes [heads, 128, v_stride], fp32 K block
    scales [heads, ceil(seq / 64)], fp32 V channel scales and K means
    [heads, 128]."""

    def __init__(self, k_codes, v_codes_t, k_scales, v_scales, k_mean, seq: int):
        self.k_codes, self.v_codes_t = k_codes, v_codes_t
        self.k_scales, self.v_scales, self.k_mean = k_scales, v_scales, k_mean
        self.heads, self.seq = int(k_codes.shape[0]), int(seq)

    @classmethod
    def empty(cls, heads: int, seq: int, device="cuda") -> "StoreF8":
        vstride = int(h3kv_f8_v_stride(seq))
        nblk = (seq + K_BLOCK_F8 - 1) // K_BLOCK_F8
        kc = torch.empty((heads, seq, HEAD_DIM), dtype=torch.uint8, device=device)
        vt = torch.empty((heads, HEAD_DIM, vstride), dtype=torch.uint8, device=device)
        ks = torch.empty((heads, nblk), dtype=torch.float32, device=device)
        vs = torch.empty((heads, HEAD_DIM), dtype=torch.float32, device=device)
        km = torch.empty((heads, HEAD_DIM), dtype=torch.float32, device=device)
        return cls(kc, vt, ks, vs, km, seq)

    def c_struct(self) -> h3kv_store_f8:
        H, L = self.heads, self.seq
        _need(self.k_codes, "store.k_codes", torch.uint8, (H, L, HEAD_DIM))
        _need(self.v_codes_t, "store.v_codes_t", torch.uint8, (H, HEAD_DIM, int(h3kv_f8_v_stride(L))))
        _need(self.k_scales, "store.k_scales", torch.float32, (H, (L + K_BLOCK_F8 - 1) // K_BLOCK_F8))
        _need(self.v_scales, "store.v_scales", torch.float32, (H, HEAD_DIM))
        _need(self.k_mean, "store.k_mean", torch.float32, (H, HEAD_DIM))
        return h3kv_store_f8(_ptr(self.k_codes), _ptr(self.v_codes_t), _ptr(self.k_scales), _ptr(self.v_scales),
                             _ptr(self.k_mean), self.heads, self.seq, HEAD_DIM)

    def nbytes(self) -> int:
        return int(h3kv_store_f8_bytes(self.heads, self.seq, HEAD_DIM))


def build_store_f8(K: torch.Tensor, V: torch.Tensor, out: StoreF8 | None = None, stream=None) -> StoreF8:
    """h3kv_build_store_f8 on bf16 K, V [heads, seq, 128] (CUDA, contiguous)."""
    _need_rows(K, "K")
    _need_rows(V, "V")
    if V.shape != K.shape:
        raise ValueError(f"V: shape {tuple(V.shape)}, K has {tuple(K.shape)}")
    heads, seq = int(K.shape[0]), int(K.shape[1])
    with _on(stream):
        out = StoreF8.empty(heads, seq, K.device) if out is None else out
    st = out.c_struct()
    check(h3kv_build_store_f8(_ptr(K), _ptr(V), heads, seq, int(K.shape[2]), ctypes.byref(st), _stream(stream)),
          "h3kv_build_store_f8")
    return out


def attend_f8(Q: torch.Tensor, store: StoreF8, q_chunk: int = 16384, kv_block: int = 0, softmax_scale: float = 0.0,
              out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """h3kv_attend_f8: kvf8s attention of bf16 Q [heads, q_seq, 128] -> fp32."""
    _need_rows(Q, "Q", store.heads)
    q_seq = int(Q.shape[1])
    with _on(stream):
        out = torch.empty(Q.shape, dtype=torch.float32, device=Q.device) if out is None else out
    _need_out(out, Q)
    st = store.c_struct()
    check(h3kv_attend_f8(_ptr(Q), q_seq, ctypes.byref(st), int(q_chunk), int(kv_block), float(softmax_scale),
                         _ptr(out), _stream(stream)), "h3kv_attend_f8")
    return out


class StoreFp4:
    """A kvfp4 store held in torch tensors: packed e2m1 codes [heads, seq, 64]
    (uint8, element 2i in the low nibble of byte i) and e4m3 block scales
    [heads, seq, 8] (uint8) for K and for V."""

    def __init__(self, k_codes, v_codes, k_scales, v_scales):
        self.k_codes, self.v_codes = k_codes, v_codes
        self.k_scales, self.v_scales = k_scales, v_scales
        self.heads, self.seq = int(k_codes.shape[0]), int(k_codes.shape[1])

    @classmethod
    def empty(cls, heads: int, seq: int, device="cuda") -> "StoreFp4":
        kc = torch.empty((heads, seq, HEAD_DIM // 2), dtype=torch.uint8, device=device)
        ks = torch.empty((heads, seq, HEAD_DIM // 16), dtype=torch.uint8, device=device)
        return cls(kc, torch.empty_like(kc), ks, torch.empty_like(ks))

    def c_struct(self) -> h3kv_store_fp4:
        H, L = self.heads, self.seq
        _need(self.k_codes, "store.k_codes", torch.uint8, (H, L, HEAD_DIM // 2))
        _need(self.v_codes, "store.v_codes", torch.uint8, (H, L, HEAD_DIM // 2))
        _need(self.k_scales, "store.k_scales", torch.uint8, (H, L, HEAD_DIM // 16))
        _need(self.v_scales, "store.v_scales", torch.uint8, (H, L, HEAD_DIM // 16))
        return h3kv_store_fp4(_ptr(self.k_codes), _ptr(self.v_codes), _ptr(self.k_scales), _ptr(self.v_scales),
                              self.heads, self.seq, HEAD_DIM)

    def nbytes(self) -> int:
        return int(h3kv_store_fp4_bytes(self.heads, self.seq, HEAD_DIM))


def build_store_fp4(K: torch.Tensor, V: torch.Tensor, out: StoreFp4 | None = None, stream=None) -> StoreFp4:
    """h3kv_build_store_fp4 on bf16 K, V [heads, seq, 128] (CUDA, contiguous)."""
    _need_rows(K, "K")
    _need_rows(V, "V")
    if V.shape != K.shape:
        raise ValueError(f"V: shape {tuple(V.shape)}, K has {tuple(K.shape)}")
    heads, seq = int(K.shape[0]), int(K.shape[1])
    with _on(stream):
        out = StoreFp4.empty(heads, seq, K.device) if out is None else out
    st = out.c_struct()
    check(h3kv_build_store_fp4(_ptr(K), _ptr(V), heads, seq, int(K.shape[2]), ctypes.byref(st), _stream(stream)),
          "h3kv_build_store_fp4")
    return out


def attend_fp4(Q: torch.Tensor, store: StoreFp4, q_chunk: int = 16384, kv_block: int = 0,
               softmax_scale: float = 0.0, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """h3kv_attend_fp4: kvfp4 attention of bf16 Q [heads, q_seq, 128] -> fp32."""
    _need_rows(Q, "Q", store.heads)
    q_seq = int(Q.shape[1])
    with _on(stream):
        out = torch.empty(Q.shape, dtype=torch.float32, device=Q.device) if out is None else out
    _need_out(out, Q)
    st = store.c_struct()
    check(h3kv_attend_fp4(_ptr(Q), q_seq, ctypes.byref(st), int(q_chunk), int(kv_block), float(softmax_scale),
                          _ptr(out), _stream(stream)), "h3kv_attend_fp4")
    return out


def sync_status(stream=None) -> None:
    """Synchronise the stream and raise if a kernel recorded a wait timeout."""
    check(h3kv_sync_status(_stream(stream)), "h3kv_sync_status")
