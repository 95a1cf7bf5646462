"""Python binding of libmoeroute: the C ABI of ``include/moeroute.h`` under the
same names, argument marshalling only.

Every function takes torch CUDA tensors (contiguous; raw bytes are what
counts, so bf16 data may be ``torch.bfloat16`` or any 2-byte dtype, fp8
payload ``torch.uint8`` or ``torch.float8_e4m3fn``), checks that each buffer
is large enough for the shape, and passes its device pointer and the current
torch stream (or ``stream=``) to the library.  The activations ``x`` and the
combined output ``out`` may instead be pinned host tensors: the kernels then
read and write them directly over the CPU-GPU link.  All work runs in the library's
CUDA kernels; there is no other implementation to fall back on, and importing
a function without the built library raises.

``MoeBuffers`` owns one set of device buffers for a shape (PyTorch is the
allocator) and strings the calls together for callers who want the whole
path:  ``dispatch`` = moe_dispatch (or route_count, exchange, dispatch_send,
dispatch_recv);  ``combine`` = moe_combine (or combine_send, combine_recv).
"""
from __future__ import annotations

import ctypes
import functools
import os
import threading

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoeroute.so")
_lock = threading.Lock()
_lib = None

MOE_OK, MOE_EINVAL, MOE_ENOTSUP, MOE_ECUDA = 0, -1, -2, -3
MOE_ST_BAD_EXPERT, MOE_ST_CAPACITY, MOE_ST_TIMEOUT = 1, 2, 4

EXPORTS = ("moe_sizes_query", "moe_route_count", "moe_exchange", "moe_route", "moe_dispatch_send",
           "moe_dispatch_recv", "moe_combine_send", "moe_combine_recv", "moe_dispatch",
           "moe_dispatch_send_recv", "moe_dispatch_signalled", "moe_dispatch_signalled_static",
           "moe_combine", "moe_combine_partial_send", "moe_combine_partial_recv",
           "moe_combine_partial", "moe_expert_standin",
           "moe_e4m3_encode", "moe_dispatch_ll", "moe_expert_standin_ll", "moe_combine_ll",
           "moe_strerror", "moe_version")


class moe_shape(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int), ("T", ctypes.c_int), ("E", ctypes.c_int),
                ("R", ctypes.c_int), ("H", ctypes.c_int), ("cap", ctypes.c_int)]


_SIZE_FIELDS = ("cap", "send_rows", "bytes_x", "bytes_topk_idx", "bytes_expert_count",
                "bytes_send_off", "bytes_expert_send_off", "bytes_grp_off", "bytes_seg_off",
                "bytes_m_sizes", "bytes_send_q", "bytes_send_s", "bytes_send_tok", "bytes_grp_q",
                "bytes_grp_s", "bytes_grp_src", "bytes_y", "ll_rows", "bytes_ll_q",
                "bytes_ll_s", "bytes_ll_src", "bytes_ll_count", "bytes_ll_y", "bytes_sig",
                "bytes_part")


class moe_sizes(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in _SIZE_FIELDS]


_BUFFER_FIELDS = ("topk_idx", "topk_w", "x", "expert_count", "send_off", "expert_send_off",
                  "slot_row", "grp_off", "seg_off", "csend_off", "m_sizes", "send_q", "send_s",
                  "send_tok", "grp_q", "grp_s", "grp_src", "y", "csend", "out", "status")


class moe_buffers(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _BUFFER_FIELDS]


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {strerror(code)} (code {code})")


def library_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded libmoeroute.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(f"{_LIB_PATH} is not built: run __graft_entry__.build() or "
                                   "python -m combine_expert_count_gb300.build")
            h = ctypes.CDLL(_LIB_PATH)
            V, I, P = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER
            sp = P(moe_shape)
            h.moe_sizes_query.argtypes = [sp, P(moe_sizes)]
            h.moe_route_count.argtypes = [sp] + [V] * 6 + [V]
            h.moe_exchange.argtypes = [sp] + [V] * 7 + [V]
            h.moe_route.argtypes = [sp] + [V] * 10 + [V]
            h.moe_dispatch.argtypes = [sp, P(moe_buffers), V]
            h.moe_dispatch_send_recv.argtypes = [sp, P(moe_buffers), V]
            h.moe_dispatch_signalled.argtypes = [sp, P(moe_buffers), V, V]
            h.moe_dispatch_signalled_static.argtypes = [sp, P(moe_buffers), V]
            h.moe_combine_partial_send.argtypes = [sp] + [V] * 7 + [V]
            h.moe_combine_partial_recv.argtypes = [sp] + [V] * 4 + [V]
            h.moe_combine_partial.argtypes = [sp, P(moe_buffers), V, V]
            h.moe_combine.argtypes = [sp, P(moe_buffers), V]
            h.moe_dispatch_send.argtypes = [sp] + [V] * 6 + [V]
            h.moe_dispatch_recv.argtypes = [sp] + [V] * 10 + [V]
            h.moe_combine_send.argtypes = [sp] + [V] * 8 + [V]
            h.moe_combine_recv.argtypes = [sp] + [V] * 8 + [V]
            h.moe_expert_standin.argtypes = [sp, I] + [V] * 4 + [V]
            h.moe_e4m3_encode.argtypes = [V, V, ctypes.c_int64, V]
            h.moe_dispatch_ll.argtypes = [sp] + [V] * 8 + [V]
            h.moe_expert_standin_ll.argtypes = [sp, I] + [V] * 4 + [V]
            h.moe_combine_ll.argtypes = [sp] + [V] * 5 + [V]
            h.moe_strerror.argtypes = [I]
            h.moe_strerror.restype = ctypes.c_char_p
            h.moe_version.argtypes = []
            for name in EXPORTS:
                if name != "moe_strerror":
                    getattr(h, name).restype = ctypes.c_int
            _lib = h
    return _lib


def strerror(code: int) -> str:
    try:
        return lib().moe_strerror(int(code)).decode()
    except RuntimeError:
        return f"code {code}"


def make_shape(N: int, T: int, E: int, R: int, H: int, cap: int = 0) -> moe_shape:
    return moe_shape(N, T, E, R, H, cap)


def _as_shape(shape) -> moe_shape:
    if isinstance(shape, moe_shape):
        return shape
    return moe_shape(shape.N, shape.T, shape.E, shape.R, shape.H, int(getattr(shape, "cap", 0)))


def _shape_key(sh: moe_shape) -> tuple:
    return (sh.N, sh.T, sh.E, sh.R, sh.H, sh.cap)


@functools.lru_cache(maxsize=256)
def _sizes_cached(key: tuple) -> moe_sizes:
    out = moe_sizes()
    sh = moe_shape(*key)
    rc = lib().moe_sizes_query(ctypes.byref(sh), ctypes.byref(out))
    if rc != MOE_OK:
        raise MoeError(rc, "moe_sizes_query")
    return out


def sizes_query(shape) -> moe_sizes:
    """Buffer sizes for a shape (the library's answer, cached per shape)."""
    return _sizes_cached(_shape_key(_as_shape(shape)))


moe_sizes_query = sizes_query


# Buffers that may live in pinned host memory: the kernels read x and write
# out directly over the CPU-GPU link (zero copy).
_HOST_OK = ("x", "out", "out_bf16")


def _p(t: torch.Tensor | None, nbytes: int, name: str):
    if t is None:
        if nbytes:
            raise ValueError(f"{name}: buffer of {nbytes} bytes required")
        return None
    if not t.is_cuda and not (name in _HOST_OK and t.is_pinned()):
        raise ValueError(f"{name}: must be a CUDA tensor"
                         + (" or pinned host memory" if name in _HOST_OK else ""))
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if t.numel() * t.element_size() < nbytes:
        raise ValueError(f"{name}: {t.numel() * t.element_size()} bytes < {nbytes} required")
    return ctypes.c_void_p(t.data_ptr())


def _s(stream) -> ctypes.c_void_p:
    st = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(st.cuda_stream)


def _check(rc: int, where: str) -> None:
    if rc != MOE_OK:
        raise MoeError(rc, where)


def moe_route_count(shape, topk_idx, expert_count, send_off, expert_send_off, slot_row, status,
                    stream=None) -> None:
    sh, z = _as_shape(shape), sizes_query(shape)
    _check(lib().moe_route_count(
        ctypes.byref(sh), _p(topk_idx, z.bytes_topk_idx, "topk_idx"),
        _p(expert_count, z.bytes_expert_count, "expert_count"),
        _p(send_off, z.bytes_send_off, "send_off"),
        _p(expert_send_off, z.bytes_expert_send_off, "expert_send_off"),
        _p(slot_row, z.bytes_topk_idx, "slot_row"), _p(status, 4, "status"), _s(stream)),
        "moe_route_count")


def moe_exchange(shape, expert_count, send_off, grp_off, seg_off, csend_off, m_sizes, status,
                 stream=None) -> None:
    sh, z = _as_shape(shape), sizes_query(shape)
    _check(lib().moe_exchange(
        ctypes.byref(sh), _p(expert_count, z.bytes_expert_count, "expert_count"),
        _p(send_off, z.bytes_send_off, "send_off"), _p(grp_off, z.bytes_grp_off, "grp_off"),
        _p(seg_off, z.bytes_seg_off, "seg_off"), _p(csend_off, z.bytes_send_off, "csend_off"),
        _p(m_sizes, z.bytes_m_sizes, "m_sizes"), _p(status, 4, "status"), _s(stream)),
        "moe_exchange")


def moe_route(shape, topk_idx, expert_count, send_off, expert_send_off, slot_row, grp_off,
              seg_off, csend_off, m_sizes, status, stream=None) -> None:
    sh, z = _as_shape(shape), sizes_query(shape)
    _check(lib().moe_route(
        ctypes.byref(sh), _p(topk_idx, z.bytes_topk_idx, "topk_idx"),
        _p(expert_count, z.bytes_expert_count, "expert_count"),
        _p(send_off, z.bytes_send_off, "send_off"),
        _p(expert_send_off, z.bytes_expert_send_off, "expert_send_off"),
        _p(slot_row, z.bytes_topk_idx, "slot_row"), _p(grp_off, z.bytes_grp_off, "grp_off"),
        _p(seg_off, z.bytes_seg_off, "seg_off"), _p(csend_off, z.bytes_send_off, "csend_off"),
        _p(m_sizes, z.bytes_m_sizes, "m_sizes"), _p(status, 4, "status"), _s(stream)),
        "moe_route")


def moe_dispatch_send(shape, x, slot_row, send_q, send_s, send_tok, status, stream=None) -> None:
    sh, z = _as_shape(shape), sizes_query(shape)
    _check(lib().moe_dispatch_send(
        ctypes.byref(sh), _p(x, z.bytes_x, "x"), _p(slot_row, z.bytes_topk_idx, "slot_row"),
        _p(send_q, z.bytes_send_q, "send_q"), _p(send_s, z.bytes_send_s, "send_s"),
        _p(send_tok, z.bytes_send_tok, "send_tok"), _p(status, 4, "status"), _s(stream)),
        "moe_dispatch_send")


def moe_dispatch_recv(shape, send_q, send_s, send_tok, expert_count, expert_send_off, seg_off,
                      grp_q, grp_s, grp_src, status, stream=None) -> None:
    sh, z = _as_shape(shape), sizes_query(shape)
    _check(lib().moe_dispatch_recv(
        ctypes.byref(sh), _p(send_q, z.bytes_send_q, "send_q"),
        _p(send_s, z.bytes_send_s, "send_s"), _p(send_tok, z.bytes_send_tok, "send_tok"),
        _p(expert_count, z.bytes_expert_count, "expert_count"),
        _p(expert_send_off, z.bytes_expert_send_off, "expert_send_off"),
        _p(seg_off, z.bytes_seg_off, "seg_off"), _p(grp_q, z.bytes_grp_q, "grp_q"),
        _p(grp_s, z.bytes_grp_s, "grp_s"), _p(grp_src, z.bytes_grp_src, "grp_src"),
        _p(status, 4, "status"), _s(stream)),
        "moe_dispatch_recv")


def moe_combine_send(shape, y, expert_count, expert_send_off, send_off, seg_off, csend_off, csend,
                     status, stream=None) -> None:
    sh, z = _as_shape(shape), sizes_query(shape)
    _check(lib().moe_combine_send(
        ctypes.byref(sh), _p(y, z.bytes_y, "y"),
        _p(expert_count, z.bytes_expert_count, "expert_count"),
        _p(expert_send_off, z.bytes_expert_send_off, "expert_send_off"),
        _p(send_off, z.bytes_send_off, "send_off"), _p(seg_off, z.bytes_seg_off, "seg_off"),
        _p(csend_off, z.bytes_send_off, "csend_off"), _p(csend, z.bytes_y, "csend"),
        _p(status, 4, "status"), _s(stream)),
        "moe_combine_send")


def moe_combine_recv(shape, csend, topk_idx, topk_w, slot_row, send_off, csend_off, out, status,
                     stream=None) -> None:
    sh, z = _as_shape(shape), sizes_query(shape)
    _check(lib().moe_combine_recv(
        ctypes.byref(sh), _p(csend, z.bytes_y, "csend"),
        _p(topk_idx, z.bytes_topk_idx, "topk_idx"), _p(topk_w, z.bytes_topk_idx, "topk_w"),
        _p(slot_row, z.bytes_topk_idx, "slot_row"), _p(send_off, z.bytes_send_off, "send_off"),
        _p(csend_off, z.bytes_send_off, "csend_off"), _p(out, z.bytes_x, "out"),
        _p(status, 4, "status"), _s(stream)),
        "moe_combine_recv")


_DISPATCH_NEEDS = {"topk_idx": "bytes_topk_idx", "x": "bytes_x",
                   "expert_count": "bytes_expert_count", "send_off": "bytes_send_off",
                   "expert_send_off": "bytes_expert_send_off", "slot_row": "bytes_topk_idx",
                   "grp_off": "bytes_grp_off", "seg_off": "bytes_seg_off",
                   "csend_off": "bytes_send_off", "m_sizes": "bytes_m_sizes",
                   "send_q": "bytes_send_q", "send_s": "bytes_send_s",
                   "send_tok": "bytes_send_tok", "grp_q": "bytes_grp_q", "grp_s": "bytes_grp_s",
                   "grp_src": "bytes_grp_src"}
_COMBINE_NEEDS = {"topk_idx": "bytes_topk_idx", "topk_w": "bytes_topk_idx", "y": "bytes_y",
                  "expert_send_off": "bytes_expert_send_off", "send_off": "bytes_send_off",
                  "slot_row": "bytes_topk_idx", "seg_off": "bytes_seg_off",
                  "csend_off": "bytes_send_off", "csend": "bytes_y", "out": "bytes_x"}


def _buffers(z: moe_sizes, tensors: dict, needs: dict) -> moe_buffers:
    b = moe_buffers()
    for name in _BUFFER_FIELDS:
        t = tensors.get(name)
        nbytes = 4 if name == "status" else getattr(z, needs[name]) if name in needs else 0
        if name in needs or name == "status" or t is not None:
            p = _p(t, nbytes, name)
            setattr(b, name, p.value if p is not None else None)
    return b


def moe_dispatch(shape, tensors: dict, stream=None) -> None:
    """Whole dispatch in one call; ``tensors`` maps moe_buffers field names
    (x, topk_idx, routing arrays, send and grouped buffers, status) to tensors."""
    sh, z = _as_shape(shape), sizes_query(shape)
    b = _buffers(z, tensors, _DISPATCH_NEEDS)
    _check(lib().moe_dispatch(ctypes.byref(sh), ctypes.byref(b), _s(stream)), "moe_dispatch")


def moe_dispatch_send_recv(shape, tensors: dict, stream=None) -> None:
    """Quantise + pack + receive shuffle in one kernel (routing arrays given)."""
    sh, z = _as_shape(shape), sizes_query(shape)
    b = _buffers(z, tensors, _DISPATCH_NEEDS)
    _check(lib().moe_dispatch_send_recv(ctypes.byref(sh), ctypes.byref(b), _s(stream)),
           "moe_dispatch_send_recv")


def moe_dispatch_signalled(shape, tensors: dict, sig, stream=None) -> None:
    """Whole dispatch (as moe_dispatch) with the send and the receive shuffle
    in one kernel that hands rows over by per-(sender, receiver) flags;
    ``sig`` is the zeroed int32 scratch of ``bytes_sig`` bytes."""
    sh, z = _as_shape(shape), sizes_query(shape)
    b = _buffers(z, tensors, _DISPATCH_NEEDS)
    _check(lib().moe_dispatch_signalled(ctypes.byref(sh), ctypes.byref(b),
                                        _p(sig, z.bytes_sig, "sig"), _s(stream)),
           "moe_dispatch_signalled")


def moe_dispatch_signalled_static(shape, tensors: dict, stream=None) -> None:
    """moe_dispatch_signalled with the library's own static flag scratch (no
    allocation; N <= 64; calls on one device must not overlap in time)."""
    sh, z = _as_shape(shape), sizes_query(shape)
    b = _buffers(z, tensors, _DISPATCH_NEEDS)
    _check(lib().moe_dispatch_signalled_static(ctypes.byref(sh), ctypes.byref(b), _s(stream)),
           "moe_dispatch_signalled_static")


def moe_combine(shape, tensors: dict, stream=None) -> None:
    """Whole combine in one call; ``tensors`` as for moe_dispatch (y, topk_idx,
    topk_w, routing arrays, csend, out, status)."""
    sh, z = _as_shape(shape), sizes_query(shape)
    b = _buffers(z, tensors, _COMBINE_NEEDS)
    _check(lib().moe_combine(ctypes.byref(sh), ctypes.byref(b), _s(stream)), "moe_combine")


def moe_combine_partial_send(shape, y, topk_idx, topk_w, slot_row, expert_send_off, seg_off, part,
                             stream=None) -> None:
    sh, z = _as_shape(shape), sizes_query(shape)
    _check(lib().moe_combine_partial_send(
        ctypes.byref(sh), _p(y, z.bytes_y, "y"), _p(topk_idx, z.bytes_topk_idx, "topk_idx"),
        _p(topk_w, z.bytes_topk_idx, "topk_w"), _p(slot_row, z.bytes_topk_idx, "slot_row"),
        _p(expert_send_off, z.bytes_expert_send_off, "expert_send_off"),
        _p(seg_off, z.bytes_seg_off, "seg_off"), _p(part, z.bytes_part, "part"), _s(stream)),
        "moe_combine_partial_send")


def moe_combine_partial_recv(shape, part, topk_idx, slot_row, out, stream=None) -> None:
    sh, z = _as_shape(shape), sizes_query(shape)
    _check(lib().moe_combine_partial_recv(
        ctypes.byref(sh), _p(part, z.bytes_part, "part"),
        _p(topk_idx, z.bytes_topk_idx, "topk_idx"), _p(slot_row, z.bytes_topk_idx, "slot_row"),
        _p(out, z.bytes_x, "out"), _s(stream)),
        "moe_combine_partial_recv")


_PARTIAL_NEEDS = {"topk_idx": "bytes_topk_idx", "topk_w": "bytes_topk_idx", "y": "bytes_y",
                  "expert_send_off": "bytes_expert_send_off", "slot_row": "bytes_topk_idx",
                  "seg_off": "bytes_seg_off", "out": "bytes_x"}


def moe_combine_partial(shape, tensors: dict, part, stream=None) -> None:
    """Combine with send-side reduction in one pass; ``part`` receives the
    partial rows [N][N][T][H] (bf16)."""
    sh, z = _as_shape(shape), sizes_query(shape)
    b = _buffers(z, tensors, _PARTIAL_NEEDS)
    _check(lib().moe_combine_partial(ctypes.byref(sh), ctypes.byref(b),
                                     _p(part, z.bytes_part, "part"), _s(stream)),
           "moe_combine_partial")


def moe_expert_standin(shape, mode: int, grp_q, grp_s, grp_off, y, stream=None) -> None:
    sh, z = _as_shape(shape), sizes_query(shape)
    _check(lib().moe_expert_standin(
        ctypes.byref(sh), int(mode), _p(grp_q, z.bytes_grp_q, "grp_q"),
        _p(grp_s, z.bytes_grp_s, "grp_s"), _p(grp_off, z.bytes_grp_off, "grp_off"),
        _p(y, z.bytes_y, "y"), _s(stream)),
        "moe_expert_standin")


def moe_e4m3_encode(v, out, stream=None) -> None:
    n = v.numel()
    _check(lib().moe_e4m3_encode(_p(v, 4 * n, "v"), _p(out, n, "out"), n, _s(stream)),
           "moe_e4m3_encode")


def moe_dispatch_ll(shape, x, topk_idx, ll_q, ll_s, ll_src, ll_count, ll_row, status,
                    stream=None) -> None:
    sh, z = _as_shape(shape), sizes_query(shape)
    _check(lib().moe_dispatch_ll(
        ctypes.byref(sh), _p(x, z.bytes_x, "x"), _p(topk_idx, z.bytes_topk_idx, "topk_idx"),
        _p(ll_q, z.bytes_ll_q, "ll_q"), _p(ll_s, z.bytes_ll_s, "ll_s"),
        _p(ll_src, z.bytes_ll_src, "ll_src"), _p(ll_count, z.bytes_ll_count, "ll_count"),
        _p(ll_row, z.bytes_topk_idx, "ll_row"), _p(status, 4, "status"), _s(stream)),
        "moe_dispatch_ll")


def moe_expert_standin_ll(shape, mode: int, ll_q, ll_s, ll_count, y_ll, stream=None) -> None:
    sh, z = _as_shape(shape), sizes_query(shape)
    _check(lib().moe_expert_standin_ll(
        ctypes.byref(sh), int(mode), _p(ll_q, z.bytes_ll_q, "ll_q"), _p(ll_s, z.bytes_ll_s, "ll_s"),
        _p(ll_count, z.bytes_ll_count, "ll_count"), _p(y_ll, z.bytes_ll_y, "y_ll"), _s(stream)),
        "moe_expert_standin_ll")


def moe_combine_ll(shape, y_ll, topk_w, ll_row, out, status, stream=None) -> None:
    sh, z = _as_shape(shape), sizes_query(shape)
    _check(lib().moe_combine_ll(
        ctypes.byref(sh), _p(y_ll, z.bytes_ll_y, "y_ll"), _p(topk_w, z.bytes_topk_idx, "topk_w"),
        _p(ll_row, z.bytes_topk_idx, "ll_row"), _p(out, z.bytes_x, "out"),
        _p(status, 4, "status"), _s(stream)),
        "moe_combine_ll")


class MoeLLBuffers:
    """Device buffers of the low-latency layout for one shape (see
    include/moeroute.h): ``dispatch`` = moe_dispatch_ll, ``expert`` =
    moe_expert_standin_ll, ``combine`` = moe_combine_ll."""

    def __init__(self, N: int, T: int, E: int, R: int, H: int,
                 device: str | torch.device = "cuda"):
        self.shape = make_shape(N, T, E, R, H)
        self.sizes = sizes_query(self.shape)
        self.N, self.T, self.E, self.R, self.H = N, T, E, R, H
        rows, Er = int(self.sizes.ll_rows), E // N
        d = torch.device(device)
        self.status = torch.zeros(1, dtype=torch.int32, device=d)
        self.ll_q = torch.empty((rows, H), dtype=torch.uint8, device=d)
        self.ll_s = torch.empty((rows, H // 128), dtype=torch.float32, device=d)
        self.ll_src = torch.empty(rows, dtype=torch.int32, device=d)
        self.ll_count = torch.empty((N, Er, N), dtype=torch.int32, device=d)
        self.ll_row = torch.empty((N, T, R), dtype=torch.int32, device=d)
        self.y_ll = torch.empty((rows, H), dtype=torch.bfloat16, device=d)
        self.out = torch.empty((N, T, H), dtype=torch.bfloat16, device=d)

    def dispatch(self, x, topk_idx, stream=None) -> None:
        moe_dispatch_ll(self.shape, x, topk_idx, self.ll_q, self.ll_s, self.ll_src,
                        self.ll_count, self.ll_row, self.status, stream)

    def expert(self, mode: int = 0, stream=None) -> None:
        moe_expert_standin_ll(self.shape, mode, self.ll_q, self.ll_s, self.ll_count, self.y_ll,
                              stream)

    def combine(self, topk_w, out=None, stream=None) -> torch.Tensor:
        out = self.out if out is None else out
        moe_combine_ll(self.shape, self.y_ll, topk_w, self.ll_row, out, self.status, stream)
        return out


class MoeBuffers:
    """Device buffers for one shape, allocated once with torch and reused.

    Attribute names and layouts are those of ``include/moeroute.h``.
    """

    def __init__(self, N: int, T: int, E: int, R: int, H: int, cap: int = 0,
                 device: str | torch.device = "cuda"):
        self.shape = make_shape(N, T, E, R, H, cap)
        z = sizes_query(self.shape)
        self.sizes = z
        self.cap = int(z.cap)
        self.N, self.T, self.E, self.R, self.H = N, T, E, R, H
        Er, Sb, cap_ = E // N, H // 128, self.cap
        d = torch.device(device)

        def e(shape, dtype):
            return torch.empty(shape, dtype=dtype, device=d)

        self.status = torch.zeros(1, dtype=torch.int32, device=d)
        self.expert_count = e((N, E), torch.int32)
        self.send_off = e((N, N + 1), torch.int32)
        self.expert_send_off = e((N, E + 1), torch.int32)
        self.slot_row = e((N, T, R), torch.int32)
        self.grp_off = e((N, Er + 1), torch.int32)
        self.seg_off = e((N, Er, N), torch.int32)
        self.csend_off = e((N, N + 1), torch.int32)
        self.m_sizes = e((N, Er), torch.int32)
        self.send_q = e((N, T * R, H), torch.uint8)
        self.send_s = e((N, T * R, Sb), torch.float32)
        self.send_tok = e((N, T * R), torch.int32)
        self.grp_q = e((N, cap_, H), torch.uint8)
        self.grp_s = e((N, cap_, Sb), torch.float32)
        self.grp_src = e((N, cap_, 2), torch.int32)
        self.y = e((N, cap_, H), torch.bfloat16)
        self.csend = e((N, cap_, H), torch.bfloat16)
        self.out = e((N, T, H), torch.bfloat16)
        # moe_dispatch_signalled's group counters and flags (zero between calls)
        self.sig = torch.zeros(int(z.bytes_sig) // 4, dtype=torch.int32, device=d)

    def partial_rows(self) -> torch.Tensor:
        """The send-side reduction's partial rows [N][N][T][H] bf16, allocated
        on first use."""
        if not hasattr(self, "part"):
            N, T, H = self.N, self.T, self.H
            self.part = torch.empty((N, N, T, H), dtype=torch.bfloat16, device=self.out.device)
        return self.part

    def device_bytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in vars(self).values()
                   if isinstance(t, torch.Tensor))

    def route(self, topk_idx, stream=None, fused: bool = True) -> None:
        """Counts, offsets and slots: one ``moe_route`` launch, or
        ``moe_route_count`` then ``moe_exchange`` with ``fused=False``."""
        if fused:
            moe_route(self.shape, topk_idx, self.expert_count, self.send_off,
                      self.expert_send_off, self.slot_row, self.grp_off, self.seg_off,
                      self.csend_off, self.m_sizes, self.status, stream)
            return
        moe_route_count(self.shape, topk_idx, self.expert_count, self.send_off,
                        self.expert_send_off, self.slot_row, self.status, stream)
        moe_exchange(self.shape, self.expert_count, self.send_off, self.grp_off, self.seg_off,
                     self.csend_off, self.m_sizes, self.status, stream)

    def tensors(self, **extra) -> dict:
        """This object's buffers by moe_buffers field name, plus ``extra``."""
        d = {n: getattr(self, n) for n in _BUFFER_FIELDS if hasattr(self, n)}
        d.update(extra)
        return d

    def _struct(self, need: dict, **inputs) -> moe_buffers:
        """moe_buffers with this object's buffers (checked once) and the
        per-call inputs (checked on every call)."""
        if not hasattr(self, "_b"):
            self._b = _buffers(self.sizes, self.tensors(), {})  # sized by construction
        b = moe_buffers.from_buffer_copy(self._b)
        for name, t in inputs.items():
            p = _p(t, getattr(self.sizes, need[name]), name)
            setattr(b, name, p.value if p is not None else None)
        return b

    def dispatch(self, x, topk_idx, stream=None, calls: str = "fused") -> None:
        """The dispatch half.  ``calls``: "fused" (one moe_dispatch call),
        "signalled" (one moe_dispatch_signalled call), "fused_route"
        (moe_route then the two dispatch calls) or "separate" (the four calls
        of the pages' steps)."""
        if calls == "fused":
            b = self._struct(_DISPATCH_NEEDS, x=x, topk_idx=topk_idx)
            _check(lib().moe_dispatch(ctypes.byref(self.shape), ctypes.byref(b), _s(stream)),
                   "moe_dispatch")
            return
        if calls == "signalled":
            b = self._struct(_DISPATCH_NEEDS, x=x, topk_idx=topk_idx)
            _check(lib().moe_dispatch_signalled(ctypes.byref(self.shape), ctypes.byref(b),
                                                ctypes.c_void_p(self.sig.data_ptr()),
                                                _s(stream)),
                   "moe_dispatch_signalled")
            return
        self.route(topk_idx, stream, calls == "fused_route")
        moe_dispatch_send(self.shape, x, self.slot_row, self.send_q, self.send_s, self.send_tok,
                          self.status, stream)
        moe_dispatch_recv(self.shape, self.send_q, self.send_s, self.send_tok, self.expert_count,
                          self.expert_send_off, self.seg_off, self.grp_q, self.grp_s,
                          self.grp_src, self.status, stream)

    def expert(self, mode: int = 0, stream=None) -> None:
        """The grouped-GEMM stand-in (identity or per-expert scale)."""
        moe_expert_standin(self.shape, mode, self.grp_q, self.grp_s, self.grp_off, self.y, stream)

    def combine(self, topk_idx, topk_w, y=None, out=None, stream=None,
                calls: str = "fused") -> torch.Tensor:
        """The combine half; returns ``out``.  ``calls``: "fused" (one
        moe_combine call), "partial" (one moe_combine_partial call: send-side
        reduction), "partial_separate" (moe_combine_partial_send then
        moe_combine_partial_recv) or anything else for moe_combine_send then
        moe_combine_recv."""
        out = self.out if out is None else out
        if calls in ("partial", "partial_separate"):
            part = self.partial_rows()
            if calls == "partial":
                b = self._struct(_PARTIAL_NEEDS, topk_idx=topk_idx, topk_w=topk_w,
                                 y=self.y if y is None else y, out=out)
                _check(lib().moe_combine_partial(ctypes.byref(self.shape), ctypes.byref(b),
                                                 ctypes.c_void_p(part.data_ptr()), _s(stream)),
                       "moe_combine_partial")
            else:
                moe_combine_partial_send(self.shape, self.y if y is None else y, topk_idx, topk_w,
                                         self.slot_row, self.expert_send_off, self.seg_off, part,
                                         stream)
                moe_combine_partial_recv(self.shape, part, topk_idx, self.slot_row, out, stream)
            return out
        if calls == "fused":
            b = self._struct(_COMBINE_NEEDS, topk_idx=topk_idx, topk_w=topk_w,
                             y=self.y if y is None else y, out=out)
            _check(lib().moe_combine(ctypes.byref(self.shape), ctypes.byref(b), _s(stream)),
                   "moe_combine")
            return out
        moe_combine_send(self.shape, self.y if y is None else y, self.expert_count,
                         self.expert_send_off, self.send_off, self.seg_off, self.csend_off,
                         self.csend, self.status, stream)
        moe_combine_recv(self.shape, self.csend, topk_idx, topk_w, self.slot_row, self.send_off,
                         self.csend_off, out, self.status, stream)
        return out
