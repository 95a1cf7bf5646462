"""Python front end of the CPU oracle (``oracle/moe_ref.c``).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg use this; the product path never does.  It imports nothing
from the CUDA package.  Arrays are numpy, bf16 values are uint16 bit patterns.

Every function below marshals numpy arrays into one C function of the oracle;
the arithmetic is all in ``moe_ref.c``.  Parity status of each function (what
pins it to something other than itself) is listed in ``tests/test_oracle.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_ref.c")
_LIB = os.path.join(_HERE, "libmoe_ref.so")
_CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]

ST_BAD_EXPERT = 1
ST_CAPACITY = 2

# Output buffers start filled with these patterns, so a row the oracle never
# writes cannot pass for zeros.
FILL_U8 = 0xA5
FILL_U16 = 0x7FA5     # a bf16 NaN
FILL_F32 = np.float32(np.nan)

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into ``oracle/libmoe_ref.so``."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *_CFLAGS, _SRC, "-lm", "-o", tmp], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _P(t):
    return ctypes.POINTER(t)


_i32p, _u8p, _u16p, _f32p, _f64p = (_P(ctypes.c_int32), _P(ctypes.c_uint8), _P(ctypes.c_uint16),
                                   _P(ctypes.c_float), _P(ctypes.c_double))
_I = ctypes.c_int

_SIGS = {
    "ref_bf16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
    "ref_f32_to_bf16_rn": (ctypes.c_uint16, [ctypes.c_float]),
    "ref_e4m3_encode": (ctypes.c_uint8, [ctypes.c_float]),
    "ref_e4m3_decode": (ctypes.c_double, [ctypes.c_uint8]),
    "ref_f32_to_bf16_array": (None, [_f32p, _u16p, ctypes.c_int64]),
    "ref_e4m3_encode_array": (None, [_f32p, _u8p, ctypes.c_int64]),
    "ref_e4m3_decode_array": (None, [_u8p, _f64p, ctypes.c_int64]),
    "ref_route_count": (_I, [_I, _I, _I, _I, _i32p, _i32p, _i32p, _i32p, _i32p]),
    "ref_exchange": (_I, [_I, _I, _I, _i32p, _i32p, _i32p, _i32p, _i32p, _i32p]),
    "ref_quant_token": (None, [_I, _u16p, _u8p, _f32p]),
    "ref_dispatch_send": (None, [_I, _I, _I, _I, _u16p, _i32p, _u8p, _f32p, _i32p]),
    "ref_dispatch_recv": (None, [_I, _I, _I, _I, _I, _I, _u8p, _f32p, _i32p, _i32p, _i32p,
                                 _i32p, _u8p, _f32p, _i32p]),
    "ref_standin_row": (None, [_I, _I, _I, _u8p, _f32p, _u16p]),
    "ref_expert_standin": (None, [_I, _I, _I, _I, _I, _u8p, _f32p, _i32p, _u16p]),
    "ref_combine_send": (None, [_I, _I, _I, _I, _I, _I, _u16p, _i32p, _i32p, _i32p, _i32p,
                                _i32p, _u16p]),
    "ref_weighted_sum": (None, [_I, _I, _u16p, _f32p, _i32p, _u16p]),
    "ref_combine_recv": (None, [_I, _I, _I, _I, _I, _I, _u16p, _i32p, _f32p, _i32p, _i32p,
                                _i32p, _u16p]),
    "ref_combine_partial_send": (None, [_I, _I, _I, _I, _I, _I, _u16p, _i32p, _f32p, _i32p,
                                        _i32p, _i32p, _u16p]),
    "ref_combine_partial_recv": (None, [_I, _I, _I, _I, _I, _u16p, _i32p, _i32p, _u16p]),
}


def lib():
    global _lib
    with _lock:
        if _lib is None:
            handle = ctypes.CDLL(build())
            for name, (res, args) in _SIGS.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _i32(a):
    return _ptr(a, ctypes.c_int32)


def _u8(a):
    return _ptr(a, ctypes.c_uint8)


def _u16(a):
    return _ptr(a, ctypes.c_uint16)


def _f32(a):
    return _ptr(a, ctypes.c_float)


# ------------------------------------------------------------------ numbers

def e4m3_encode(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    lib().ref_e4m3_encode_array(_f32(v), _u8(out), v.size)
    return out


def e4m3_decode(c: np.ndarray) -> np.ndarray:
    c = np.ascontiguousarray(c, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    lib().ref_e4m3_decode_array(_u8(c), _ptr(out, ctypes.c_double), c.size)
    return out


def f32_to_bf16_array(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint16)
    lib().ref_f32_to_bf16_array(_f32(v), _u16(out), v.size)
    return out


def f32_to_bf16(v: float) -> int:
    return int(lib().ref_f32_to_bf16_rn(ctypes.c_float(v)))


def bf16_to_f32(b: int) -> float:
    return float(lib().ref_bf16_to_f32(ctypes.c_uint16(b)))


# ------------------------------------------------------------------ steps

def route_count(N: int, T: int, E: int, R: int, topk_idx: np.ndarray) -> dict:
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32).reshape(N, T, R)
    cnt = np.zeros((N, E), np.int32)
    send_off = np.zeros((N, N + 1), np.int32)
    eso = np.zeros((N, E + 1), np.int32)
    slot = np.zeros((N, T, R), np.int32)
    st = lib().ref_route_count(N, T, E, R, _i32(idx), _i32(cnt), _i32(send_off), _i32(eso),
                               _i32(slot))
    return dict(expert_count=cnt, send_off=send_off, expert_send_off=eso, slot_row=slot,
                status=int(st))


def exchange(N: int, E: int, cap: int, expert_count: np.ndarray, send_off: np.ndarray) -> dict:
    Er = E // N
    grp_off = np.zeros((N, Er + 1), np.int32)
    seg_off = np.zeros((N, Er, N), np.int32)
    csend_off = np.zeros((N, N + 1), np.int32)
    m_sizes = np.zeros((N, Er), np.int32)
    st = lib().ref_exchange(N, E, cap, _i32(np.ascontiguousarray(expert_count)),
                            _i32(np.ascontiguousarray(send_off)), _i32(grp_off), _i32(seg_off),
                            _i32(csend_off), _i32(m_sizes))
    return dict(grp_off=grp_off, seg_off=seg_off, csend_off=csend_off, m_sizes=m_sizes,
                status=int(st))


def quant_token(H: int, x_row: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    xr = np.ascontiguousarray(x_row, dtype=np.uint16).reshape(H)
    q = np.empty(H, np.uint8)
    sc = np.empty(H // 128, np.float32)
    lib().ref_quant_token(H, _u16(xr), _u8(q), _f32(sc))
    return q, sc


def dispatch_send(N: int, T: int, R: int, H: int, x: np.ndarray, slot_row: np.ndarray) -> dict:
    x = np.ascontiguousarray(x, dtype=np.uint16).reshape(N, T, H)
    slot_row = np.ascontiguousarray(slot_row, dtype=np.int32)
    send_q = np.full((N, T * R, H), FILL_U8, np.uint8)
    send_s = np.full((N, T * R, H // 128), FILL_F32, np.float32)
    send_tok = np.full((N, T * R), -1, np.int32)
    lib().ref_dispatch_send(N, T, R, H, _u16(x), _i32(slot_row), _u8(send_q), _f32(send_s),
                            _i32(send_tok))
    return dict(send_q=send_q, send_s=send_s, send_tok=send_tok)


def dispatch_recv(N, T, E, R, H, cap, send_q, send_s, send_tok, expert_count, expert_send_off,
                  seg_off) -> dict:
    grp_q = np.full((N, cap, H), FILL_U8, np.uint8)
    grp_s = np.full((N, cap, H // 128), FILL_F32, np.float32)
    grp_src = np.full((N, cap, 2), -1, np.int32)
    c = np.ascontiguousarray
    lib().ref_dispatch_recv(N, T, E, R, H, cap, _u8(c(send_q)), _f32(c(send_s)),
                            _i32(c(send_tok)), _i32(c(expert_count)), _i32(c(expert_send_off)),
                            _i32(c(seg_off)), _u8(grp_q), _f32(grp_s), _i32(grp_src))
    return dict(grp_q=grp_q, grp_s=grp_s, grp_src=grp_src)


def standin_row(H: int, mode: int, e: int, q: np.ndarray, scales: np.ndarray) -> np.ndarray:
    y = np.empty(H, np.uint16)
    lib().ref_standin_row(H, mode, e, _u8(np.ascontiguousarray(q, dtype=np.uint8)),
                          _f32(np.ascontiguousarray(scales, dtype=np.float32)), _u16(y))
    return y


def expert_standin(N, E, H, cap, mode, grp_q, grp_s, grp_off) -> np.ndarray:
    y = np.full((N, cap, H), FILL_U16, np.uint16)
    c = np.ascontiguousarray
    lib().ref_expert_standin(N, E, H, cap, mode, _u8(c(grp_q)), _f32(c(grp_s)),
                             _i32(c(grp_off)), _u16(y))
    return y


def combine_send(N, T, E, R, H, cap, y, expert_count, expert_send_off, send_off, seg_off,
                 csend_off) -> np.ndarray:
    csend = np.full((N, cap, H), FILL_U16, np.uint16)
    c = np.ascontiguousarray
    lib().ref_combine_send(N, T, E, R, H, cap, _u16(c(y)), _i32(c(expert_count)),
                           _i32(c(expert_send_off)), _i32(c(send_off)), _i32(c(seg_off)),
                           _i32(c(csend_off)), _u16(csend))
    return csend


def weighted_sum(rows: np.ndarray, w: np.ndarray, use: np.ndarray | None = None) -> np.ndarray:
    rows = np.ascontiguousarray(rows, dtype=np.uint16)
    R, H = rows.shape
    use = np.ones(R, np.int32) if use is None else np.ascontiguousarray(use, dtype=np.int32)
    out = np.empty(H, np.uint16)
    lib().ref_weighted_sum(R, H, _u16(rows), _f32(np.ascontiguousarray(w, dtype=np.float32)),
                           _i32(use), _u16(out))
    return out


def combine_recv(N, T, E, R, H, cap, csend, topk_idx, topk_w, slot_row, send_off,
                 csend_off) -> np.ndarray:
    out = np.full((N, T, H), FILL_U16, np.uint16)
    c = np.ascontiguousarray
    lib().ref_combine_recv(N, T, E, R, H, cap, _u16(c(csend)), _i32(c(topk_idx)),
                           _f32(c(topk_w, dtype=np.float32)), _i32(c(slot_row)),
                           _i32(c(send_off)), _i32(c(csend_off)), _u16(out))
    return out


def combine_partial_send(N, T, E, R, H, cap, y, topk_idx, topk_w, slot_row, expert_send_off,
                         seg_off) -> np.ndarray:
    """Send-side reduction: one bf16 partial row per (expert rank, sender,
    token); rows never written keep the fill pattern."""
    part = np.full((N, N, T, H), FILL_U16, np.uint16)
    c = np.ascontiguousarray
    lib().ref_combine_partial_send(N, T, E, R, H, cap, _u16(c(y)), _i32(c(topk_idx)),
                                   _f32(c(topk_w, dtype=np.float32)), _i32(c(slot_row)),
                                   _i32(c(expert_send_off)), _i32(c(seg_off)), _u16(part))
    return part


def combine_partial_recv(N, T, E, R, H, part, topk_idx, slot_row) -> np.ndarray:
    out = np.full((N, T, H), FILL_U16, np.uint16)
    c = np.ascontiguousarray
    lib().ref_combine_partial_recv(N, T, E, R, H, _u16(c(part)), _i32(c(topk_idx)),
                                   _i32(c(slot_row)), _u16(out))
    return out


# ------------------------------------------------------------------ a whole layer

def layer(N, T, E, R, H, cap, x, topk_idx, topk_w, mode: int = 0) -> dict:
    """All steps in the pages' order: count, scan, quantise + pack, exchange,
    receive shuffle, expert stand-in, combine send, combine receive."""
    out = route_count(N, T, E, R, topk_idx)
    st = out["status"]
    out.update(exchange(N, E, cap, out["expert_count"], out["send_off"]))
    out["status"] = st | out["status"]
    out.update(dispatch_send(N, T, R, H, x, out["slot_row"]))
    out.update(dispatch_recv(N, T, E, R, H, cap, out["send_q"], out["send_s"], out["send_tok"],
                             out["expert_count"], out["expert_send_off"], out["seg_off"]))
    out["y"] = expert_standin(N, E, H, cap, mode, out["grp_q"], out["grp_s"], out["grp_off"])
    out["csend"] = combine_send(N, T, E, R, H, cap, out["y"], out["expert_count"],
                                out["expert_send_off"], out["send_off"], out["seg_off"],
                                out["csend_off"])
    out["out"] = combine_recv(N, T, E, R, H, cap, out["csend"], topk_idx, topk_w,
                              out["slot_row"], out["send_off"], out["csend_off"])
    return out


class LayerTimer:
    """The six steps of one layer timed on preallocated arrays, for the
    benchmark's CPU baseline: route_count, exchange, dispatch_send and
    dispatch_recv (the dispatch), combine_send and combine_recv (the
    combine).  The routing and the expert stand-in run once when the timer is
    built (the stand-in is not a timed step; its output is the same every
    step, as on the GPU), the grouped buffers hold exactly the rows the
    routing sends to the busiest rank, and no output array is allocated or
    filled inside a timed step."""

    def __init__(self, N, T, E, R, H, x, topk_idx, topk_w, mode: int = 0):
        self.N, self.T, self.E, self.R, self.H = N, T, E, R, H
        Er, Sb = E // N, H // 128
        # private copies: the caller's arrays are never written
        self.x = np.array(x, dtype=np.uint16, order="C").reshape(N, T, H)
        self.idx = np.array(topk_idx, dtype=np.int32, order="C").reshape(N, T, R)
        self.w = np.array(topk_w, dtype=np.float32, order="C").reshape(N, T, R)
        inputs = (self.x, self.idx, self.w)
        rc = route_count(N, T, E, R, self.idx)
        ex = exchange(N, E, 1 << 30, rc["expert_count"], rc["send_off"])
        self.cap = cap = max(1, int(ex["grp_off"][:, -1].max()))
        z = np.zeros
        self.cnt, self.send_off = z((N, E), np.int32), z((N, N + 1), np.int32)
        self.eso, self.slot = z((N, E + 1), np.int32), z((N, T, R), np.int32)
        self.grp_off, self.seg_off = z((N, Er + 1), np.int32), z((N, Er, N), np.int32)
        self.csend_off, self.m_sizes = z((N, N + 1), np.int32), z((N, Er), np.int32)
        self.send_q, self.send_s = z((N, T * R, H), np.uint8), z((N, T * R, Sb), np.float32)
        self.send_tok = z((N, T * R), np.int32)
        self.grp_q, self.grp_s = z((N, cap, H), np.uint8), z((N, cap, Sb), np.float32)
        self.grp_src = z((N, cap, 2), np.int32)
        self.csend, self.out = z((N, cap, H), np.uint16), z((N, T, H), np.uint16)
        for a in vars(self).values():   # touch every output page once, outside any timed step
            if isinstance(a, np.ndarray) and not any(a is i for i in inputs):
                a.fill(0)
        self.dispatch()
        self.y = expert_standin(N, E, H, cap, mode, self.grp_q, self.grp_s, self.grp_off)

    def dispatch(self) -> None:
        L, N, T, E, R, H, cap = lib(), self.N, self.T, self.E, self.R, self.H, self.cap
        L.ref_route_count(N, T, E, R, _i32(self.idx), _i32(self.cnt), _i32(self.send_off),
                          _i32(self.eso), _i32(self.slot))
        L.ref_exchange(N, E, cap, _i32(self.cnt), _i32(self.send_off), _i32(self.grp_off),
                       _i32(self.seg_off), _i32(self.csend_off), _i32(self.m_sizes))
        L.ref_dispatch_send(N, T, R, H, _u16(self.x), _i32(self.slot), _u8(self.send_q),
                            _f32(self.send_s), _i32(self.send_tok))
        L.ref_dispatch_recv(N, T, E, R, H, cap, _u8(self.send_q), _f32(self.send_s),
                            _i32(self.send_tok), _i32(self.cnt), _i32(self.eso),
                            _i32(self.seg_off), _u8(self.grp_q), _f32(self.grp_s),
                            _i32(self.grp_src))

    def combine(self) -> None:
        L, N, T, E, R, H, cap = lib(), self.N, self.T, self.E, self.R, self.H, self.cap
        L.ref_combine_send(N, T, E, R, H, cap, _u16(self.y), _i32(self.cnt), _i32(self.eso),
                           _i32(self.send_off), _i32(self.seg_off), _i32(self.csend_off),
                           _u16(self.csend))
        L.ref_combine_recv(N, T, E, R, H, cap, _u16(self.csend), _i32(self.idx), _f32(self.w),
                           _i32(self.slot), _i32(self.send_off), _i32(self.csend_off),
                           _u16(self.out))

    def step(self) -> tuple[float, float]:
        """One layer; returns (dispatch seconds, combine seconds)."""
        import time
        t0 = time.perf_counter()
        self.dispatch()
        t1 = time.perf_counter()
        self.combine()
        return t1 - t0, time.perf_counter() - t1


def layer_partial(N, T, E, R, H, cap, x, topk_idx, topk_w, mode: int = 0) -> dict:
    """``layer``, plus the combine with send-side reduction on the same expert
    outputs: ``part`` (partial rows) and ``out_partial``."""
    out = layer(N, T, E, R, H, cap, x, topk_idx, topk_w, mode)
    out["part"] = combine_partial_send(N, T, E, R, H, cap, out["y"], topk_idx, topk_w,
                                       out["slot_row"], out["expert_send_off"], out["seg_off"])
    out["out_partial"] = combine_partial_recv(N, T, E, R, H, out["part"], topk_idx,
                                              out["slot_row"])
    return out


# ------------------------------------------------------------------ low latency

def ll_rows(N, T, E, R, topk_idx) -> dict:
    ll_row = np.full((N, T, R), -7, np.int32)
    ll_count = np.zeros((N, E // N, N), np.int32)
    st = lib().ref_ll_rows(N, T, E, R, _i32(np.ascontiguousarray(topk_idx, dtype=np.int32)),
                           _i32(ll_row), _i32(ll_count))
    return dict(ll_row=ll_row, ll_count=ll_count, status=int(st))


def dispatch_ll(N, T, E, R, H, x, ll_row) -> dict:
    rows = N * E * T
    ll_q = np.full((rows, H), FILL_U8, np.uint8)
    ll_s = np.full((rows, H // 128), FILL_F32, np.float32)
    ll_src = np.full(rows, -1, np.int32)
    lib().ref_dispatch_ll(N, T, R, H, _u16(np.ascontiguousarray(x, dtype=np.uint16)),
                          _i32(np.ascontiguousarray(ll_row)), _u8(ll_q), _f32(ll_s), _i32(ll_src))
    return dict(ll_q=ll_q, ll_s=ll_s, ll_src=ll_src)


def standin_ll(N, T, E, H, mode, ll_q, ll_s, ll_count) -> np.ndarray:
    y = np.full((N * E * T, H), FILL_U16, np.uint16)
    c = np.ascontiguousarray
    lib().ref_standin_ll(N, T, E, H, mode, _u8(c(ll_q)), _f32(c(ll_s)), _i32(c(ll_count)), _u16(y))
    return y


def combine_ll(N, T, R, H, y_ll, topk_w, ll_row) -> np.ndarray:
    out = np.full((N, T, H), FILL_U16, np.uint16)
    c = np.ascontiguousarray
    lib().ref_combine_ll(N, T, R, H, _u16(c(y_ll)), _f32(c(topk_w, dtype=np.float32)),
                         _i32(c(ll_row)), _u16(out))
    return out


def layer_ll(N, T, E, R, H, x, topk_idx, topk_w, mode: int = 0) -> dict:
    """The low-latency path: rows, dispatch, stand-in, combine."""
    out = ll_rows(N, T, E, R, topk_idx)
    out.update(dispatch_ll(N, T, E, R, H, x, out["ll_row"]))
    out["y_ll"] = standin_ll(N, T, E, H, mode, out["ll_q"], out["ll_s"], out["ll_count"])
    out["out"] = combine_ll(N, T, R, H, out["y_ll"], topk_w, out["ll_row"])
    return out
