"""CPU oracle of the routed-expert MoE FFN layer -- TEST INFRASTRUCTURE ONLY.

A ctypes front end for oracle.c (plain fp64 C).  Only the tests, the smoke
check and the benchmark's CPU-baseline leg import this package; the product
library never does, and this package never imports the product library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = [os.path.join(_HERE, "oracle.c"), os.path.join(_HERE, "oracle.h")]
_SO = os.path.join(_HERE, "_oracle.so")
_lock = threading.Lock()
_handle = None


def build(force: bool = False) -> str:
    """Compile oracle.c into _oracle.so (fp contraction off; OpenMP when available)."""
    newest = max(os.path.getmtime(p) for p in _SRC)
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= newest:
        return _SO
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           _SRC[0], "-o", _SO + ".tmp", "-lm"]
    try:
        subprocess.run(cmd[:1] + ["-fopenmp"] + cmd[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(cmd, check=True, capture_output=True)
    os.replace(_SO + ".tmp", _SO)
    return _SO


class _Layer(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("H", "I", "E", "k", "n_shared", "SI")] + \
               [(n, ctypes.c_void_p) for n in ("w_gate", "w_up", "w_down", "s_gate", "s_up", "s_down",
                                              "sh_gate", "sh_up", "sh_down",
                                              "sh_s_gate", "sh_s_up", "sh_s_down")]


def _lib():
    global _handle
    with _lock:
        if _handle is None:
            lib = ctypes.CDLL(build())
            vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
            lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_decode.restype = ctypes.c_double
            lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
            lib.oracle_e4m3_encode.restype = ctypes.c_uint8
            lib.oracle_exp32.argtypes = [ctypes.c_float]
            lib.oracle_exp32.restype = ctypes.c_float
            lib.oracle_quant_1x128.argtypes = [vp, i32, vp, vp]
            lib.oracle_logits.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp]
            lib.oracle_route_from_logits.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp, vp]
            lib.oracle_forward.argtypes = [ctypes.POINTER(_Layer), vp, i32, vp, vp, vp, i32, i32, i32, vp, vp]
            lib.oracle_forward.restype = ctypes.c_int
            lib.oracle_forward_ex.argtypes = [ctypes.POINTER(_Layer), vp, i32, vp, vp, vp, i32, i32, vp, vp, vp, vp, vp,
                                              i32, vp, vp]
            lib.oracle_forward_ex.restype = ctypes.c_int
            lib.oracle_threads.restype = ctypes.c_int
            lib.oracle_e4m3_encode_n.argtypes = [vp, i64, vp]
            lib.oracle_e4m3_decode_n.argtypes = [vp, i64, vp]
            lib.oracle_exp32_n.argtypes = [vp, i64, vp]
            _handle = lib
    return _handle


def _ptr(a):
    return None if a is None else a.ctypes.data


def threads() -> int:
    """Threads the oracle's parallel loops use by default."""
    return int(_lib().oracle_threads())


def e4m3_decode(codes) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    _lib().oracle_e4m3_decode_n(c.ctypes.data, c.size, out.ctypes.data)
    return out


def e4m3_encode(values) -> np.ndarray:
    v = np.ascontiguousarray(values, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    _lib().oracle_e4m3_encode_n(v.ctypes.data, v.size, out.ctypes.data)
    return out


def exp32(x) -> np.ndarray:
    v = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.float32)
    _lib().oracle_exp32_n(v.ctypes.data, v.size, out.ctypes.data)
    return out


def quant_1x128(v):
    """Per-row 1x128 E4M3FN quantisation of fp32 rows v [..., n] -> (q u8, s f32)."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    n = v.shape[-1]
    if n % 128:
        raise ValueError("row length must be a multiple of 128")
    q = np.empty(v.shape, dtype=np.uint8)
    s = np.empty(v.shape[:-1] + (n // 128,), dtype=np.float32)
    rows = v.reshape(-1, n)
    qr, sr = q.reshape(-1, n), s.reshape(-1, n // 128)
    lib = _lib()
    for r in range(rows.shape[0]):
        lib.oracle_quant_1x128(rows[r].ctypes.data, n, qr[r].ctypes.data, sr[r].ctypes.data)
    return q, s


def logits(x_bf16, router_w, router_b=None, n_threads: int = 0) -> np.ndarray:
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    W = np.ascontiguousarray(router_w, dtype=np.float32)
    b = None if router_b is None else np.ascontiguousarray(router_b, dtype=np.float32)
    T, H = x.shape
    E = W.shape[0]
    out = np.empty((T, E), dtype=np.float32)
    _lib().oracle_logits(x.ctypes.data, W.ctypes.data, _ptr(b), T, H, E, n_threads, out.ctypes.data)
    return out


def route_from_logits(L, k: int) -> dict:
    L = np.ascontiguousarray(L, dtype=np.float32)
    T, E = L.shape
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    off = np.empty(E + 1, dtype=np.int32)
    st = np.empty(T * k, dtype=np.int32)
    inv = np.empty((T, k), dtype=np.int32)
    _lib().oracle_route_from_logits(L.ctypes.data, T, E, k, ids.ctypes.data, w.ctypes.data,
                                    off.ctypes.data, st.ctypes.data, inv.ctypes.data)
    return {"ids": ids, "w": w, "offsets": off, "sorted_token": st, "inv_row": inv}


def forward(inp: dict, k: int, ids, w, rows=None, exact_act: bool = False, n_threads: int = 0,
            want_f64: bool = False, hq_in=None, sh_in=None, want_h: bool = False):
    """The layer on the host.  inp holds the arrays of synth.make_inputs.
    Returns y as bf16 bits [n_rows][H]; with want_f64 also the fp64 sums; with
    want_h also a dict of this oracle's h records (h32, hq, sh), each
    [n_rows][slots][I (/128)] with slots = k routed (rank order) + shared.
    hq_in/sh_in ([T][slots][I], [T][slots][I/128]) override the h codes the
    down projection consumes."""
    x = np.ascontiguousarray(inp["x"], dtype=np.uint16)
    T, H = x.shape
    wg = inp["w_gate"]
    E, I = wg.shape[0], wg.shape[1]
    has_sh = "sh_gate" in inp
    SI = inp["sh_gate"].shape[1] if has_sh else 0
    keep = {}

    def c(name, dt):
        a = np.ascontiguousarray(inp[name], dtype=dt)
        keep[name] = a
        return a.ctypes.data

    lay = _Layer(H, I, E, k, 1 if has_sh else 0, SI,
                 c("w_gate", np.uint8), c("w_up", np.uint8), c("w_down", np.uint8),
                 c("s_gate", np.float32), c("s_up", np.float32), c("s_down", np.float32),
                 c("sh_gate", np.uint8) if has_sh else None, c("sh_up", np.uint8) if has_sh else None,
                 c("sh_down", np.uint8) if has_sh else None,
                 c("sh_s_gate", np.float32) if has_sh else None, c("sh_s_up", np.float32) if has_sh else None,
                 c("sh_s_down", np.float32) if has_sh else None)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    rws = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    n = T if rws is None else rws.size
    S = k + (1 if has_sh else 0)
    Imax = max(I, SI)
    y = np.empty((n, H), dtype=np.uint16)
    y64 = np.empty((n, H), dtype=np.float64) if want_f64 else None
    hrec = None
    if want_h:
        hrec = {"h32": np.empty((n, S, Imax), np.float32), "hq": np.empty((n, S, Imax), np.uint8),
                "sh": np.empty((n, S, Imax // 128), np.float32)}
    hq_in = None if hq_in is None else np.ascontiguousarray(hq_in, dtype=np.uint8).reshape(T, S, Imax)
    sh_in = None if sh_in is None else np.ascontiguousarray(sh_in, dtype=np.float32).reshape(T, S, Imax // 128)
    rc = _lib().oracle_forward_ex(ctypes.byref(lay), x.ctypes.data, T, ids.ctypes.data, w.ctypes.data,
                                  _ptr(rws), n, 1 if exact_act else 0, _ptr(hq_in), _ptr(sh_in),
                                  _ptr(hrec["h32"]) if hrec else None, _ptr(hrec["hq"]) if hrec else None,
                                  _ptr(hrec["sh"]) if hrec else None, n_threads, y.ctypes.data, _ptr(y64))
    if rc != 0:
        raise ValueError("oracle_forward rejected its arguments")
    out = [y]
    if want_f64:
        out.append(y64)
    if want_h:
        out.append(hrec)
    return out[0] if len(out) == 1 else tuple(out)
