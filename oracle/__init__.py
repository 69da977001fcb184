"""CPU oracle of the NVFP4 routed-MoE layer -- TEST INFRASTRUCTURE ONLY.

Only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline leg of `bench.py` may import
this package.  The CUDA library never imports, links or calls it, and this package imports
nothing from the library: the two meet only in the seeded inputs drawn by `synth`.

The oracle is plain C++ (`moe_oracle.cpp`) compiled with g++ into `_build/liboracle.so` and
called through ctypes.  Every function computes the plain definition of its step in fp64; the
quantizer's steps are fp32 operations, because its input weights are fp32 and the recipe states
each step on those fp32 values.  What each function follows is cited in `moe_oracle.h` /
`moe_oracle.cpp`.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
_HDR = os.path.join(_HERE, "moe_oracle.h")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle (g++ -O2 -ffp-contract=off, no fast-math) and return the .so path."""
    os.makedirs(_BUILD, exist_ok=True)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= newest:
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-pthread", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            _declare(_lib)
    return _lib


def _declare(L):
    P, I64, I32, F, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_double
    L.orc_e2m1_value.argtypes, L.orc_e2m1_value.restype = [I32], D
    L.orc_e4m3_value.argtypes, L.orc_e4m3_value.restype = [I32], D
    L.orc_e2m1_encode.argtypes, L.orc_e2m1_encode.restype = [F], I32
    L.orc_e4m3_encode.argtypes, L.orc_e4m3_encode.restype = [F], I32
    L.orc_quantize.argtypes, L.orc_quantize.restype = [P, I64, I64, I64, P, P, P], I32
    L.orc_dequantize.argtypes, L.orc_dequantize.restype = [P, P, P, I64, I64, I64, P], I32
    L.orc_router_logits.argtypes, L.orc_router_logits.restype = [P, P, P, P, I32, I32, I32, P], I32
    L.orc_route.argtypes, L.orc_route.restype = [P, I32, I32, I32, P, P], I32
    L.orc_permute.argtypes, L.orc_permute.restype = [P, I32, I32, I32, P, P, P, P], I32
    L.orc_moe_forward.argtypes = [P] * 8 + [I32] * 6 + [P, I32, P, P, P, I32]
    L.orc_moe_forward.restype = I32
    L.orc_quant_rows_e4m3.argtypes, L.orc_quant_rows_e4m3.restype = [P, I64, I64, P, P], I32
    L.orc_prepare_fp8.argtypes, L.orc_prepare_fp8.restype = [P, P, I64, I64, I64, P, P], I32
    L.orc_moe_forward_fp8.argtypes = [P] * 8 + [I32] * 6 + [P, I32, P, P, P, I32]
    L.orc_moe_forward_fp8.restype = I32


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _np(t, dtype):
    """Contiguous numpy array of `dtype` from a numpy array or a (CPU or CUDA) torch tensor.
    bf16 tensors are taken as their raw 16-bit patterns."""
    if hasattr(t, "detach"):
        import torch
        t = t.detach().cpu()
        if t.dtype == torch.bfloat16:
            t = t.view(torch.int16)
        t = t.numpy()
    a = np.asarray(t)
    dt = np.dtype(dtype)
    if a.dtype != dt:
        if a.dtype.kind in "ui" and dt.kind in "ui" and a.dtype.itemsize == dt.itemsize:
            a = a.view(dt)
        else:
            a = a.astype(dt)
    return np.ascontiguousarray(a)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (status {rc})")


def e2m1_value(code: int) -> float:
    return lib().orc_e2m1_value(int(code))


def e4m3_value(code: int) -> float:
    return lib().orc_e4m3_value(int(code))


def e2m1_encode(v: float) -> int:
    return lib().orc_e2m1_encode(float(v))


def e4m3_encode(v: float) -> int:
    return lib().orc_e4m3_encode(float(v))


def quantize(w) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """fp32 [G, N, K] -> (packed u8 [G,N,K/2], scales u8 [G,N,K/16], scale2 f32 [G])."""
    w = _np(w, np.float32)
    G, N, K = w.shape
    packed = np.empty((G, N, K // 2), np.uint8)
    scales = np.empty((G, N, K // 16), np.uint8)
    scale2 = np.empty((G,), np.float32)
    _check(lib().orc_quantize(_ptr(w), G, N, K, _ptr(packed), _ptr(scales), _ptr(scale2)), "quantize")
    return packed, scales, scale2


def dequantize(packed, scales, scale2) -> np.ndarray:
    packed, scales, scale2 = _np(packed, np.uint8), _np(scales, np.uint8), _np(scale2, np.float32)
    G, N, K2 = packed.shape
    out = np.empty((G, N, 2 * K2), np.float64)
    _check(lib().orc_dequantize(_ptr(packed), _ptr(scales), _ptr(scale2), G, N, 2 * K2, _ptr(out)),
           "dequantize")
    return out


def router_logits(x, router) -> np.ndarray:
    """fp64 [T, E] router logits of bf16 x [T, H] against one NVFP4 projection
    router = (packed [1, E, H/2] or [E, H/2], scales [.., E, H/16], scale2 [1])."""
    xb = _np(x, np.uint16)
    p, s_, z = _np(router[0], np.uint8), _np(router[1], np.uint8), _np(router[2], np.float32)
    T, H = xb.shape
    E = p.shape[-2]
    out = np.empty((T, E), np.float64)
    _check(lib().orc_router_logits(_ptr(xb), _ptr(p), _ptr(s_), _ptr(z), T, H, E, _ptr(out)), "router_logits")
    return out


def route(logits, k: int) -> tuple[np.ndarray, np.ndarray]:
    """fp32 [T, E] -> (ids int32 [T, k], weights fp64 [T, k])."""
    logits = _np(logits, np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    _check(lib().orc_route(_ptr(logits), T, E, k, _ptr(ids), _ptr(w)), "route")
    return ids, w


def permute(ids, E: int):
    """int32 [T, k] -> (counts [E], offsets [E+1], sorted_slot [T*k], slot_pos [T*k])."""
    ids = _np(ids, np.int32)
    T, k = ids.shape
    counts = np.empty((E,), np.int32)
    offsets = np.empty((E + 1,), np.int32)
    sorted_slot = np.empty((T * k,), np.int32)
    slot_pos = np.empty((T * k,), np.int32)
    _check(lib().orc_permute(_ptr(ids), T, E, k, _ptr(counts), _ptr(offsets), _ptr(sorted_slot),
                             _ptr(slot_pos)), "permute")
    return counts, offsets, sorted_slot, slot_pos


def moe_forward(x, logits, gate_up, down, k: int, has_shared: int = 1, tokens=None,
                dumps: bool = False, n_threads: int = 0):
    """fp64 layer output for the listed tokens (default all).

    x: bf16 [T, H] (torch) or its uint16 bits; logits fp32 [T, E];
    gate_up / down: (packed, scales, scale2) with G = E + has_shared groups.
    Returns out [n, H] (and h [n, k+1, I], y [n, k+1, H] when dumps=True).
    """
    xb = _np(x, np.uint16)
    lg = _np(logits, np.float32)
    T, H = xb.shape
    E = lg.shape[1]
    gp, gs, g2 = (_np(gate_up[0], np.uint8), _np(gate_up[1], np.uint8), _np(gate_up[2], np.float32))
    dp, ds, d2 = (_np(down[0], np.uint8), _np(down[1], np.uint8), _np(down[2], np.float32))
    I = gp.shape[1] // 2
    if tokens is None:
        tok = None
        n = T
    else:
        tok = np.ascontiguousarray(np.asarray(tokens, np.int32))
        n = tok.shape[0]
    J = k + (1 if has_shared else 0)
    out = np.empty((n, H), np.float64)
    h = np.empty((n, J, I), np.float64) if dumps else None
    y = np.empty((n, J, H), np.float64) if dumps else None
    rc = lib().orc_moe_forward(_ptr(xb), _ptr(lg), _ptr(gp), _ptr(gs), _ptr(g2), _ptr(dp), _ptr(ds),
                               _ptr(d2), T, H, I, E, k, int(has_shared),
                               None if tok is None else _ptr(tok), n, _ptr(out),
                               None if h is None else _ptr(h), None if y is None else _ptr(y),
                               int(n_threads))
    _check(rc, "moe_forward")
    return (out, h, y) if dumps else out


def quant_rows_e4m3(v) -> tuple[np.ndarray, np.ndarray]:
    """fp32 [rows, K] -> (e4m3 codes u8 [rows, K], row scales f32 [rows]) by the row rule of the
    FP8-activation arm (see moe_oracle.h)."""
    v = _np(v, np.float32)
    rows, K = v.shape
    codes = np.empty((rows, K), np.uint8)
    scale = np.empty((rows,), np.float32)
    _check(lib().orc_quant_rows_e4m3(_ptr(v), rows, K, _ptr(codes), _ptr(scale)), "quant_rows_e4m3")
    return codes, scale


def prepare_fp8(packed, scales) -> tuple[np.ndarray, np.ndarray]:
    """NVFP4 (packed [G, N, K/2], scales [G, N, K/16]) -> (e4m3 codes [G, N, K], row scales [G, N])."""
    packed, scales = _np(packed, np.uint8), _np(scales, np.uint8)
    G, N, K2 = packed.shape
    codes = np.empty((G, N, 2 * K2), np.uint8)
    rs = np.empty((G, N), np.float32)
    _check(lib().orc_prepare_fp8(_ptr(packed), _ptr(scales), G, N, 2 * K2, _ptr(codes), _ptr(rs)), "prepare_fp8")
    return codes, rs


def moe_forward_fp8(x, logits, gate_up, down, k: int, has_shared: int = 1, tokens=None,
                    dumps: bool = False, n_threads: int = 0):
    """fp64 output of the FP8-activation arm for the listed tokens (default all).

    gate_up / down: (codes [G, N, K] u8, row_scale [G, N] f32, scale2 [G] f32) as prepare_fp8
    gives them plus the NVFP4 scale2.  Returns out [n, H] (and h [n, k+1, I], y [n, k+1, H]
    when dumps=True)."""
    xb = _np(x, np.uint16)
    lg = _np(logits, np.float32)
    T, H = xb.shape
    E = lg.shape[1]
    gc, gr, g2 = (_np(gate_up[0], np.uint8), _np(gate_up[1], np.float32), _np(gate_up[2], np.float32))
    dc, dr, d2 = (_np(down[0], np.uint8), _np(down[1], np.float32), _np(down[2], np.float32))
    I = gc.shape[1] // 2
    if tokens is None:
        tok, n = None, T
    else:
        tok = np.ascontiguousarray(np.asarray(tokens, np.int32))
        n = tok.shape[0]
    J = k + (1 if has_shared else 0)
    out = np.empty((n, H), np.float64)
    h = np.empty((n, J, I), np.float64) if dumps else None
    y = np.empty((n, J, H), np.float64) if dumps else None
    rc = lib().orc_moe_forward_fp8(_ptr(xb), _ptr(lg), _ptr(gc), _ptr(gr), _ptr(g2), _ptr(dc), _ptr(dr),
                                   _ptr(d2), T, H, I, E, k, int(has_shared),
                                   None if tok is None else _ptr(tok), n, _ptr(out),
                                   None if h is None else _ptr(h), None if y is None else _ptr(y),
                                   int(n_threads))
    _check(rc, "moe_forward_fp8")
    return (out, h, y) if dumps else out
