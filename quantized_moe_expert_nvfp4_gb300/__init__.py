"""Python binding of `libmoe_nvfp4.so`, the GB300 (sm_103a) NVFP4 routed-MoE layer.

Argument marshalling only: each function checks dtypes, shapes and devices of torch tensors,
passes their device pointers and the current CUDA stream to the C ABI declared in
`include/moe_nvfp4.h`, and raises `MoeError` on a non-zero status.  Every step of the layer runs
in the library's CUDA kernels; there is no CPU or PyTorch fallback, and importing a function
that needs the library fails loudly when `libmoe_nvfp4.so` has not been built
(`python -c "import __graft_entry__ as g; g.build()"`).

PyTorch provides device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libmoe_nvfp4.so")

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", -1: "MOE_ERR_INVALID_ARG", -2: "MOE_ERR_UNSUPPORTED_SHAPE",
                -3: "MOE_ERR_WORKSPACE_TOO_SMALL", -4: "MOE_ERR_ARCH", -5: "MOE_ERR_CUDA",
                -6: "MOE_ERR_DEVICE_TIMEOUT"}
DECODE_MAX_T = 64   # largest batch the CUDA-core grouped-GEMV arm (1) takes, for shapes arm 2 cannot


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} returned {STATUS_NAMES.get(status, status)}: "
                         f"{load().moe_status_string(status).decode()}")


class MoeShape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("has_shared", ctypes.c_int32)]


class MoeWeights(ctypes.Structure):
    _fields_ = [("packed", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("scale2", ctypes.c_void_p),
                ("G", ctypes.c_int32), ("N", ctypes.c_int32), ("K", ctypes.c_int32)]


class MoeFp8Weights(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("row_scale", ctypes.c_void_p), ("scale2", ctypes.c_void_p),
                ("G", ctypes.c_int32), ("N", ctypes.c_int32), ("K", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def load() -> ctypes.CDLL:
    """Load libmoe_nvfp4.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build the CUDA library first "
                                   "(python -c 'import __graft_entry__ as g; g.build()')")
            lib = ctypes.CDLL(LIB_PATH)
            _declare(lib)
            _lib = lib
    return _lib


def _declare(L):
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    SH, W, W8 = ctypes.POINTER(MoeShape), ctypes.POINTER(MoeWeights), ctypes.POINTER(MoeFp8Weights)
    sigs = {
        "moe_workspace_size": ([SH], SZ),
        "moe_route_topk": ([P, SH, P, P, P], I32),
        "moe_permute": ([P, SH, P, P, P, P, P, SZ, P], I32),
        "moe_grouped_gate_up": ([P, P, P, W, SH, P, P, SZ, P], I32),
        "moe_grouped_down": ([P, P, W, SH, P, P, SZ, P], I32),
        "moe_combine": ([P, P, P, SH, P, I32, P], I32),
        "moe_forward": ([P, P, W, W, SH, P, I32, P, SZ, P], I32),
        "moe_forward_profiled": ([P, P, W, W, SH, P, I32, P, SZ, P, P], I32),
        "moe_quantize_nvfp4": ([P, I64, I64, I64, P, P, P, P], I32),
        "moe_get_device_status": ([P, ctypes.POINTER(I32), P], I32),
        "moe_status_string": ([I32], ctypes.c_char_p),
        "moe_forward_arm": ([SH], I32),
        "moe_router_logits": ([P, W, SH, P, P, SZ, P], I32),
        "moe_forward_routed": ([P, W, W, W, SH, P, I32, P, SZ, P], I32),
        "moe_prepare_fp8": ([W, P, P, P], I32),
        "moe_quantize_rows_e4m3": ([P, I64, I32, P, P, P], I32),
        "moe_forward_fp8": ([P, P, W8, W8, SH, P, I32, P, SZ, P], I32),
        "moe_set_narrow_rows": ([I32], I32),
    }
    for name, (args, res) in sigs.items():
        fn = getattr(L, name)
        fn.argtypes, fn.restype = args, res


def _check(fn: str, status: int):
    if status != MOE_OK:
        raise MoeError(fn, status)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t: torch.Tensor | None, dtype=None, name="tensor") -> ctypes.c_void_p:
    if t is None:
        return ctypes.c_void_p(0)
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


@dataclass
class Shape:
    T: int
    H: int
    I: int
    E: int
    k: int
    has_shared: int = 1

    @property
    def S(self) -> int:
        return self.T * self.k

    def c(self) -> MoeShape:
        return MoeShape(self.T, self.H, self.I, self.E, self.k, self.has_shared)


@dataclass
class NVFP4Weights:
    """One projection of every group: packed u8 [G, N, K/2], scales u8 [G, N, K/16] (e4m3
    bytes), scale2 fp32 [G]; all on the device."""
    packed: torch.Tensor
    scales: torch.Tensor
    scale2: torch.Tensor

    def c(self) -> MoeWeights:
        G, N, K2 = self.packed.shape
        for name, t, dt in (("packed", self.packed, torch.uint8), ("scales", self.scales, torch.uint8),
                            ("scale2", self.scale2, torch.float32)):
            _ptr(t, dt, name)
        return MoeWeights(self.packed.data_ptr(), self.scales.data_ptr(), self.scale2.data_ptr(),
                          G, N, 2 * K2)


@dataclass
class FP8Weights:
    """One projection of every group re-quantized to e4m3 (FP8-activation arm): codes u8
    [G, N, K], row_scale fp32 [G, N], scale2 fp32 [G] (the NVFP4 projection's own)."""
    codes: torch.Tensor
    row_scale: torch.Tensor
    scale2: torch.Tensor

    def c(self) -> MoeFp8Weights:
        G, N, K = self.codes.shape
        for name, t, dt in (("codes", self.codes, torch.uint8), ("row_scale", self.row_scale, torch.float32),
                            ("scale2", self.scale2, torch.float32)):
            _ptr(t, dt, name)
        return MoeFp8Weights(self.codes.data_ptr(), self.row_scale.data_ptr(), self.scale2.data_ptr(), G, N, K)


def workspace_size(shape: Shape) -> int:
    n = load().moe_workspace_size(ctypes.byref(shape.c()))
    if n == 0:
        raise MoeError("moe_workspace_size", -2)
    return n


def workspace(shape: Shape, device="cuda") -> torch.Tensor:
    """A zero-filled workspace buffer for `shape` (uint8, 256-byte aligned as torch allocates).
    Zero-filling clears the device status word the library keeps in its first bytes."""
    return torch.zeros(workspace_size(shape), dtype=torch.uint8, device=device)


def quantize_nvfp4(w: torch.Tensor, stream=None) -> NVFP4Weights:
    """Load-time NVFP4 quantization of fp32 weights [G, N, K] on the GPU."""
    G, N, K = w.shape
    dev = w.device
    packed = torch.empty(G, N, K // 2, dtype=torch.uint8, device=dev)
    scales = torch.empty(G, N, K // 16, dtype=torch.uint8, device=dev)
    scale2 = torch.empty(G, dtype=torch.float32, device=dev)
    _check("moe_quantize_nvfp4", load().moe_quantize_nvfp4(
        _ptr(w, torch.float32, "w"), G, N, K, _ptr(packed), _ptr(scales), _ptr(scale2), _stream(stream)))
    return NVFP4Weights(packed, scales, scale2)


def route_topk(logits: torch.Tensor, shape: Shape, topk_ids=None, topk_w=None, stream=None):
    dev = logits.device
    ids = topk_ids if topk_ids is not None else torch.empty(shape.T, shape.k, dtype=torch.int32, device=dev)
    w = topk_w if topk_w is not None else torch.empty(shape.T, shape.k, dtype=torch.float32, device=dev)
    _check("moe_route_topk", load().moe_route_topk(
        _ptr(logits, torch.float32, "logits"), ctypes.byref(shape.c()), _ptr(ids, torch.int32, "topk_ids"),
        _ptr(w, torch.float32, "topk_w"), _stream(stream)))
    return ids, w


def permute(topk_ids: torch.Tensor, shape: Shape, ws: torch.Tensor, stream=None):
    dev = topk_ids.device
    counts = torch.empty(shape.E, dtype=torch.int32, device=dev)
    offsets = torch.empty(shape.E + 1, dtype=torch.int32, device=dev)
    sorted_slot = torch.empty(max(shape.S, 1), dtype=torch.int32, device=dev)
    slot_pos = torch.empty(max(shape.S, 1), dtype=torch.int32, device=dev)
    _check("moe_permute", load().moe_permute(
        _ptr(topk_ids, torch.int32, "topk_ids"), ctypes.byref(shape.c()), _ptr(counts), _ptr(offsets),
        _ptr(sorted_slot), _ptr(slot_pos), _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)))
    return counts, offsets, sorted_slot[:shape.S], slot_pos[:shape.S]


def grouped_gate_up(x, sorted_slot, offsets, gate_up: NVFP4Weights, shape: Shape, ws, h=None, stream=None):
    h = h if h is not None else torch.empty(shape.S + shape.T, shape.I, dtype=torch.bfloat16, device=x.device)
    _check("moe_grouped_gate_up", load().moe_grouped_gate_up(
        _ptr(x, torch.bfloat16, "x"), _ptr(sorted_slot, torch.int32, "sorted_slot"),
        _ptr(offsets, torch.int32, "offsets"), ctypes.byref(gate_up.c()), ctypes.byref(shape.c()),
        _ptr(h, torch.bfloat16, "h"), _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)))
    return h


def grouped_down(h, offsets, down: NVFP4Weights, shape: Shape, ws, y=None, stream=None):
    y = y if y is not None else torch.empty(shape.S + shape.T, shape.H, dtype=torch.float32, device=h.device)
    _check("moe_grouped_down", load().moe_grouped_down(
        _ptr(h, torch.bfloat16, "h"), _ptr(offsets, torch.int32, "offsets"), ctypes.byref(down.c()),
        ctypes.byref(shape.c()), _ptr(y, torch.float32, "y"), _ptr(ws, torch.uint8, "ws"), ws.numel(),
        _stream(stream)))
    return y


def combine(y, slot_pos, topk_w, shape: Shape, out=None, out_fp32: bool = False, stream=None):
    dt = torch.float32 if out_fp32 else torch.bfloat16
    out = out if out is not None else torch.empty(shape.T, shape.H, dtype=dt, device=y.device)
    _check("moe_combine", load().moe_combine(
        _ptr(y, torch.float32, "y"), _ptr(slot_pos, torch.int32, "slot_pos"), _ptr(topk_w, torch.float32, "topk_w"),
        ctypes.byref(shape.c()), _ptr(out, dt, "out"), int(out_fp32), _stream(stream)))
    return out


def forward(x, logits, gate_up: NVFP4Weights, down: NVFP4Weights, shape: Shape, ws, out=None,
            out_fp32: bool = False, stream=None):
    """The whole layer (route, permute, grouped gate_up+SiLU, grouped down, combine, shared)."""
    dt = torch.float32 if out_fp32 else torch.bfloat16
    out = out if out is not None else torch.empty(shape.T, shape.H, dtype=dt, device=x.device)
    _check("moe_forward", load().moe_forward(
        _ptr(x, torch.bfloat16, "x"), _ptr(logits, torch.float32, "logits"), ctypes.byref(gate_up.c()),
        ctypes.byref(down.c()), ctypes.byref(shape.c()), _ptr(out, dt, "out"), int(out_fp32),
        _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)))
    return out


def forward_profiled(x, logits, gate_up: NVFP4Weights, down: NVFP4Weights, shape: Shape, ws, out,
                     stage_events, out_fp32: bool = False, stream=None):
    """forward() that also records 5 torch.cuda.Event (timing enabled) at the stage
    boundaries: before routing, after permute, after gate_up, after down, after combine."""
    dt = torch.float32 if out_fp32 else torch.bfloat16
    arr = (ctypes.c_void_p * 5)(*[ctypes.c_void_p(ev.cuda_event) for ev in stage_events])
    _check("moe_forward_profiled", load().moe_forward_profiled(
        _ptr(x, torch.bfloat16, "x"), _ptr(logits, torch.float32, "logits"), ctypes.byref(gate_up.c()),
        ctypes.byref(down.c()), ctypes.byref(shape.c()), _ptr(out, dt, "out"), int(out_fp32),
        _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream), arr))
    return out


def router_logits(x, router: NVFP4Weights, shape: Shape, ws, logits=None, stream=None):
    """fp32 [T, E] router logits of bf16 x against one NVFP4 projection (G = 1, N = E, K = H)."""
    logits = logits if logits is not None else torch.empty(shape.T, shape.E, dtype=torch.float32, device=x.device)
    _check("moe_router_logits", load().moe_router_logits(
        _ptr(x, torch.bfloat16, "x"), ctypes.byref(router.c()), ctypes.byref(shape.c()),
        _ptr(logits, torch.float32, "logits"), _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)))
    return logits


def forward_routed(x, router: NVFP4Weights, gate_up: NVFP4Weights, down: NVFP4Weights, shape: Shape, ws,
                   out=None, out_fp32: bool = False, stream=None):
    """The layer from x alone: router GEMM, then forward() on its logits."""
    dt = torch.float32 if out_fp32 else torch.bfloat16
    out = out if out is not None else torch.empty(shape.T, shape.H, dtype=dt, device=x.device)
    _check("moe_forward_routed", load().moe_forward_routed(
        _ptr(x, torch.bfloat16, "x"), ctypes.byref(router.c()), ctypes.byref(gate_up.c()),
        ctypes.byref(down.c()), ctypes.byref(shape.c()), _ptr(out, dt, "out"), int(out_fp32),
        _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)))
    return out


def prepare_fp8(w: NVFP4Weights, stream=None) -> FP8Weights:
    """Load-time re-quantization of an NVFP4 projection to e4m3 rows with fp32 row scales."""
    G, N, K2 = w.packed.shape
    codes = torch.empty(G, N, 2 * K2, dtype=torch.uint8, device=w.packed.device)
    rs = torch.empty(G, N, dtype=torch.float32, device=w.packed.device)
    _check("moe_prepare_fp8", load().moe_prepare_fp8(ctypes.byref(w.c()), _ptr(codes), _ptr(rs), _stream(stream)))
    return FP8Weights(codes, rs, w.scale2)


def quantize_rows_e4m3(x: torch.Tensor, stream=None):
    """bf16 [rows, K] -> (e4m3 codes u8 [rows, K], row scales fp32 [rows])."""
    rows, K = x.shape
    codes = torch.empty(rows, K, dtype=torch.uint8, device=x.device)
    scale = torch.empty(rows, dtype=torch.float32, device=x.device)
    _check("moe_quantize_rows_e4m3", load().moe_quantize_rows_e4m3(
        _ptr(x, torch.bfloat16, "x"), rows, K, _ptr(codes), _ptr(scale), _stream(stream)))
    return codes, scale


def forward_fp8(x, logits, gate_up: FP8Weights, down: FP8Weights, shape: Shape, ws, out=None,
                out_fp32: bool = False, stream=None):
    """The layer on the FP8-activation arm (e4m3 x e4m3 grouped GEMMs with row scales)."""
    dt = torch.float32 if out_fp32 else torch.bfloat16
    out = out if out is not None else torch.empty(shape.T, shape.H, dtype=dt, device=x.device)
    _check("moe_forward_fp8", load().moe_forward_fp8(
        _ptr(x, torch.bfloat16, "x"), _ptr(logits, torch.float32, "logits"), ctypes.byref(gate_up.c()),
        ctypes.byref(down.c()), ctypes.byref(shape.c()), _ptr(out, dt, "out"), int(out_fp32),
        _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)))
    return out


def device_status(ws: torch.Tensor, stream=None) -> int:
    v = ctypes.c_int32(0)
    _check("moe_get_device_status", load().moe_get_device_status(
        _ptr(ws, torch.uint8, "ws"), ctypes.byref(v), _stream(stream)))
    return v.value


def debug_timeout_probe(ws: torch.Tensor, limit_ns: int, stream=None) -> None:
    """Run the decode kernel's bounded wait on a barrier nothing arrives at (test hook): it runs
    out after limit_ns and records MOE_ERR_DEVICE_TIMEOUT in the workspace status word."""
    lib = load()
    lib.moe_debug_timeout_probe.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p]
    lib.moe_debug_timeout_probe.restype = ctypes.c_int32
    _check("moe_debug_timeout_probe", lib.moe_debug_timeout_probe(
        _ptr(ws, torch.uint8, "ws"), int(limit_ns), _stream(stream)))


ARM_NAMES = {0: "decode, one cooperative launch (tensor-core grouped GEMV)",
             1: "decode, three launches (grouped GEMV)",
             2: "batched decode / prefill, tcgen05 grouped GEMM", 3: "prefill, CUDA-core grouped GEMM"}


def forward_arm(shape: Shape) -> int:
    """Which kernels moe_forward runs for this shape (see moe_forward_arm in the header)."""
    return load().moe_forward_arm(ctypes.byref(shape.c()))


def set_narrow_rows(rows: int) -> None:
    """Row bound of the register arm inside the tcgen05 grouped GEMMs (moe_set_narrow_rows):
    expert groups of at most `rows` tokens run on mma.sync in the same launch; 0 = none, -1 =
    the library's default."""
    _check("moe_set_narrow_rows", load().moe_set_narrow_rows(int(rows)))


def status_string(status: int) -> str:
    return load().moe_status_string(status).decode()


__all__ = ["Shape", "NVFP4Weights", "MoeError", "load", "workspace_size", "workspace",
           "quantize_nvfp4", "route_topk", "permute", "grouped_gate_up", "grouped_down", "combine",
           "forward", "forward_profiled", "forward_arm", "router_logits", "forward_routed", "FP8Weights",
           "prepare_fp8", "quantize_rows_e4m3", "forward_fp8", "ARM_NAMES", "device_status", "status_string",
           "set_narrow_rows", "DECODE_MAX_T", "LIB_PATH"]
