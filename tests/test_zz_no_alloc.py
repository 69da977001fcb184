"""The allocation-free decode entry point (moe_forward_decode_static_scratch).

It serves callers that cannot allocate device memory, so it keeps its scratch in a fixed array
inside the library instead of a caller workspace.  This test calls it through the C ABI and
checks it against the CPU oracle and against moe_forward (the workspace-based entry point) on two
calls in a row, with the layer tolerance the other parity tests use.  It sits in a file of its own, collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from moe_cases import Layer, check_layer_close, moe_shape, to_np

pytestmark = pytest.mark.gpu

CASES = [
    (3, 2048, 16, 4, 512, 1, "none", 201),
    (8, 2048, 512, 10, 512, 1, "none", 202),
    # k = 16 at the largest H and I of the one-launch arm (h and y: 2.5 MB of the 4 MiB array)
    (8, 4096, 64, 16, 1024, 1, "zipf", 203),
]


def _call(moe, x, logits, gu, dn, ms, out, fp32):
    L = moe.load()
    fn = L.moe_forward_decode_static_scratch
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(moe.MoeWeights),
                   ctypes.POINTER(moe.MoeWeights), ctypes.POINTER(moe.MoeShape), ctypes.c_void_p,
                   ctypes.c_int32, ctypes.c_void_p]
    fn.restype = ctypes.c_int32
    gu_c, dn_c, sh_c = gu.c(), dn.c(), ms.c()
    st = fn(x.data_ptr(), logits.data_ptr(), ctypes.byref(gu_c), ctypes.byref(dn_c), ctypes.byref(sh_c),
            out.data_ptr(), int(fp32), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


def _oracle_ref(L):
    s = L.shape
    ogu, odn = L.oracle_weights(L.used_groups(list(range(s.T))))
    return oracle.moe_forward(L.x.cpu(), L.logits.cpu(), ogu, odn, s.k, s.has_shared)


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"T{c[0]}_H{c[1]}_E{c[2]}")
def test_static_scratch_matches_oracle_and_moe_forward(cuda_lib, case):
    """Two calls in a row of each output type, each checked against the CPU oracle and against
    moe_forward (the workspace entry point), with the layer tolerance."""
    moe = cuda_lib
    T, H, E, k, I, sh, bias, seed = case
    L = Layer(synth.Shape(T=T, H=H, E=E, k=k, I=I, has_shared=sh), seed, logit_bias=bias,
              gen_device="cuda" if H >= 2048 else "cpu")
    ms = moe_shape(moe, L.shape)
    assert moe.forward_arm(ms) == 0
    gu, dn = L.gpu_weights(moe)
    x, logits = L.x.cuda(), L.logits.cuda()
    ws = moe.workspace(ms)
    oref = _oracle_ref(L)
    for fp32 in (False, True):
        dt = torch.float32 if fp32 else torch.bfloat16
        ref = moe.forward(x, logits, gu, dn, ms, ws, out_fp32=fp32)
        for _ in range(2):   # two calls in a row share the same scratch
            out = torch.full((T, H), float("nan"), dtype=dt, device="cuda")
            assert _call(moe, x, logits, gu, dn, ms, out, fp32) == 0
            torch.cuda.synchronize()
            check_layer_close(to_np(out), oref, f"static scratch vs oracle, fp32={fp32}", rounded_bf16=not fp32)
            check_layer_close(to_np(out), to_np(ref).astype(np.float64), f"static scratch vs moe_forward, fp32={fp32}")


def test_static_scratch_after_a_device_timeout(cuda_lib):
    """A device-side bounded wait that ran out (the timeout probe, on a workspace) leaves the
    context usable: the next static-scratch call is still correct."""
    moe = cuda_lib
    T, H, E, k, I, sh, bias, seed = CASES[0]
    L = Layer(synth.Shape(T=T, H=H, E=E, k=k, I=I, has_shared=sh), seed, logit_bias=bias, gen_device="cuda")
    ms = moe_shape(moe, L.shape)
    ws = moe.workspace(ms)
    moe.debug_timeout_probe(ws, 2_000_000)
    assert moe.device_status(ws) == -6   # MOE_ERR_DEVICE_TIMEOUT
    gu, dn = L.gpu_weights(moe)
    out = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    assert _call(moe, L.x.cuda(), L.logits.cuda(), gu, dn, ms, out, False) == 0
    torch.cuda.synchronize()
    check_layer_close(to_np(out), _oracle_ref(L), "static scratch after a timeout", rounded_bf16=True)


def test_static_scratch_rejects_other_shapes(cuda_lib):
    moe = cuda_lib
    ms = moe.Shape(T=16, H=2048, I=512, E=512, k=10)      # not a one-launch decode shape
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    w = moe.NVFP4Weights(dummy.view(1, 1, 16), dummy.view(1, 1, 16), torch.zeros(1, device="cuda"))
    out = torch.empty(16, 2048, dtype=torch.bfloat16, device="cuda")
    x = torch.empty(16, 2048, dtype=torch.bfloat16, device="cuda")
    lg = torch.empty(16, 512, device="cuda")
    assert _call(moe, x, lg, w, w, ms, out, False) == -2
