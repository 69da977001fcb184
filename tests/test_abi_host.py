"""C-ABI checks that need no GPU: the library builds and loads, exports every function that
include/moe_nvfp4.h declares, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_nvfp4.h")


@pytest.fixture(scope="module")
def lib():
    from quantized_moe_expert_nvfp4_gb300 import build
    build.build()
    import quantized_moe_expert_nvfp4_gb300 as moe
    return moe, moe.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    moe, L = lib
    names = declared_functions()
    assert "moe_forward" in names and len(names) >= 10
    for n in names:
        assert hasattr(L, n), n


def _shape(moe, **kw):
    base = dict(T=8, H=2048, I=512, E=512, k=10, has_shared=1)
    base.update(kw)
    return moe.Shape(**base).c()


def test_workspace_size_and_unsupported_shapes(lib):
    moe, L = lib
    ok = _shape(moe)
    assert L.moe_workspace_size(ctypes.byref(ok)) > 0
    for bad in (dict(H=100), dict(H=64), dict(I=96), dict(E=0), dict(E=2048), dict(k=0), dict(k=17),
                dict(E=4, k=5), dict(T=-1), dict(has_shared=2), dict(T=1 << 30)):
        assert L.moe_workspace_size(ctypes.byref(_shape(moe, **bad))) == 0, bad


def test_host_validation_errors(lib):
    moe, L = lib
    P = ctypes.c_void_p
    shape = _shape(moe)
    ws_need = L.moe_workspace_size(ctypes.byref(shape))
    fake = P(0x100000)      # aligned, never dereferenced: validation fails before any CUDA call
    mis = P(0x100008)       # misaligned
    w_gu = moe.MoeWeights(0x200000, 0x300000, 0x400000, 513, 1024, 2048)
    w_dn = moe.MoeWeights(0x200000, 0x300000, 0x400000, 513, 2048, 512)
    call = lambda **o: L.moe_forward(o.get("x", fake), o.get("lg", fake), ctypes.byref(o.get("gu", w_gu)),
                                     ctypes.byref(o.get("dn", w_dn)), ctypes.byref(o.get("shape", shape)),
                                     o.get("out", fake), o.get("fp32", 0), o.get("ws", fake),
                                     o.get("ws_bytes", ws_need), None)
    assert call(x=P(0)) == -1
    assert call(out=mis) == -1
    assert call(fp32=2) == -1
    assert call(gu=moe.MoeWeights(0x200000, 0x300000, 0x400000, 512, 1024, 2048)) == -1
    assert call(dn=moe.MoeWeights(0x200000, 0x300000, 0x400000, 513, 1024, 512)) == -1
    assert call(shape=_shape(moe, H=100)) == -2
    assert call(ws_bytes=ws_need - 1) == -3
    assert call(ws=P(0x100010)) == -1   # workspace must be 256-byte aligned
    assert L.moe_route_topk(fake, ctypes.byref(shape), P(0), fake, None) == -1
    assert L.moe_combine(fake, fake, fake, ctypes.byref(shape), fake, 3, None) == -1
    assert L.moe_quantize_nvfp4(fake, 1, 16, 20, fake, fake, fake, None) == -2
    assert L.moe_quantize_nvfp4(mis, 1, 16, 32, fake, fake, fake, None) == -1
    for code in range(-6, 1):
        assert L.moe_status_string(code)


def test_arm_selection_on_the_host(lib):
    """moe_forward_arm is host logic (no CUDA call): the arm boundaries of the header."""
    moe, L = lib
    arm = lambda **kw: moe.forward_arm(moe.Shape(**{**dict(T=1, H=2048, I=512, E=512, k=10), **kw}))
    # one-launch decode kernel: T <= 8, H % 512 == 0, H <= 4096, I % 256 == 0, I <= 1024
    assert [arm(T=t) for t in (1, 2, 4, 8)] == [0, 0, 0, 0]
    assert arm(T=4, H=4096, I=1024) == 0 and arm(T=4, H=1024, I=256) == 0 and arm(T=3, H=512, E=16, k=4, I=256) == 0
    # three-launch decode arm for the other small-T shapes
    assert arm(T=4, H=8192) == 1 and arm(T=4, I=2048) == 1 and arm(T=4, I=128) == 1 and arm(T=4, I=640) == 1
    assert arm(T=4, H=256) == 1 and arm(T=9, I=128) == 1 and arm(T=64, I=128) == 1
    # tcgen05 grouped GEMMs above 8 tokens (H, I multiples of 256); CUDA-core GEMMs otherwise
    assert arm(T=9) == 2 and arm(T=64) == 2 and arm(T=65) == 2 and arm(T=4096) == 2
    assert arm(T=65, I=128) == 3
    assert arm(H=100) == -1


def test_static_scratch_fits_every_one_launch_shape(lib):
    """The no-allocation entry point's size rule, on the host only: its scratch (dominated by h and
    the expert outputs, T (k+1) (2 I + 4 H) bytes) fits the 4 MiB array for every one-launch decode
    shape, so a shape of arm 0 passes the size check (and then fails here only for want of a
    device), while shapes of other arms are rejected with MOE_ERR_UNSUPPORTED_SHAPE before any CUDA
    call.  Skipped where a GPU is visible: fake pointers must never reach a launch."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("host-only check; needs a machine without a GPU")
    moe, L = lib
    fn = L.moe_forward_decode_static_scratch
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(moe.MoeWeights),
                   ctypes.POINTER(moe.MoeWeights), ctypes.POINTER(moe.MoeShape), ctypes.c_void_p,
                   ctypes.c_int32, ctypes.c_void_p]
    fn.restype = ctypes.c_int32
    limit = 4 << 20
    n = 0
    for T in (1, 3, 8):
        for H in (512, 2048, 4096):
            for I in (256, 512, 1024):
                for k in (1, 10, 16):
                    E = 64
                    sh = moe.Shape(T=T, H=H, I=I, E=E, k=k, has_shared=1)
                    assert moe.forward_arm(sh) == 0
                    assert T * (k + 1) * (2 * I + 4 * H) + (64 << 10) <= limit
                    gu = moe.MoeWeights(0x200000, 0x300000, 0x400000, E + 1, 2 * I, H)
                    dn = moe.MoeWeights(0x200000, 0x300000, 0x400000, E + 1, H, I)
                    st = fn(0x100000, 0x100000, ctypes.byref(gu), ctypes.byref(dn), ctypes.byref(sh.c()),
                            0x100000, 0, None)
                    assert st != -2, (T, H, I, k, st)
                    n += 1
    for sh in (moe.Shape(T=9, H=2048, I=512, E=64, k=10), moe.Shape(T=4, H=8192, I=512, E=64, k=10)):
        assert moe.forward_arm(sh) != 0
        gu = moe.MoeWeights(0x200000, 0x300000, 0x400000, 65, 2 * sh.I, sh.H)
        dn = moe.MoeWeights(0x200000, 0x300000, 0x400000, 65, sh.H, sh.I)
        assert fn(0x100000, 0x100000, ctypes.byref(gu), ctypes.byref(dn), ctypes.byref(sh.c()), 0x100000, 0, None) == -2
    assert n == 81


def test_fp8_arm_host_validation(lib):
    """The FP8-activation arm's calls reject bad arguments before any CUDA call."""
    moe, L = lib
    P = ctypes.c_void_p
    fake, mis = P(0x100000), P(0x100008)
    shape = _shape(moe, T=4096)
    need = L.moe_workspace_size(ctypes.byref(shape))
    gu8 = moe.MoeFp8Weights(0x200000, 0x300000, 0x400000, 513, 1024, 2048)
    dn8 = moe.MoeFp8Weights(0x200000, 0x300000, 0x400000, 513, 2048, 512)
    call = lambda **o: L.moe_forward_fp8(o.get("x", fake), fake, ctypes.byref(o.get("gu", gu8)),
                                         ctypes.byref(o.get("dn", dn8)), ctypes.byref(o.get("shape", shape)),
                                         fake, o.get("fp32", 0), fake, o.get("ws", need), None)
    assert call(shape=_shape(moe, T=8)) == -2                      # decode batches: not this arm
    assert call(shape=_shape(moe, T=4096, I=128)) == -2            # I not a multiple of 256
    assert call(x=mis) == -1
    assert call(gu=moe.MoeFp8Weights(0x200000, 0x300000, 0x400000, 512, 1024, 2048)) == -1   # wrong G
    assert call(dn=moe.MoeFp8Weights(0x200000, 0x300008, 0x400000, 513, 2048, 512)) == -1   # misaligned
    assert call(fp32=2) == -1
    assert call(ws=need - 1) == -3
    w = moe.MoeWeights(0x200000, 0x300000, 0x400000, 513, 1024, 2048)
    assert L.moe_prepare_fp8(ctypes.byref(w), fake, mis, None) == -1
    assert L.moe_prepare_fp8(ctypes.byref(moe.MoeWeights(0x200000, 0x300000, 0x400000, 513, 1024, 200)),
                             fake, fake, None) == -2
    assert L.moe_quantize_rows_e4m3(fake, 4, 100, fake, fake, None) == -2
    assert L.moe_quantize_rows_e4m3(mis, 4, 256, fake, fake, None) == -1


def test_register_arm_row_bound_is_checked(lib):
    """moe_set_narrow_rows is host state (no CUDA call): -1..8 accepted, anything else rejected."""
    moe, L = lib
    for bad in (-2, 9, 64):
        with pytest.raises(moe.MoeError):
            moe.set_narrow_rows(bad)
    for ok in (0, 8, 3, -1):
        moe.set_narrow_rows(ok)
