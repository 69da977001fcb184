"""GPU parity of the router GEMM (moe_router_logits) and of the layer from x alone
(moe_forward_routed) against the CPU oracle (needs a GB300).

The router's logits are fp32 sums of H products; they are checked against the oracle's fp64
logits with the bound that fp32 accumulation implies.  The top-k on them is then bit-exact
against the oracle's top-k on its own logits wherever the k-th and (k+1)-th logits of a token are
further apart than that bound (elsewhere both choices are correct), and the layer output is
checked against the oracle's layer routed on its own logits with the layer tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from moe_cases import Layer, check_layer_close, moe_shape, to_np

pytestmark = pytest.mark.gpu

# (T, H, E, k, I, seed): the CUDA-core router (T <= 32, or E not a multiple of 128) and the
# tensor-core one (ragged token tiles, several tiles, the full prefill chunk), both sides of the
# boundary
CASES = [
    (4, 256, 16, 2, 128, 300),
    (1, 2048, 512, 10, 512, 301),
    (8, 2048, 512, 10, 512, 302),
    (9, 384, 48, 3, 256, 303),
    (32, 2048, 512, 10, 512, 307),
    (33, 512, 256, 8, 256, 308),
    (64, 2048, 512, 10, 512, 304),
    (300, 512, 256, 8, 256, 305),
    (4096, 2048, 512, 10, 512, 306),
]


def _router(moe, shape, seed, device):
    w = synth.router_weights(shape, seed, device=device)
    q = moe.quantize_nvfp4(w.to("cuda"))
    o = oracle.quantize(w.cpu().numpy())
    assert np.array_equal(q.packed.cpu().numpy(), o[0]) and np.array_equal(q.scales.cpu().numpy(), o[1])
    return q, (o[0][0], o[1][0], o[2]), w


def _logit_bound(x, o):
    """Per-logit bound for an fp32 sum of H products: 2e-5 of sum_h |w x|."""
    wd = oracle.dequantize(o[0][None], o[1][None], o[2])[0]
    xv = x.float().double().cpu().numpy()
    return 2e-5 * (np.abs(xv) @ np.abs(wd).T) + 1e-30


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"T{c[0]}_H{c[1]}_E{c[2]}")
def test_router_logits(cuda_lib, case):
    moe = cuda_lib
    T, H, E, k, I, seed = case
    shape = synth.Shape(T=T, H=H, E=E, k=k, I=I)
    dev = "cuda" if T * H > 1 << 20 else "cpu"
    x = synth.activations(T, H, seed, device=dev)
    q, o, _ = _router(moe, shape, seed, dev)
    ms = moe_shape(moe, shape)
    ws = moe.workspace(ms)
    logits = moe.router_logits(x.cuda(), q, ms, ws)
    torch.cuda.synchronize()
    assert moe.device_status(ws) == 0
    ref = oracle.router_logits(x.cpu(), o)
    err = np.abs(logits.cpu().numpy().astype(np.float64) - ref)
    bound = _logit_bound(x, o)
    assert (err <= bound).all(), f"worst err/bound {(err / bound).max():.3e}"


def _clear_tokens(ref, k, margin):
    """Tokens whose k-th and (k+1)-th logits differ by more than the margin (and so route the
    same on any logits within it)."""
    s = -np.sort(-ref, axis=1)
    if s.shape[1] == k:
        return np.ones(ref.shape[0], bool)
    gap = s[:, k - 1] - s[:, k]
    return gap > 2 * margin.max(axis=1)


@pytest.mark.parametrize("case", [CASES[0], CASES[2], CASES[3], CASES[5]], ids=lambda c: f"T{c[0]}_H{c[1]}_E{c[2]}")
def test_forward_routed_matches_oracle(cuda_lib, case):
    moe = cuda_lib
    T, H, E, k, I, seed = case
    shape = synth.Shape(T=T, H=H, E=E, k=k, I=I)
    dev = "cuda" if H >= 2048 else "cpu"
    L = Layer(shape, seed, gen_device=dev)
    q, o, _ = _router(moe, shape, seed + 1000, dev)
    ms = moe_shape(moe, shape)
    gu, dn = L.gpu_weights(moe)
    ws = moe.workspace(ms)
    x = L.x.cuda()
    out = moe.forward_routed(x, q, gu, dn, ms, ws, out_fp32=True)
    glog = moe.router_logits(x, q, ms, moe.workspace(ms))
    ids, _ = moe.route_topk(glog, ms)
    torch.cuda.synchronize()
    assert moe.device_status(ws) == 0
    ref_logits = oracle.router_logits(L.x.cpu(), o)
    clear = _clear_tokens(ref_logits, k, _logit_bound(L.x, o))
    assert clear.mean() > 0.9, "too many near-ties for a meaningful check"
    oids, _ = oracle.route(ref_logits.astype(np.float32), k)
    assert np.array_equal(ids.cpu().numpy()[clear], oids[clear])
    ogu, odn = L.oracle_weights(sorted(set(oids.reshape(-1).tolist()) | {E}))
    ref = oracle.moe_forward(L.x.cpu(), ref_logits.astype(np.float32), ogu, odn, k, 1)
    toks = np.nonzero(clear)[0]
    check_layer_close(to_np(out)[toks], ref[toks], "forward_routed fp32")
