"""Test helpers: build one MoE layer's inputs for both sides and compare against the oracle.

Both sides start from the same seeded fp32 tensors drawn by `synth`.  The GPU side quantizes
with the library's quantizer, the oracle side with the oracle's own; tests assert the two byte
streams are identical before comparing layer outputs.
"""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np
import torch

import oracle
import synth

# Layer tolerance (max over a row of |err| relative to that row's RMS; mean relative error
# as sum|err| / sum|ref| over the whole output).
ROW_RMS_TOL = 2e-2
MEAN_REL_TOL = 3e-3


BF16_HALF_ULP = 2.0 ** -9   # |bf16(v) - v| <= 2^-9 |v| for round-to-nearest-even (normal v)


def check_layer_close(got, ref, what="output", rounded_bf16=False, row_rms_tol=ROW_RMS_TOL):
    """The layer tolerance on the layer's result: max over a row of |err| <= 2e-2 * RMS(ref row)
    and sum|err| / sum|ref| <= 3e-3.  With rounded_bf16=True `got` is a bf16 output, i.e. the
    layer's fp32 result rounded to nearest even, and each element may further differ by that
    rounding: half a bf16 ulp, at most 2^-9 of its magnitude."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    err = np.abs(got - ref)
    rms = np.sqrt((ref ** 2).mean(axis=-1))
    allow = BF16_HALF_ULP * np.maximum(np.abs(got), np.abs(ref)) if rounded_bf16 else 0.0
    excess = np.maximum(err - allow, 0.0)
    ratio = excess.max(axis=-1) / np.maximum(rms, 1e-300)
    assert (excess.max(axis=-1) <= row_rms_tol * rms).all(), \
        f"{what}: worst max|err|/rms = {ratio.max():.3e} (row {int(ratio.argmax())})"
    denom = np.abs(ref).sum()
    rel = err.sum() / denom if denom > 0 else err.sum()
    assert rel <= MEAN_REL_TOL, f"{what}: mean relative error {rel:.3e}"
    return float(ratio.max()), float(rel)


def bf16_round_bits(x32: torch.Tensor) -> torch.Tensor:
    """fp32 -> bf16 round to nearest even (torch's conversion), as raw bits."""
    return x32.to(torch.bfloat16).view(torch.int16)


def check_bf16_stage_close(got, ref, what="stage"):
    """Bound for a bf16-rounded intermediate (h = SiLU(g)*u): one round-to-nearest bf16 step
    (relative error <= 2^-9, taken as 2^-8 for the fp32 work before it) plus 1e-3 of the row RMS
    for the fp32 accumulation-order differences.  The layer tolerance itself is checked on the
    layer output; this bound is per element and so catches any wrong element."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    rms = np.sqrt((ref ** 2).mean(axis=-1, keepdims=True))
    err = np.abs(got - ref)
    bound = 2.0 ** -8 * np.abs(ref) + 1e-3 * rms
    worst = (err / np.maximum(bound, 1e-300)).max()
    assert (err <= bound).all(), f"{what}: worst err/bound = {worst:.3e}"
    rel = err.sum() / max(np.abs(ref).sum(), 1e-300)
    assert rel <= MEAN_REL_TOL, f"{what}: mean relative error {rel:.3e}"
    return float(worst)


def to_np(t):
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy()
    return t.cpu().numpy()


class Layer:
    """Seeded inputs of one layer.  gen_device picks where synth draws (cpu for small shapes so
    both sides get identical tensors by copying; cuda for full-size shapes, where the oracle's
    groups are re-drawn one by one on the same device)."""

    def __init__(self, shape: synth.Shape, seed: int, layer: int = 0, logit_bias="none",
                 outlier_frac=0.0, gen_device="cpu"):
        self.shape, self.seed, self.layer, self.gen_device = shape, seed, layer, gen_device
        self.x = synth.activations(shape.T, shape.H, seed, layer, outlier_frac, device=gen_device)
        self.logits = synth.router_logits(shape.T, shape.E, seed, layer, logit_bias, device=gen_device)
        self.G = shape.E + shape.has_shared

    def fp32(self, proj, groups):
        return synth.projection_weights(self.shape, self.seed, self.layer, proj, groups, device=self.gen_device)

    def gpu_weights(self, moe, chunk=32):
        """NVFP4 weights of every group, quantized on the GPU by the library."""
        s = self.shape
        out = {}
        for proj, (N, K) in (("gate_up", (2 * s.I, s.H)), ("down", (s.H, s.I))):
            packed = torch.empty(self.G, N, K // 2, dtype=torch.uint8, device="cuda")
            scales = torch.empty(self.G, N, K // 16, dtype=torch.uint8, device="cuda")
            scale2 = torch.empty(self.G, dtype=torch.float32, device="cuda")
            for g0 in range(0, self.G, chunk):
                gs = list(range(g0, min(self.G, g0 + chunk)))
                q = moe.quantize_nvfp4(self.fp32(proj, gs).to("cuda"))
                packed[g0:g0 + len(gs)] = q.packed
                scales[g0:g0 + len(gs)] = q.scales
                scale2[g0:g0 + len(gs)] = q.scale2
            out[proj] = moe.NVFP4Weights(packed, scales, scale2)
        return out["gate_up"], out["down"]

    def oracle_weights(self, groups=None):
        """Oracle-quantized weights; only `groups` are filled (default: all), others zero."""
        s = self.shape
        groups = list(range(self.G)) if groups is None else sorted(set(groups))
        res = []
        for proj, (N, K) in (("gate_up", (2 * s.I, s.H)), ("down", (s.H, s.I))):
            packed = np.zeros((self.G, N, K // 2), np.uint8)
            scales = np.zeros((self.G, N, K // 16), np.uint8)
            scale2 = np.zeros((self.G,), np.float32)

            def one(g):
                w = self.fp32(proj, [g]).cpu().numpy()
                return g, oracle.quantize(w)

            with cf.ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
                for g, (p, sc, s2) in ex.map(one, groups):
                    packed[g], scales[g], scale2[g] = p[0], sc[0], s2[0]
            res.append((packed, scales, scale2))
        return res[0], res[1]

    def used_groups(self, tokens):
        ids, _ = oracle.route(self.logits.cpu(), self.shape.k)
        used = set(ids[tokens].reshape(-1).tolist())
        if self.shape.has_shared:
            used.add(self.shape.E)
        return sorted(used)


def moe_shape(moe, s: synth.Shape):
    return moe.Shape(T=s.T, H=s.H, I=s.I, E=s.E, k=s.k, has_shared=s.has_shared)
