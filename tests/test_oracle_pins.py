"""Pins of the CPU oracle to facts outside itself (CPU only).

Each test checks the oracle against something it does not compute itself: the golden fixtures
under tests/golden/ (format tables and hand-worked layers with closed forms), library routines
(torch's float8_e4m3fn codec, numpy's stable argsort, torch's softmax and matmul), brute force
on tiny inputs, and invariants of the method.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ----------------------------------------------------------------------------- formats

def test_e2m1_table_matches_golden():
    for code, val in _golden("e2m1_values.txt"):
        got = oracle.e2m1_value(int(code))
        want = float(val)
        assert got == want and math.copysign(1, got) == math.copysign(1, want), (code, got, want)


def test_e4m3_decode_matches_torch_float8_for_all_256_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    lib_vals = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = oracle.e4m3_value(c)
        if math.isnan(lib_vals[c]):
            assert math.isnan(got), c
        else:
            assert got == lib_vals[c] and math.copysign(1, got) == math.copysign(1, lib_vals[c]), c


def test_e4m3_golden_points():
    for code, val in _golden("e4m3_points.txt"):
        got = oracle.e4m3_value(int(code, 16))
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val)), code


def test_e2m1_encode_midpoints_and_saturation():
    for v, code in _golden("e2m1_ties.txt"):
        assert oracle.e2m1_encode(float(v)) == int(code), v


def _brute_nearest_even(v, values):
    """Brute-force nearest entry of `values` (index == code, increasing), ties to even code."""
    best = None
    for c, t in enumerate(values):
        d = abs(v - t)
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
            best = (d, c)
    return best[1]


def test_e2m1_encode_brute_force_sweep():
    mags = [abs(oracle.e2m1_value(c)) for c in range(8)]
    vals = np.concatenate([np.linspace(0, 7, 2801), synth.random_floats(2000, 11, scale=3).numpy()])
    for v in vals.astype(np.float32):
        want = _brute_nearest_even(min(abs(float(v)), 6.0), mags) | (8 if np.signbit(v) else 0)
        assert oracle.e2m1_encode(float(v)) == want, v


def test_e4m3_encode_agrees_with_torch_rne_in_range():
    vals = torch.cat([torch.linspace(0, 448, 20001), torch.rand(20000) * 448,
                      torch.exp2(torch.linspace(-12, 8.8, 5000))]).to(torch.float32)
    vals = vals[vals <= 448]
    lib_codes = vals.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for v, c in zip(vals.numpy(), lib_codes):
        assert oracle.e4m3_encode(float(v)) == int(c), float(v)


def test_e4m3_encode_saturates():
    assert oracle.e4m3_encode(448.0) == 0x7E
    assert oracle.e4m3_encode(464.0) == 0x7E
    assert oracle.e4m3_encode(1e30) == 0x7E
    assert oracle.e4m3_encode(-1e30) == 0xFE


def test_every_e2m1_times_e4m3_product_is_exact_in_bf16():
    # The W4A16 arm dequantizes e2m1 x e4m3 into bf16 before the MMA; every one of the 16 x 254
    # finite products must survive the bf16 rounding unchanged.
    a = np.array([oracle.e2m1_value(c) for c in range(16)])
    b = np.array([oracle.e4m3_value(c) for c in range(256) if c not in (0x7F, 0xFF)])
    prod = torch.tensor(np.outer(a, b), dtype=torch.float64)
    assert torch.equal(prod.to(torch.bfloat16).to(torch.float64), prod)


# ----------------------------------------------------------------------------- quantizer

def _numpy_quantize(w):
    """Second derivation of the quantizer: numpy float32 steps, nearest-entry searches over value
    tables taken from torch's float8 decoder and the golden e2m1 table."""
    G, N, K = w.shape
    e4 = torch.arange(127, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    e2 = np.array([float(v) for _, v in _golden("e2m1_values.txt")[:8]], np.float32)
    packed = np.zeros((G, N, K // 2), np.uint8)
    scales = np.zeros((G, N, K // 16), np.uint8)
    scale2 = np.zeros(G, np.float32)
    for g in range(G):
        amax = np.float32(np.abs(w[g]).max())
        s2 = np.float32(amax / np.float32(2688.0))
        scale2[g] = s2
        for n in range(N):
            for b in range(K // 16):
                blk = w[g, n, b * 16:(b + 1) * 16]
                bamax = np.float32(np.abs(blk).max())
                sc = 0 if s2 == 0 else _brute_nearest_even(
                    min(float(np.float32(np.float32(bamax / np.float32(6.0)) / s2)), 448.0), e4)
                scales[g, n, b] = sc
                d = np.float32(np.float32(e4[sc]) * s2)
                codes = []
                for v in blk:
                    if d == 0:
                        codes.append(0)
                    else:
                        q = np.float32(v / d)
                        codes.append(_brute_nearest_even(min(abs(float(q)), 6.0), e2) | (8 if np.signbit(q) else 0))
                for i in range(8):
                    packed[g, n, b * 8 + i] = codes[2 * i] | (codes[2 * i + 1] << 4)
    return packed, scales, scale2


def test_quantizer_matches_independent_derivation():
    w = synth.projection_weights(synth.Shape(T=1, H=64, E=2, k=1, I=16), seed=3, layer=0, proj="gate_up").numpy()
    w[1, 3, :16] = 0.0           # an all-zero block
    w[1, 4, 5] = -0.0            # a negative zero in a live block
    p, s, s2 = oracle.quantize(w)
    p2, s_2, s2_2 = _numpy_quantize(w)
    assert np.array_equal(s2, s2_2)
    assert np.array_equal(s, s_2)
    assert np.array_equal(p, p2)


def test_quantizer_largest_block_gets_scale_448_and_zero_tensor():
    w = synth.projection_weights(synth.Shape(T=1, H=128, E=3, k=1, I=32), seed=4, layer=0, proj="down").numpy()
    p, s, s2 = oracle.quantize(w)
    for g in range(w.shape[0]):
        blocks = np.abs(w[g]).reshape(w.shape[1], -1, 16).max(-1)
        n, b = np.unravel_index(np.argmax(blocks), blocks.shape)
        assert s[g, n, b] == 0x7E
        assert s2[g] == np.float32(np.abs(w[g]).max() / np.float32(2688))
    z = np.zeros((1, 4, 32), np.float32)
    p, s, s2 = oracle.quantize(z)
    assert not p.any() and not s.any() and s2[0] == 0


def test_quantizer_round_trip_exact_for_representable_weights():
    rng = np.random.default_rng(5)
    G, N, K = 2, 8, 64
    codes = rng.integers(0, 16, size=(G, N, K))
    codes[..., ::16] = 7                        # every block holds a +6 so its amax is 6*scale
    sc = rng.integers(0x20, 0x60, size=(G, N, K // 16))
    sc[:, 0, 0] = 0x7E                           # the largest block of each group gets 448
    scale2 = np.array([0.125, 2.0 ** -20], np.float32)
    e2 = np.array([oracle.e2m1_value(c) for c in range(16)])
    e4 = np.array([oracle.e4m3_value(c) for c in range(256)])
    w = (e2[codes] * np.repeat(e4[sc], 16, axis=-1) * scale2[:, None, None]).astype(np.float32)
    p, s, s2 = oracle.quantize(w)
    assert np.array_equal(s2, scale2)
    assert np.array_equal(s, sc.astype(np.uint8))
    # code 8 (-0) and code 0 (+0) decode to the same value; compare values, then codes off zero
    deq = oracle.dequantize(p, s, s2)
    assert np.array_equal(deq, w.astype(np.float64))
    lo = p & 0xF
    hi = p >> 4
    got = np.stack([lo, hi], -1).reshape(G, N, K)
    nz = (codes % 8) != 0
    assert np.array_equal(got[nz], codes[nz])


def test_dequantize_layout_low_nibble_is_even_k():
    packed = np.zeros((1, 1, 8), np.uint8)
    packed[0, 0, 0] = 0x2 | (0x5 << 4)   # k=0 -> code 2 (1.0), k=1 -> code 5 (3.0)
    scales = np.full((1, 1, 1), 0x38, np.uint8)
    out = oracle.dequantize(packed, scales, np.ones(1, np.float32))
    assert out[0, 0, 0] == 1.0 and out[0, 0, 1] == 3.0 and not out[0, 0, 2:].any()


# ----------------------------------------------------------------------------- routing

def _nan_as_neg_inf(l):
    l = np.array(l, np.float64)
    l[np.isnan(l)] = -np.inf
    return l


def test_topk_brute_force_tiny():
    rng = np.random.default_rng(0)
    for trial in range(400):
        E = int(rng.integers(2, 9))
        k = int(rng.integers(1, min(E, 3) + 1))
        pool = np.array([-1.0, 0.0, -0.0, 0.5, 2.0, np.nan, -np.inf, 1.5], np.float32)
        l = pool[rng.integers(0, len(pool), size=E)] if trial % 2 else rng.standard_normal(E).astype(np.float32)
        ids, w = oracle.route(l[None, :], k)
        key = _nan_as_neg_inf(l)
        # the selected set: every selected expert beats every other under (value desc, index asc)
        best = None
        for sub in itertools.combinations(range(E), k):
            rest = [e for e in range(E) if e not in sub]
            if all((key[a] > key[b]) or (key[a] == key[b] and a < b) for a in sub for b in rest):
                assert best is None
                best = sub
        assert set(ids[0]) == set(best)
        ranked = sorted(best, key=lambda e: (-key[e], e))
        assert list(ids[0]) == ranked


def test_topk_matches_numpy_stable_argsort_with_ties():
    rng = np.random.default_rng(1)
    T, E, k = 64, 32, 5
    l = rng.integers(-3, 4, size=(T, E)).astype(np.float32)   # many exact ties
    l[3, :] = np.nan
    l[4, ::2] = np.nan
    l[5, :] = -np.inf
    l[6, 7] = -0.0
    ids, _ = oracle.route(l, k)
    ref = np.argsort(-_nan_as_neg_inf(l), axis=1, kind="stable")[:, :k]
    assert np.array_equal(ids, ref)


def test_topk_matches_torch_topk_on_distinct_logits():
    l = synth.router_logits(16, 512, seed=9)
    ids, _ = oracle.route(l, 10)
    assert np.array_equal(ids, torch.topk(l, 10, dim=1).indices.numpy())


def test_route_weights_are_renormalised_softmax():
    l = synth.router_logits(32, 64, seed=2, bias="normal")
    ids, w = oracle.route(l, 6)
    full = torch.softmax(l.double(), dim=1)
    picked = torch.gather(full, 1, torch.from_numpy(ids).long())
    ref = picked / picked.sum(1, keepdim=True)
    np.testing.assert_allclose(w, ref.numpy(), rtol=1e-13, atol=0)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=0, atol=1e-12)
    assert all(len(set(r)) == 6 for r in ids)


def test_route_degenerate_rows():
    l = np.zeros((3, 8), np.float32)
    l[0, :] = -np.inf                 # no finite logit: weights are 0
    l[1, :] = np.nan
    l[2, [1, 6]] = np.inf             # two +inf share the mass
    ids, w = oracle.route(l, 3)
    assert list(ids[0]) == [0, 1, 2] and not w[0].any()
    assert list(ids[1]) == [0, 1, 2] and not w[1].any()
    assert list(ids[2]) == [1, 6, 0] and list(w[2]) == [0.5, 0.5, 0.0]


# ----------------------------------------------------------------------------- permutation

def test_permute_matches_stable_argsort_and_invariants():
    l = synth.router_logits(300, 40, seed=3, bias="zipf")
    ids, _ = oracle.route(l, 4)
    counts, offsets, sorted_slot, slot_pos = oracle.permute(ids, 40)
    flat = ids.reshape(-1)
    assert np.array_equal(counts, np.bincount(flat, minlength=40))
    assert offsets[0] == 0 and np.array_equal(offsets[1:], np.cumsum(counts))
    assert np.array_equal(sorted_slot, np.argsort(flat, kind="stable"))
    assert np.array_equal(slot_pos[sorted_slot], np.arange(flat.size))
    assert np.array_equal(np.sort(sorted_slot), np.arange(flat.size))   # each slot exactly once
    assert counts.sum() == 300 * 4


# ----------------------------------------------------------------------------- layer

def _const_weights(vals, N, K):
    """packed/scales/scale2 (scale2 = 1) for groups whose rows are constants: vals[g] is a list
    of (row_count, value) and each value is written as an e2m1 code times an e4m3 scale."""
    e2 = {oracle.e2m1_value(c): c for c in list(range(1, 8)) + list(range(9, 16))}

    def encode(v):
        for sc in (0x38, 0x30, 0x28, 0x40):        # scales 1, 0.5, 0.25, 2
            if v / oracle.e4m3_value(sc) in e2:
                return e2[v / oracle.e4m3_value(sc)], sc
        raise ValueError(v)

    G = len(vals)
    packed = np.zeros((G, N, K // 2), np.uint8)
    scales = np.zeros((G, N, K // 16), np.uint8)
    for g, v in enumerate(vals):
        rows = []
        for count, val in v:
            rows += [val] * count
        for n, val in enumerate(rows):
            c, sc = encode(val)
            packed[g, n, :] = c | (c << 4)
            scales[g, n, :] = sc
    return packed, scales, np.ones(G, np.float32)


def silu(v):
    return v / (1.0 + math.exp(-v))


def test_hand_layer_case_a_constant_experts():
    H, I, E, k = 16, 16, 2, 2
    x = torch.tensor([[c / 16 for c in range(16)]], dtype=torch.bfloat16)
    logits = torch.tensor([[0.5, -0.25]], dtype=torch.float32)
    gate = [1.0, -0.5, 0.5]
    up = [0.5, 1.5, 1.0]
    dn = [0.25, 1.0, 0.5]
    gu = _const_weights([[(I, gate[g]), (I, up[g])] for g in range(3)], 2 * I, H)
    d = _const_weights([[(H, dn[g])] for g in range(3)], H, I)
    out, h, y = oracle.moe_forward(x, logits, gu, d, k, dumps=True)
    X = 7.5
    w0 = 1.0 / (1.0 + math.exp(-0.75))
    w = [w0, 1.0 - w0]
    ref = sum(w[e] * dn[e] * I * silu(gate[e] * X) * up[e] * X for e in range(2))
    ref += dn[2] * I * silu(gate[2] * X) * up[2] * X
    np.testing.assert_allclose(out, ref, rtol=1e-14)
    np.testing.assert_allclose(h[0, 2], silu(0.5 * X) * X, rtol=1e-14)


def test_hand_layer_case_b_single_paths():
    H, I = 32, 16
    x = synth.activations(1, H, seed=12)
    xv = x.float().double().numpy()[0]
    gu_p = np.zeros((1, 2 * I, H // 2), np.uint8)
    gu_s = np.full((1, 2 * I, H // 16), 0x38, np.uint8)
    gu_p[0, 5, 17 // 2] = 5 << 4          # gate[5, 17] = 3.0 (odd k -> high nibble)
    gu_p[0, I + 5, 2 // 2] = 4            # up[5, 2] = 2.0 (even k -> low nibble)
    gu_s[0, I + 5, 0] = 0x30              # with that block's scale 0.5
    dn_p = np.zeros((1, H, I // 2), np.uint8)
    dn_s = np.full((1, H, I // 16), 0x38, np.uint8)
    dn_p[0, 30, 5 // 2] = 6 << 4          # down[30, 5] = 4.0
    logits = torch.zeros(1, 1)
    out, h, y = oracle.moe_forward(x, logits, (gu_p, gu_s, np.ones(1, np.float32)),
                                   (dn_p, dn_s, np.ones(1, np.float32)), 1, has_shared=0, dumps=True)
    h5 = silu(3.0 * xv[17]) * (2.0 * 0.5) * xv[2]
    want_h = np.zeros(I)
    want_h[5] = h5
    want = np.zeros(H)
    want[30] = 4.0 * h5
    np.testing.assert_allclose(h[0, 0], want_h, rtol=1e-15, atol=0)
    np.testing.assert_allclose(out[0], want, rtol=1e-15, atol=0)


def _small_layer(T=6, H=64, E=6, k=3, I=32, seed=21):
    shape = synth.Shape(T=T, H=H, E=E, k=k, I=I)
    x = synth.activations(T, H, seed)
    logits = synth.router_logits(T, E, seed)
    gu = oracle.quantize(synth.projection_weights(shape, seed, 0, "gate_up"))
    d = oracle.quantize(synth.projection_weights(shape, seed, 0, "down"))
    return shape, x, logits, gu, d


def test_layer_against_torch_fp64_composition():
    """Same layer composed from library routines: torch float8 decoding of the scales, torch
    matmul, softmax and topk (distinct logits), fp64 throughout."""
    shape, x, logits, gu, d = _small_layer()
    out = oracle.moe_forward(x, logits, gu, d, shape.k)
    e2 = torch.tensor([float(v) for _, v in _golden("e2m1_values.txt")], dtype=torch.float64)

    def deq(p, s, s2):
        p = torch.from_numpy(p).long()
        codes = torch.stack([p & 15, p >> 4], -1).reshape(p.shape[0], p.shape[1], -1)
        sc = torch.from_numpy(s).view(torch.float8_e4m3fn).double().repeat_interleave(16, -1)
        return e2[codes] * sc * torch.from_numpy(s2).double()[:, None, None]

    Wgu, Wd = deq(*gu), deq(*d)
    xd = x.double()
    top = torch.topk(logits.double(), shape.k, dim=1)
    wts = torch.softmax(top.values, dim=1)
    ref = torch.zeros(shape.T, shape.H, dtype=torch.float64)
    for t in range(shape.T):
        for j, e in enumerate(list(top.indices[t]) + [shape.E]):
            gu_out = Wgu[e] @ xd[t]
            a = torch.nn.functional.silu(gu_out[:shape.I]) * gu_out[shape.I:]
            yv = Wd[e] @ a
            ref[t] += (wts[t, j] if j < shape.k else 1.0) * yv
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-10, atol=1e-12)


def test_layer_invariants():
    shape, x, logits, gu, d = _small_layer(T=5, E=4, k=2, seed=33)
    base, h, y = oracle.moe_forward(x, logits, gu, d, shape.k, dumps=True)
    # doubling the routed experts' down scale2 doubles the routed part only
    d2 = (d[0], d[1], d[2].copy())
    d2[2][:shape.E] *= 2
    out2 = oracle.moe_forward(x, logits, gu, d2, shape.k)
    shared = y[:, shape.k, :]
    np.testing.assert_allclose(out2 - shared, 2 * (base - shared), rtol=1e-12, atol=1e-12)
    # identical routed experts: the output does not depend on the routing
    gu_same = tuple(np.repeat(a[:1], shape.E + 1, 0) for a in gu[:2]) + (np.repeat(gu[2][:1], shape.E + 1),)
    d_same = tuple(np.repeat(a[:1], shape.E + 1, 0) for a in d[:2]) + (np.repeat(d[2][:1], shape.E + 1),)
    o1 = oracle.moe_forward(x, logits, gu_same, d_same, shape.k)
    o2 = oracle.moe_forward(x, torch.flip(logits, [1]), gu_same, d_same, shape.k)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-12)
    # a token subset gives the same rows as the full evaluation, and threading does not matter
    sub = oracle.moe_forward(x, logits, gu, d, shape.k, tokens=[4, 1], n_threads=1)
    np.testing.assert_array_equal(sub, base[[4, 1]])


# ----------------------------------------------------------------------------- router GEMM

def _golden_case(tag):
    for line in open(os.path.join(os.path.dirname(__file__), "golden", "hand_layer.txt")):
        if line.startswith(tag + " "):
            return dict(kv.split("=") for kv in line.split()[1:])
    raise KeyError(tag)


def test_router_constant_rows_closed_form():
    g = _golden_case("caseR1")
    H, E = int(g["H"]), int(g["E"])
    x = torch.tensor([[c / 16 for c in range(H)]], dtype=torch.bfloat16)
    p, sc, _ = _const_weights([[(1, 1.0), (1, -0.5), (1, 6.0)]], E, H)
    logits = oracle.router_logits(x, (p, sc, np.array([0.25], np.float32)))
    want = [float(g["l0"]), float(g["l1"]), float(g["l2"])]
    np.testing.assert_array_equal(logits[0], want)


def test_router_single_weights_pin_row_column_nibble_and_scale():
    g = _golden_case("caseR2")
    H, E, c0, c1 = int(g["H"]), int(g["E"]), int(g["c0"]), int(g["c1"])
    x = synth.activations(3, H, seed=31)
    xv = x.float().double().numpy()
    p = np.zeros((E, H // 2), np.uint8)
    sc = np.full((E, H // 16), 0x38, np.uint8)
    p[0, c0 // 2] = 3 << 4           # 1.5 in the high nibble (odd column)
    sc[0, c0 // 16] = 0x40           # that block's scale 2.0
    p[1, c1 // 2] = 14               # -4.0 in the low nibble (even column)
    logits = oracle.router_logits(x, (p, sc, np.ones(1, np.float32)))
    np.testing.assert_array_equal(logits[:, 0], 3.0 * xv[:, c0])
    np.testing.assert_array_equal(logits[:, 1], -4.0 * xv[:, c1])


def test_router_is_linear_in_scale2_and_permutes_with_rows():
    H, E, T = 64, 8, 5
    x = synth.activations(T, H, seed=32)
    w = synth.expert_weight(E, H, seed=33, layer=0, group=0, proj="gate_up")
    p, sc, s2 = oracle.quantize(w.numpy()[None])
    a = oracle.router_logits(x, (p[0], sc[0], s2))
    b = oracle.router_logits(x, (p[0], sc[0], 2 * s2))
    np.testing.assert_array_equal(b, 2 * a)
    perm = np.array([3, 0, 7, 1, 6, 2, 5, 4])
    c = oracle.router_logits(x, (p[0][perm], sc[0][perm], s2))
    np.testing.assert_array_equal(c, a[:, perm])


# ----------------------------------------------------------------------------- FP8-activation arm
# (the "long-context cold prefill" issue: e4m3 x e4m3 transposed kernels, weights re-quantized to
# e4m3, option (a) a per-token-row e4m3 activation scale applied in the f32 epilogue)

def test_fp8_row_rule_closed_form():
    # amax 4: inv = 448 / 4 = 112 and scale = 4 / 448; every product is an e4m3 value
    codes, scale = oracle.quant_rows_e4m3(np.array([[1.0, 2.0, -4.0, 0.5]], np.float32))
    assert codes.tolist() == [[0x6E, 0x76, 0xFE, 0x66]]           # 112, 224, -448, 56
    assert scale[0] == np.float32(4.0) / np.float32(448.0)
    # amax 448: inv = scale = 1, so the codes are the nearest-even e4m3 of the values:
    # 38 is the midpoint of 36 (0x61) and 40 (0x62) -> the even code; 37.9 -> 36; 2^-9 is the
    # smallest subnormal; 2^-10 is the midpoint of 0 and 2^-9 -> 0
    row = np.array([[448.0, 38.0, -38.0, 37.9, 2.0 ** -9, 2.0 ** -10, 0.0, -448.0]], np.float32)
    codes, scale = oracle.quant_rows_e4m3(row)
    assert codes.tolist() == [[0x7E, 0x62, 0xE2, 0x61, 0x01, 0x00, 0x00, 0xFE]]
    assert scale[0] == 1.0
    # an all-zero row keeps scale 1 and codes 0
    codes, scale = oracle.quant_rows_e4m3(np.zeros((1, 16), np.float32))
    assert not codes.any() and scale[0] == 1.0


def test_fp8_row_rule_matches_torch_float8_on_random_rows():
    rng = np.random.default_rng(5)
    v = (rng.standard_normal((64, 256)) * np.exp2(rng.integers(-20, 20, (64, 1)))).astype(np.float32)
    v[3, 17] *= 40.0                                              # an outlier row
    codes, scale = oracle.quant_rows_e4m3(v)
    amax = np.abs(v).max(axis=1)
    inv = (np.float32(448.0) / amax).astype(np.float32)
    q = (v * inv[:, None]).astype(np.float32)                     # one fp32 multiply
    ref = torch.from_numpy(np.minimum(np.abs(q), 448.0) * np.sign(q)).to(torch.float8_e4m3fn)
    assert np.array_equal(codes, ref.view(torch.uint8).numpy())
    assert np.array_equal(scale, (amax / np.float32(448.0)).astype(np.float32))


def _fp8_exact_nvfp4(G, N, K, seed):
    """NVFP4 weights whose values are e4m3-exact with row amax 448 (so the re-quantization is
    lossless with row scale 1): e2m1 codes of one significant bit (0, 0.5, 1, 2, 4) times normal
    e4m3 block scales <= 112, and element 0 of every row is 4 x 112 = 448."""
    rng = np.random.default_rng(seed)
    one_bit = [0, 1, 2, 4, 6, 9, 10, 12, 14]                      # 0, +-0.5, +-1, +-2, +-4
    codes = rng.choice(one_bit, size=(G, N, K))
    scl = rng.choice([c for c in range(0x10, 0x6F)], size=(G, N, K // 16))   # 2^-5 .. 112
    codes[:, :, 0] = 6
    scl[:, :, 0] = 0x6E
    packed = (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)
    return packed, scl.astype(np.uint8)


def test_fp8_weight_requant_lossless_on_e4m3_exact_weights():
    packed, scl = _fp8_exact_nvfp4(2, 8, 64, 11)
    codes, rs = oracle.prepare_fp8(packed, scl)
    assert np.all(rs == 1.0)
    deq = oracle.dequantize(packed, scl, np.ones(2, np.float32))
    vals = np.vectorize(oracle.e4m3_value)(codes.astype(int))
    assert np.array_equal(vals, deq)


def test_fp8_weight_requant_is_the_row_rule_on_dequantized_rows():
    shape = synth.Shape(T=1, H=128, E=3, k=1, I=32)
    p, s_, _ = oracle.quantize(synth.projection_weights(shape, 4, 0, "gate_up"))
    codes, rs = oracle.prepare_fp8(p, s_)
    deq = oracle.dequantize(p, s_, np.ones(p.shape[0], np.float32)).astype(np.float32)   # exact in fp32
    c2, s2 = oracle.quant_rows_e4m3(deq.reshape(-1, deq.shape[-1]))
    assert np.array_equal(codes.reshape(c2.shape), c2) and np.array_equal(rs.reshape(-1), s2)


def _bf16_rne(a):
    """Round fp64 values to bf16 (8 significant bits, ties to even) with numpy."""
    m, e = np.frexp(a)
    return np.ldexp(np.round(np.ldexp(m, 8)), e - 8)   # np.round: half to even


def test_fp8_layer_gate_up_equals_w4a16_on_exact_inputs_and_down_wiring():
    """With e4m3-exact weights (row scale 1) and x rows whose quantization is exact (values e4m3
    x 2^-8 with amax 1.75, so inv = 256 and scale = 2^-8), the FP8 layer's SiLU(g)*u equals the
    W4A16 layer's.  Down weights 448 x a permutation (output n reads h element n mod I) then make
    y[n] = 448 * scale2 * (the e4m3-quantized bf16 h)[n mod I], checked through the row rule."""
    T, H, E, k, I = 5, 64, 3, 2, 32
    G = E + 1
    rng = np.random.default_rng(3)
    gp, gs = _fp8_exact_nvfp4(G, 2 * I, H, 12)
    g2 = np.array([0.5, 0.25, 1.0, 2.0], np.float32)
    # down: row n has the single value 448 = 4 x 112 at column n mod I
    dcodes = np.zeros((G, H, I), np.int64)
    dscl = np.full((G, H, I // 16), 0x38, np.int64)
    for n in range(H):
        dcodes[:, n, n % I] = 6
        dscl[:, n, (n % I) // 16] = 0x6E
    dp = (dcodes[..., 0::2] | (dcodes[..., 1::2] << 4)).astype(np.uint8)
    ds = dscl.astype(np.uint8)
    d2 = np.array([1.0, 0.5, 2.0, 0.25], np.float32)
    ev = np.array([oracle.e4m3_value(c) for c in range(0x08, 0x7F)])   # positive normal e4m3
    xv = rng.choice(ev, size=(T, H)) * rng.choice([-1.0, 1.0], size=(T, H))
    xv[:, 0] = 448.0
    xv = xv * 2.0 ** -8
    x = torch.from_numpy(xv.astype(np.float32)).to(torch.bfloat16)
    assert torch.equal(x.float().double(), torch.from_numpy(xv))
    logits = torch.from_numpy(rng.standard_normal((T, E)).astype(np.float32))
    gc, gr = oracle.prepare_fp8(gp, gs)
    dc, dr = oracle.prepare_fp8(dp, ds)
    assert np.all(gr == 1.0) and np.all(dr == 1.0)
    _, h8, y8 = oracle.moe_forward_fp8(x, logits, (gc, gr, g2), (dc, dr, d2), k, 1, dumps=True)
    _, h16, _ = oracle.moe_forward(x, logits, (gp, gs, g2), (dp, ds, d2), k, 1, dumps=True)
    np.testing.assert_allclose(h8, h16, rtol=1e-12, atol=0)
    ids, _ = oracle.route(logits, k)
    groups = np.concatenate([ids, np.full((T, 1), E)], axis=1)     # rank j's group, shared last
    hq, hs = oracle.quant_rows_e4m3(_bf16_rne(h8.reshape(-1, I)).astype(np.float32))
    hval = np.vectorize(oracle.e4m3_value)(hq.astype(int)) * hs[:, None].astype(np.float64)
    hval = hval.reshape(T, k + 1, I)
    want = 448.0 * d2[groups][:, :, None] * hval[:, :, np.arange(H) % I]
    np.testing.assert_allclose(y8, want, rtol=1e-15, atol=0)
