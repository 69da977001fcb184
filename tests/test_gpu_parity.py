"""GPU parity of every stage and of moe_forward against the CPU oracle (needs a GB300).

Integer results (top-k ids, counts, offsets, permutation, quantized bytes) must be bit-exact;
floating-point results must satisfy the layer tolerance (max |err| <= 2e-2 * row RMS and mean
relative error <= 3e-3) against the oracle's fp64 values.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from moe_cases import Layer, bf16_round_bits, check_bf16_stage_close, check_layer_close, moe_shape, to_np

pytestmark = pytest.mark.gpu

# (T, H, E, k, I, has_shared, logit bias, seed): the tiny workload itself, every arm, the arm
# boundaries (T = 8 / 9, 64 / 65), k = 16, no shared expert, E = 1024, ragged tails everywhere.
SMALL = [
    (4, 256, 16, 2, 128, 1, "none", 0),
    (1, 256, 16, 2, 128, 1, "none", 101),
    (7, 384, 24, 3, 256, 1, "normal", 102),
    (64, 256, 32, 4, 128, 1, "zipf", 103),
    (65, 256, 32, 4, 128, 1, "zipf", 104),
    (200, 512, 40, 6, 256, 1, "zipf", 105),
    (300, 256, 16, 16, 128, 0, "none", 106),
    (3000, 256, 64, 8, 128, 1, "normal", 107),
    (16, 128, 1024, 16, 128, 1, "none", 108),
    # one-launch decode arm (T <= 8, H % 512 == 0, H <= 4096, I % 256 == 0, I <= 1024): E = 1024
    # with k = 16 and no shared expert, a skewed batch where experts are shared by several tokens
    (3, 512, 16, 4, 256, 1, "none", 112),
    (8, 1024, 64, 8, 256, 1, "zipf", 113),
    (5, 512, 1024, 16, 256, 0, "none", 114),
    # tcgen05 arm (T > 8, H and I multiples of 256): ragged token tiles, several tiles per
    # expert, no shared expert, the N tail of a single 16-column step, single-token experts
    (9, 256, 16, 2, 256, 1, "none", 116),
    (48, 512, 32, 4, 256, 1, "zipf", 117),
    (129, 256, 8, 2, 256, 0, "none", 109),
    (1000, 512, 64, 8, 256, 1, "zipf", 110),
    (700, 1024, 32, 6, 512, 1, "normal", 111),
    # k = 16 on the tcgen05 arm with enough tokens that each thread of the compact-y combine's
    # resident grid (one CTA per SM above 10 ranks) walks several (token, 8-column) units
    (2000, 512, 64, 16, 256, 1, "zipf", 145),
]


def _small_layer(case):
    T, H, E, k, I, sh, bias, seed = case
    return Layer(synth.Shape(T=T, H=H, E=E, k=k, I=I, has_shared=sh), seed, logit_bias=bias)


@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"T{c[0]}_H{c[1]}_E{c[2]}_k{c[3]}_I{c[4]}_sh{c[5]}")
def test_small_layers_all_stages(cuda_lib, case):
    moe = cuda_lib
    L = _small_layer(case)
    s = L.shape
    ms = moe_shape(moe, s)
    gu, dn = L.gpu_weights(moe)
    ogu, odn = L.oracle_weights()
    # quantizer: identical bytes
    for q, o in ((gu, ogu), (dn, odn)):
        assert np.array_equal(q.packed.cpu().numpy(), o[0])
        assert np.array_equal(q.scales.cpu().numpy(), o[1])
        assert np.array_equal(q.scale2.cpu().numpy(), o[2])
    x, logits = L.x.cuda(), L.logits.cuda()
    ws = moe.workspace(ms)
    # route
    ids, w = moe.route_topk(logits, ms)
    oids, ow = oracle.route(L.logits, s.k)
    assert np.array_equal(ids.cpu().numpy(), oids)
    np.testing.assert_allclose(w.cpu().numpy(), ow, rtol=2e-6, atol=1e-7)
    # permute
    counts, offsets, sorted_slot, slot_pos = moe.permute(ids, ms, ws)
    oc, oo, oss, osp = oracle.permute(oids, s.E)
    assert np.array_equal(counts.cpu().numpy(), oc)
    assert np.array_equal(offsets.cpu().numpy(), oo)
    assert np.array_equal(sorted_slot.cpu().numpy(), oss)
    assert np.array_equal(slot_pos.cpu().numpy(), osp)
    # stages vs the oracle's dumps
    out_ref, h_ref, y_ref = oracle.moe_forward(L.x, L.logits, ogu, odn, s.k, s.has_shared, dumps=True)
    h = moe.grouped_gate_up(x, sorted_slot, offsets, gu, ms, ws)
    y = moe.grouped_down(h, offsets, dn, ms, ws)
    S = s.T * s.k
    slot_of_row = oss  # routed row p holds slot oss[p] = t*k + j
    t_of, j_of = slot_of_row // s.k, slot_of_row % s.k
    check_bf16_stage_close(to_np(h[:S]), h_ref[t_of, j_of], "h routed")
    check_layer_close(to_np(y[:S]), y_ref[t_of, j_of], "y routed")
    if s.has_shared:
        check_bf16_stage_close(to_np(h[S:]), h_ref[:, s.k], "h shared")
        check_layer_close(to_np(y[S:]), y_ref[:, s.k], "y shared")
    for fp32 in (False, True):
        out = moe.combine(y, slot_pos, w, ms, out_fp32=fp32)
        check_layer_close(to_np(out), out_ref, f"combine fp32={fp32}", rounded_bf16=not fp32)
    # the fused forward, both output types
    for fp32 in (False, True):
        out = torch.full((s.T, s.H), float("nan"), device="cuda",
                         dtype=torch.float32 if fp32 else torch.bfloat16)
        moe.forward(x, logits, gu, dn, ms, ws, out=out, out_fp32=fp32)
        torch.cuda.synchronize()
        assert moe.device_status(ws) == 0
        check_layer_close(to_np(out), out_ref, f"forward fp32={fp32} arm={moe.forward_arm(ms)}",
                          rounded_bf16=not fp32)


def test_forward_arm_selection(cuda_lib):
    moe = cuda_lib
    arm = lambda **kw: moe.forward_arm(moe.Shape(**{**dict(T=1, H=2048, I=512, E=512, k=10), **kw}))
    assert arm(T=1) == 0 and arm(T=8) == 0 and arm(T=4, H=4096, I=1024) == 0 and arm(T=4, H=1024, I=256) == 0
    assert arm(T=4, I=128) == 1 and arm(T=4, I=640) == 1   # the one-launch kernel wants I % 256 == 0
    assert arm(T=4, H=8192) == 1 and arm(T=4, I=2048) == 1
    assert arm(T=4, H=256) == 1 and arm(T=9, I=128) == 1 and arm(T=64, I=128) == 1
    assert arm(T=9) == 2 and arm(T=64) == 2 and arm(T=65) == 2 and arm(T=4096) == 2
    assert arm(T=65, I=128) == 3
    assert arm(H=100) == -1


def _compact_y_bound(y, slot_pos, w, ms, staged):
    """Largest difference the tensor-core forward's compact y allows against the staged combine
    over fp32 y: every y value is rounded once to f16 (relative error at most 2^-11, taken as
    2^-10 with the products' roundings) before it is weighted and summed, plus fp32 rounding of
    the sums and the absolute error of values in f16's subnormal range."""
    S, T, k = ms.S, ms.T, ms.k
    valid = y if ms.has_shared else y[:S]     # rows S.. hold the shared expert's outputs only if it exists
    rows = slot_pos.view(T, k).long()
    b = (w.abs()[:, :, None] * valid.abs()[rows]).sum(1)
    if ms.has_shared:
        b = b + y[S:].abs()
    return 2.0 ** -10 * b + 1e-6 * staged.abs() + 1e-6 * valid.abs().max() + 1e-30


def test_forward_deterministic_and_matches_stages(cuda_lib):
    """Repeated forwards are bit-identical, and moe_forward matches the staged calls (route,
    permute, gate_up, down, combine over fp32 y): bit for bit on the CUDA-core grouped arm; on the
    tensor-core arm, which hands y to the combine as f16 of the raw accumulator, within one f16
    rounding of each weighted y value."""
    moe = cuda_lib
    for case in (SMALL[2], SMALL[4], SMALL[5], SMALL[7], SMALL[12], SMALL[14], SMALL[15], SMALL[16], SMALL[17]):
        L = _small_layer(case)
        ms = moe_shape(moe, L.shape)
        gu, dn = L.gpu_weights(moe)
        x, logits = L.x.cuda(), L.logits.cuda()
        ws = moe.workspace(ms)
        a = moe.forward(x, logits, gu, dn, ms, ws, out_fp32=True)
        b = moe.forward(x, logits, gu, dn, ms, ws, out_fp32=True)
        assert torch.equal(a, b)
        if moe.forward_arm(ms) < 2:
            continue
        ids, w = moe.route_topk(logits, ms)
        _, offsets, sorted_slot, slot_pos = moe.permute(ids, ms, ws)
        h = moe.grouped_gate_up(x, sorted_slot, offsets, gu, ms, ws)
        y = moe.grouped_down(h, offsets, dn, ms, ws)
        staged = moe.combine(y, slot_pos, w, ms, out_fp32=True)
        fused = moe.forward(x, logits, gu, dn, ms, ws, out_fp32=True)
        torch.cuda.synchronize()
        assert moe.device_status(ws) == 0
        if moe.forward_arm(ms) == 2:
            bound = _compact_y_bound(y, slot_pos, w, ms, staged)
            err = (fused - staged).abs()
            assert (err <= bound).all(), (case, float((err / bound).max()))
        else:
            assert torch.equal(fused.view(torch.int32), staged.view(torch.int32)), case


def test_one_launch_consecutive_calls(cuda_lib):
    """Consecutive one-launch forwards on one workspace alternate the kernel's counter sets (the
    parity of its launch count): five calls with different token/logit pairings, so the routing
    differs from call to call, each against the oracle."""
    moe = cuda_lib
    L = _small_layer((8, 1024, 64, 8, 256, 1, "zipf", 113))
    s = L.shape
    ms = moe_shape(moe, s)
    assert moe.forward_arm(ms) == 0
    gu, dn = L.gpu_weights(moe)
    ogu, odn = L.oracle_weights()
    ws = moe.workspace(ms)
    for r in range(5):
        x = torch.roll(L.x, shifts=r, dims=0)
        lg = torch.roll(L.logits, shifts=3 * r, dims=0)
        out = torch.full((s.T, s.H), float("nan"), device="cuda", dtype=torch.bfloat16)
        moe.forward(x.cuda(), lg.cuda(), gu, dn, ms, ws, out=out)
        torch.cuda.synchronize()
        assert moe.device_status(ws) == 0
        ref = oracle.moe_forward(x, lg, ogu, odn, s.k, s.has_shared)
        check_layer_close(to_np(out), ref, f"call {r}", rounded_bf16=True)


def test_device_timeout_is_reported_without_fault(cuda_lib):
    """The decode kernel's bounded wait, run on a barrier nothing arrives at with a 2 ms limit,
    records MOE_ERR_DEVICE_TIMEOUT in the status word; the read clears it and the context stays
    usable (a forward afterwards is correct)."""
    moe = cuda_lib
    L = _small_layer((3, 512, 16, 4, 256, 1, "none", 112))
    s = L.shape
    ms = moe_shape(moe, s)
    ws = moe.workspace(ms)
    assert moe.device_status(ws) == 0
    moe.debug_timeout_probe(ws, 2_000_000)
    assert moe.device_status(ws) == -6   # MOE_ERR_DEVICE_TIMEOUT
    assert moe.device_status(ws) == 0
    gu, dn = L.gpu_weights(moe)
    ogu, odn = L.oracle_weights()
    out = torch.full((s.T, s.H), float("nan"), device="cuda", dtype=torch.bfloat16)
    moe.forward(L.x.cuda(), L.logits.cuda(), gu, dn, ms, ws, out=out)
    torch.cuda.synchronize()
    assert moe.device_status(ws) == 0
    check_layer_close(to_np(out), oracle.moe_forward(L.x, L.logits, ogu, odn, s.k, s.has_shared), "after the probe",
                      rounded_bf16=True)


def test_forward_profiled_matches_forward(cuda_lib):
    """forward_profiled on the default stream (no capture) gives forward's bytes and five
    ordered stage events, for every arm."""
    moe = cuda_lib
    for case in (SMALL[0], SMALL[2], SMALL[5]):
        L = _small_layer(case)
        ms = moe_shape(moe, L.shape)
        gu, dn = L.gpu_weights(moe)
        x, logits = L.x.cuda(), L.logits.cuda()
        ws = moe.workspace(ms)
        a = moe.forward(x, logits, gu, dn, ms, ws, out_fp32=True)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        for e in ev:
            e.record()
        b = torch.full_like(a, float("nan"))
        moe.forward_profiled(x, logits, gu, dn, ms, ws, b, ev, out_fp32=True)
        torch.cuda.synchronize()
        assert torch.equal(a, b)
        assert all(ev[i].elapsed_time(ev[i + 1]) >= 0.0 for i in range(4))
        assert moe.device_status(ws) == 0


def test_route_edge_rows(cuda_lib):
    moe = cuda_lib
    E, k = 16, 4
    l = np.random.default_rng(3).standard_normal((9, E)).astype(np.float32)
    l[0] = 1.0                                  # all tied: lowest indices win
    l[1] = np.nan                               # all NaN: weights 0
    l[2] = -np.inf
    l[3, ::2] = np.nan                          # NaN never wins
    l[4, [3, 9]] = np.inf                       # two +inf share the mass
    l[5, :] = 0.0
    l[5, 7] = -0.0                              # -0 ties +0
    l[6, :] = np.float32(2.0)
    l[6, 5] = np.float32(2.0000002)             # one ulp above the tie
    l[7, :k] = -np.inf                          # -inf are ranked last among finite
    l[8] = np.arange(E)[::-1].astype(np.float32)
    ms = moe.Shape(T=9, H=128, I=128, E=E, k=k)
    ids, w = moe.route_topk(torch.from_numpy(l).cuda(), ms)
    oids, ow = oracle.route(l, k)
    assert np.array_equal(ids.cpu().numpy(), oids)
    np.testing.assert_allclose(w.cpu().numpy(), ow, rtol=2e-6, atol=1e-7)



@pytest.mark.parametrize("E,k", [(512, 10), (1024, 16), (64, 8), (24, 3)])
def test_route_rows_with_clustered_winners(cuda_lib, E, k):
    """Rows whose largest logits sit in a few lanes of the ranking warp (entries e, e + 32, ...
    share a lane), so that more than 32 entries reach the lane-maxima threshold and the ranking
    takes its k-round path; rows with ties inside one lane; random rows.  Every routing call
    (moe_route_topk, and the forward's own routing on each arm) against the oracle."""
    moe = cuda_lib
    rng = np.random.default_rng(E + k)
    T = 12
    l = rng.standard_normal((T, E)).astype(np.float32)
    l[0, ::32] += 50.0                                   # lane 0 holds the top entries
    l[1, 5::32] = 7.0                                    # ties within lane 5
    l[2, ::32] += 50.0
    l[2, 1::32] += 49.0                                  # two lanes hold them
    l[3, :] = np.float32(1.0)
    l[3, 31::32] = np.float32(1.0000001)                 # lane 31 just above the rest
    l[4, ::16] = np.nan
    l[4, 3::32] = np.inf
    ms = moe.Shape(T=T, H=256, I=256, E=E, k=k)
    ids, w = moe.route_topk(torch.from_numpy(l).cuda(), ms)
    oids, ow = oracle.route(l, k)
    assert np.array_equal(ids.cpu().numpy(), oids)
    np.testing.assert_allclose(w.cpu().numpy(), ow, rtol=2e-6, atol=1e-7)


def test_empty_batch_is_a_noop(cuda_lib):
    moe = cuda_lib
    L = _small_layer(SMALL[0])
    gu, dn = L.gpu_weights(moe)
    ms = moe.Shape(T=0, H=256, I=128, E=16, k=2)
    ws = moe.workspace(moe.Shape(T=1, H=256, I=128, E=16, k=2))
    x = torch.zeros(1, 256, dtype=torch.bfloat16, device="cuda")
    lg = torch.zeros(1, 16, device="cuda")
    out = torch.full((1, 256), 7.0, dtype=torch.bfloat16, device="cuda")
    moe.forward(x, lg, gu, dn, ms, ws, out=out)
    torch.cuda.synchronize()
    assert (out == 7.0).all()


# --------------------------------------------------------------------------- full sizes

def _full_case(w: synth.Workload, T, seed, layer=0, n_sample=None, rng_seed=0):
    shape = w.shape(T)
    L = Layer(shape, synth.layer_seed(w, seed, layer), layer=0, logit_bias=w.logit_bias,
              outlier_frac=w.outlier_frac, gen_device="cuda")
    return L


def _check_full(moe, L, tokens):
    """Routing and permutation in full (bit-exact); the layer output of the listed tokens in both
    output types: the fp32 result against the oracle with the layer tolerance, the bf16 output
    bit for bit the round-to-nearest-even of that fp32 result (and so within the tolerance plus
    the rounding's half ulp)."""
    s = L.shape
    ms = moe_shape(moe, s)
    gu, dn = L.gpu_weights(moe)
    x, logits = L.x, L.logits
    ws = moe.workspace(ms)
    out = torch.full((s.T, s.H), float("nan"), device="cuda", dtype=torch.bfloat16)
    out32 = torch.full((s.T, s.H), float("nan"), device="cuda", dtype=torch.float32)
    moe.forward(x, logits, gu, dn, ms, ws, out=out)
    moe.forward(x, logits, gu, dn, ms, ws, out=out32, out_fp32=True)
    torch.cuda.synchronize()
    assert moe.device_status(ws) == 0
    assert torch.equal(out.view(torch.int16), bf16_round_bits(out32)), "bf16 output != rounded fp32 output"
    ids, w = moe.route_topk(logits, ms)
    oids, ow = oracle.route(logits.cpu(), s.k)
    assert np.array_equal(ids.cpu().numpy(), oids)
    np.testing.assert_allclose(w.cpu().numpy(), ow, rtol=2e-6, atol=1e-7)
    counts, offsets, sorted_slot, slot_pos = moe.permute(ids, ms, ws)
    oc, oo, oss, osp = oracle.permute(oids, s.E)
    assert np.array_equal(counts.cpu().numpy(), oc)
    assert np.array_equal(offsets.cpu().numpy(), oo)
    assert np.array_equal(sorted_slot.cpu().numpy(), oss)
    assert np.array_equal(slot_pos.cpu().numpy(), osp)
    groups = L.used_groups(tokens)
    ogu, odn = L.oracle_weights(groups)
    for q, o in ((gu, ogu), (dn, odn)):
        gi = torch.tensor(groups, device="cuda")
        assert np.array_equal(q.packed[gi].cpu().numpy(), o[0][groups])
        assert np.array_equal(q.scales[gi].cpu().numpy(), o[1][groups])
        assert np.array_equal(q.scale2[gi].cpu().numpy(), o[2][groups])
    ref = oracle.moe_forward(x.cpu(), logits.cpu(), ogu, odn, s.k, s.has_shared, tokens=tokens)
    sel = torch.tensor(tokens, device="cuda")
    check_layer_close(to_np(out32[sel]), ref, "forward fp32, checked rows")
    check_layer_close(to_np(out[sel]), ref, "forward bf16, checked rows", rounded_bf16=True)
    torch.cuda.synchronize()
    assert moe.device_status(ws) == 0


# one-launch decode arm at larger shapes than the small cases: E = 1024 with k = 16 and no
# shared expert, a skewed batch where experts are shared by several tokens, I = 1024, H = 4096.
# Weights drawn on the GPU; the oracle quantizes the groups the batch uses.
ONE_LAUNCH = [
    (2, 2048, 1024, 16, 512, 0, "none", 118),
    (8, 2048, 64, 8, 512, 1, "zipf", 120),
    (2, 2048, 32, 2, 1024, 1, "normal", 115),
    (4, 4096, 64, 4, 512, 1, "zipf", 119),
    # rows of h wider than rows of x (I > H): the down units' staging of h sizes the shared area
    (7, 512, 64, 8, 1024, 1, "zipf", 121),
]


@pytest.mark.parametrize("case", ONE_LAUNCH, ids=lambda c: f"T{c[0]}_H{c[1]}_E{c[2]}_k{c[3]}_I{c[4]}_sh{c[5]}")
def test_one_launch_decode_shapes(cuda_lib, case):
    T, H, E, k, I, sh, bias, seed = case
    L = Layer(synth.Shape(T=T, H=H, E=E, k=k, I=I, has_shared=sh), seed, logit_bias=bias, gen_device="cuda")
    assert cuda_lib.forward_arm(moe_shape(cuda_lib, L.shape)) == 0
    _check_full(cuda_lib, L, list(range(T)))


@pytest.mark.parametrize("T,seed", list(zip(synth.WORKLOADS["decode"].Ts, synth.WORKLOADS["decode"].seeds)))
def test_decode_sweep_full_size(cuda_lib, T, seed):
    L = _full_case(synth.WORKLOADS["decode"], T, seed)
    _check_full(cuda_lib, L, list(range(T)))


def test_batched_decode_full_size(cuda_lib):
    """Every row of the skewed T = 64 batch."""
    w = synth.WORKLOADS["batched"]
    L = _full_case(w, 64, w.seeds[0])
    _check_full(cuda_lib, L, list(range(64)))


def test_prefill_chunk_full_size(cuda_lib):
    """Every row of the T = 4096 prefill chunk, outlier rows included."""
    w = synth.WORKLOADS["prefill"]
    L = _full_case(w, 4096, w.seeds[0])
    outliers = torch.nonzero(L.x.float().abs().amax(1) > 8).flatten().tolist()
    assert len(outliers) >= 30
    _check_full(cuda_lib, L, list(range(4096)))


TC_TILE = 128   # token rows per work item of the tensor-core arm


def _edge_tokens(L, n_total, rng_seed):
    """Tokens of the rows where a tiling error would show first, then random ones up to n_total:
    every row of the most popular expert's first and last 128-row tile, every row of the last
    routed expert's last tile and of the shared expert's last tile (the last work item), and the
    first and last token."""
    s = L.shape
    ids, _ = oracle.route(L.logits.cpu(), s.k)
    counts, offsets, sorted_slot, _ = oracle.permute(ids, s.E)
    toks = {0, s.T - 1}
    hot = int(np.argmax(counts))
    c, o = int(counts[hot]), int(offsets[hot])
    last_tile = (c - 1) // TC_TILE * TC_TILE
    rows = list(range(o, o + min(TC_TILE, c))) + list(range(o + last_tile, o + c))
    e_last = int(np.nonzero(counts)[0][-1])
    c2, o2 = int(counts[e_last]), int(offsets[e_last])
    rows += list(range(o2 + (c2 - 1) // TC_TILE * TC_TILE, o2 + c2))
    toks.update(int(sorted_slot[r]) // s.k for r in rows)
    toks.update(range(s.T - ((s.T - 1) % TC_TILE + 1), s.T))   # the shared expert's last tile
    rng = np.random.default_rng(rng_seed)
    rest = np.setdiff1d(np.arange(s.T), np.fromiter(toks, int))
    extra = max(0, n_total - len(toks))
    toks.update(rng.choice(rest, size=min(extra, rest.size), replace=False).tolist())
    return sorted(toks), counts[hot]


@pytest.mark.parametrize("layer", [0, 1, 2, 3])
def test_long_prefill_full_size(cuda_lib, layer):
    """Each of the four T = 32768 Zipf layers: at least 512 rows, including every row of the
    hottest expert's first and last tile and of the last work items."""
    w = synth.WORKLOADS["long"]
    L = _full_case(w, 32768, w.seeds[0], layer=layer)
    tokens, hot_count = _edge_tokens(L, 512, 1000 + layer)
    assert len(tokens) >= 512 and hot_count > 10 * TC_TILE
    _check_full(cuda_lib, L, tokens)


def test_zipf_prefill_8192_every_row(cuda_lib):
    """One Zipf-routed layer of the long-prefill shape at T = 8192, every row checked."""
    w = synth.WORKLOADS["long"]
    L = Layer(w.shape(8192), 7_900, layer=0, logit_bias="zipf", gen_device="cuda")
    _check_full(cuda_lib, L, list(range(8192)))


# batches of 9..64 tokens on the tensor-core arm: routing, permutation, work list and the
# expert-ordered f16 rows of x come from one launch whose CTAs each rank the whole batch;
# E = 1024 with k = 16 fills its shared-memory slot table (64 x 16)
SMALL_BATCH = [
    (9, 512, 16, 2, 256, 1, "normal", 141),
    (33, 512, 1024, 16, 256, 0, "zipf", 142),
    (64, 512, 1024, 16, 256, 1, "normal", 143),
    (64, 256, 8, 8, 256, 1, "none", 144),
]


@pytest.mark.parametrize("case", SMALL_BATCH, ids=lambda c: f"T{c[0]}_H{c[1]}_E{c[2]}_k{c[3]}_I{c[4]}_sh{c[5]}")
def test_small_batch_tensor_core_forward(cuda_lib, case):
    T, H, E, k, I, sh, bias, seed = case
    L = Layer(synth.Shape(T=T, H=H, E=E, k=k, I=I, has_shared=sh), seed, logit_bias=bias, gen_device="cuda")
    assert cuda_lib.forward_arm(moe_shape(cuda_lib, L.shape)) == 2
    _check_full(cuda_lib, L, list(range(T)))
