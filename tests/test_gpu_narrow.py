"""The per-expert register arm inside the tcgen05 grouped GEMMs (moe_set_narrow_rows): work items
whose expert group has at most `rows` token rows run on mma.sync in the same launch as the
tensor-core items.  Parity against the oracle exactly as for the tensor-core items (same layer
tolerance), with batches that mix both kinds of item (skewed routing: many one- and two-token
experts next to wide ones), and the tail tiles of wide experts.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from moe_cases import Layer, check_layer_close, moe_shape, to_np
import test_gpu_parity as parity
from test_gpu_parity import SMALL, _check_full, _full_case

pytestmark = pytest.mark.gpu


@pytest.fixture
def narrow(cuda_lib):
    """Sets the register arm's row bound for one test and restores the library default after."""
    def set_rows(rows):
        cuda_lib.set_narrow_rows(rows)
    yield set_rows
    cuda_lib.set_narrow_rows(-1)


def _tile_rows(counts, tile):
    """Row counts of the work items the tensor-core arm builds from per-expert counts."""
    rows = []
    for c in counts:
        c = int(c)
        while c > 0:
            rows.append(min(c, tile))
            c -= tile
    return rows


TC_SMALL = [c for c in SMALL if c[0] > 8 and c[1] % 256 == 0 and c[4] % 256 == 0]


@pytest.mark.parametrize("rows", [8, 3])
@pytest.mark.parametrize("case", TC_SMALL, ids=lambda c: f"T{c[0]}_H{c[1]}_E{c[2]}_k{c[3]}_I{c[4]}_sh{c[5]}")
def test_register_arm_small_layers(cuda_lib, narrow, case, rows):
    """Every stage (h and y of both projections, combine, forward) against the oracle with the
    register arm taking the items of at most `rows` rows."""
    narrow(rows)
    T, H, E, k, I, sh, bias, seed = case
    ms = moe_shape(cuda_lib, synth.Shape(T=T, H=H, E=E, k=k, I=I, has_shared=sh))
    assert cuda_lib.forward_arm(ms) == 2
    parity.test_small_layers_all_stages(cuda_lib, case)


def test_register_arm_batched_full_size(cuda_lib, narrow):
    """Every row of the skewed T = 64 batch with the register arm on: about two thirds of its
    ~100 experts have at most 8 tokens, the rest up to ~50."""
    narrow(8)
    w = synth.WORKLOADS["batched"]
    L = _full_case(w, 64, w.seeds[0])
    ids, _ = oracle.route(L.logits.cpu(), L.shape.k)
    rows = _tile_rows(np.bincount(ids.ravel(), minlength=L.shape.E), 64)
    assert sum(r <= 8 for r in rows) > 20 and sum(r > 8 for r in rows) > 5
    _check_full(cuda_lib, L, list(range(64)))


@pytest.mark.parametrize("T,seed", [(24, 131), (200, 132), (512, 133)])
def test_register_arm_matches_tensor_core_arm(cuda_lib, narrow, T, seed):
    """The same layer with the register arm off and on: both within the layer tolerance of the
    oracle on sampled rows, and within twice that of each other everywhere (only the MMA's
    accumulation order differs)."""
    shape = synth.Shape(T=T, H=2048, E=512, k=10, I=512, has_shared=1)
    L = Layer(shape, seed, logit_bias="normal", gen_device="cuda")
    ms = moe_shape(cuda_lib, shape)
    assert cuda_lib.forward_arm(ms) == 2
    gu, dn = L.gpu_weights(cuda_lib)
    ws = cuda_lib.workspace(ms)
    outs = []
    for rows in (0, 8):
        narrow(rows)
        out = torch.full((T, shape.H), float("nan"), device="cuda", dtype=torch.float32)
        cuda_lib.forward(L.x, L.logits, gu, dn, ms, ws, out=out, out_fp32=True)
        torch.cuda.synchronize()
        assert cuda_lib.device_status(ws) == 0
        outs.append(to_np(out))
    check_layer_close(outs[1], outs[0], "register arm vs tensor-core arm", row_rms_tol=4e-2)
    tokens = sorted(set(np.random.default_rng(seed).choice(T, size=min(T, 6), replace=False).tolist()) | {T - 1})
    groups = L.used_groups(tokens)
    ogu, odn = L.oracle_weights(groups)
    ref = oracle.moe_forward(L.x.cpu(), L.logits.cpu(), ogu, odn, shape.k, shape.has_shared, tokens=tokens)
    for o in outs:
        check_layer_close(o[tokens], ref, "sampled rows")



@pytest.mark.parametrize("T,seed", [(200, 132), (48, 7), (512, 133)])
def test_register_arm_is_deterministic(cuda_lib, narrow, T, seed):
    """Repeated stage calls give identical bytes with the register arm on (128-row tiles have two
    activation stages, 64-row tiles four: both rings' phase tracking is exercised)."""
    narrow(8)
    shape = synth.Shape(T=T, H=2048, E=512, k=10, I=512, has_shared=1)
    L = Layer(shape, seed, logit_bias="normal", gen_device="cuda")
    ms = moe_shape(cuda_lib, shape)
    gu, dn = L.gpu_weights(cuda_lib)
    ws = cuda_lib.workspace(ms)
    ids, _ = cuda_lib.route_topk(L.logits, ms)
    counts, offsets, sorted_slot, _ = cuda_lib.permute(ids, ms, ws)
    tile = 64 if T <= cuda_lib.DECODE_MAX_T else 128
    assert sum(r <= 8 for r in _tile_rows(counts.cpu().numpy(), tile)) > 0
    h0 = cuda_lib.grouped_gate_up(L.x, sorted_slot, offsets, gu, ms, ws).clone()
    y0 = cuda_lib.grouped_down(h0, offsets, dn, ms, ws).clone()
    for _ in range(6):
        h = cuda_lib.grouped_gate_up(L.x, sorted_slot, offsets, gu, ms, ws)
        assert torch.equal(h.view(torch.int16), h0.view(torch.int16))
        y = cuda_lib.grouped_down(h0, offsets, dn, ms, ws)
        assert torch.equal(y.view(torch.int32), y0.view(torch.int32))
    torch.cuda.synchronize()
    assert cuda_lib.device_status(ws) == 0
