"""GPU parity of the prefill rail on prepacked weights (MOE_RAIL_GROUPED_MX4:
tcgen05.mma kind::mxf4 with x as six E2M1 terms and h as four) against the float64
layer and against the oracle evaluated on the same E2M1-term operands."""

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from synthetic import make_layer, make_tokens, spec_for
from tests.gpu_helpers import PREFILL_MX_TOL, PREFILL_TOL, dev, empty, status
from tests.test_gpu_layer import tile_boundary_tokens

pytestmark = pytest.mark.gpu

_LAYERS = {}


def packed_layer(moe, key):
    if key not in _LAYERS:
        spec = spec_for(1, D=192, F=320, E=6, k=3, name="rect") if key == "rect" else spec_for(key)
        L = make_layer(spec, with_tokens=False)
        _LAYERS[key] = (spec, L, moe.MoeLayer(L, k=spec.k, packed=True), O.ExpertCache(L))
    return _LAYERS[key]


def check_mx4(moe, key, T, seed, sample=None):
    spec, L, layer, cache = packed_layer(moe, key)
    k = spec.k
    x = make_tokens(spec, T=T, seed=seed)
    ids = empty((T, k), torch.int32)
    w = empty((T, k), torch.float32)
    y = layer(dev(x), rail=moe.MOE_RAIL_GROUPED_MX4, ids_out=ids, weights_out=w)
    torch.cuda.synchronize()
    assert status(moe) == 0
    y, ids = y.cpu().numpy(), ids.cpu().numpy()
    logits = O.router_logits(x, L["w_router"], L["b_router"])
    clear = O.routing_margins(logits, k) > 1e-4 * np.abs(logits).max()
    ids_ref, _ = O.topk_softmax(logits, k)
    assert np.array_equal(ids[clear], ids_ref[clear])
    toks = np.arange(T) if sample is None else tile_boundary_tokens(ids, spec.E, k)
    sel = np.take_along_axis(logits, ids.astype(np.int64), 1)
    w_ref = np.exp(sel - sel[:, :1])
    w_ref /= w_ref.sum(1, keepdims=True)
    y64, _, _, _ = O.moe_layer(L, x, k, token_idx=toks, ids=ids, weights=w_ref, cache=cache)
    ym, _, _, _ = O.moe_layer(L, x, k, token_idx=toks, ids=ids, weights=w_ref, cache=cache, operands="e2m1_terms")
    err64 = O.rownorm_rel_err(y[toks], y64).max()
    errm = O.rownorm_rel_err(y[toks], ym).max()
    print(f"mx4 rail {key} T={T} ({len(toks)} tokens checked): vs float64 {err64:.2e}, vs E2M1-term operands "
          f"{errm:.2e}")
    assert err64 <= PREFILL_TOL
    assert errm <= PREFILL_MX_TOL


@pytest.mark.parametrize("key,T,seed", [(0, 8, 1), (0, 37, 2), (0, 1, 3), ("rect", 50, 4), ("rect", 300, 5),
                                        (1, 16, 6), (1, 64, 7)])
def test_mx4_rail_parity(moe, key, T, seed):
    check_mx4(moe, key, T, seed)


def test_mx4_rail_prefill_T512_tile_edges(moe):
    check_mx4(moe, 2, 512, 8, sample="tiles")


def test_mx4_rail_skew_T4096_tile_edges(moe):
    check_mx4(moe, 4, 4096, 9, sample="tiles")


def test_mx4_rail_is_the_packed_automatic_choice_beyond_decode_sizes(moe):
    spec, L, layer, _ = packed_layer(moe, 0)
    assert moe.moe_ffn_packed_workspace_bytes(9, spec.D, spec.F, spec.E, spec.k, moe.MOE_RAIL_AUTO) == \
        moe.moe_ffn_packed_workspace_bytes(9, spec.D, spec.F, spec.E, spec.k, moe.MOE_RAIL_GROUPED_MX4) > 0
    x = dev(make_tokens(spec, T=20, seed=10))
    ya = torch.empty((20, spec.D), device="cuda")
    ws = layer.workspace(20, moe.MOE_RAIL_GROUPED_MX4)
    assert moe.moe_ffn_layer_packed(layer.packed_struct, x, 20, moe.MOE_RAIL_AUTO, ws, ws.numel(), ya) == 0
    yb = layer(x, rail=moe.MOE_RAIL_GROUPED_MX4)
    torch.cuda.synchronize()
    assert O.rownorm_rel_err(ya.cpu().numpy(), yb.cpu().numpy().astype(np.float64)).max() <= 1e-5
