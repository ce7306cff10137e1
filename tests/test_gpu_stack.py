"""GPU parity through a stack of distinct layers: the stacked-layer workload's
recipe (distinct seeded layers of the gpt-oss shape, an RMS renormalisation
between layers), decoded one token through three of its layers.

The renormalisation is a step of this test, not of the library. At every
layer the oracle takes the GPU's own input, so the check is per layer
(routing and the 1e-4 decode tolerance) and errors cannot compound.
"""

import gc

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from synthetic import make_layer, make_tokens, spec_for
from tests.gpu_helpers import DECODE_TOL, dev, empty, status

pytestmark = pytest.mark.gpu


def rms_renorm(y: np.ndarray) -> np.ndarray:
    y64 = y.astype(np.float64)
    return (y64 / np.sqrt(np.mean(y64 ** 2, axis=-1, keepdims=True))).astype(np.float32)


def test_stack_three_distinct_layers_decode(moe):
    spec = spec_for(3)
    k = spec.k
    x = make_tokens(spec, T=1, seed=77)
    seen = set()
    for li in range(3):
        L = make_layer(spec, li, with_tokens=False)
        layer = moe.MoeLayer(L, k=k)
        ids = empty((1, k), torch.int32)
        w = empty((1, k), torch.float32)
        y = layer(dev(x), rail=moe.MOE_RAIL_GEMV, ids_out=ids, weights_out=w)
        torch.cuda.synchronize()
        assert status(moe) == 0
        y, ids = y.cpu().numpy(), ids.cpu().numpy()
        logits = O.router_logits(x, L["w_router"], L["b_router"])
        ids_ref, _ = O.topk_softmax(logits, k)
        if O.routing_margins(logits, k)[0] > 1e-4 * np.abs(logits).max():
            assert np.array_equal(ids, ids_ref)
        sel = np.take_along_axis(logits, ids.astype(np.int64), 1)
        w_ref = np.exp(sel - sel[:, :1])
        w_ref /= w_ref.sum(1, keepdims=True)
        y64, _, _, _ = O.moe_layer(L, x, k, ids=ids, weights=w_ref)
        err = O.rownorm_rel_err(y, y64).max()
        assert err <= DECODE_TOL, (li, err)
        seen.add(tuple(ids[0].tolist()))
        x = rms_renorm(y)
        del layer, L
        gc.collect()
        torch.cuda.empty_cache()
    assert len(seen) >= 2  # distinct layers route the token differently


def test_stack_two_distinct_layers_prefill_T512(moe):
    """The stacked workload at T=512: two distinct full-size layers, the library's
    renormalisation between them on the GPU, each layer checked on the tokens at
    its bucket-tile edges against the oracle fed that layer's GPU input."""
    from tests.gpu_helpers import PREFILL_TOL
    from tests.test_gpu_layer import tile_boundary_tokens

    spec = spec_for(3)
    k, T, D = spec.k, 512, spec.D
    x = make_tokens(spec, T=T, seed=78)
    xd = dev(x)
    for li in range(2):
        L = make_layer(spec, li, with_tokens=False)
        layer = moe.MoeLayer(L, k=k)
        ids = empty((T, k), torch.int32)
        w = empty((T, k), torch.float32)
        y = layer(xd, rail=moe.MOE_RAIL_GROUPED_MM, ids_out=ids, weights_out=w)
        torch.cuda.synchronize()
        assert status(moe) == 0
        ids_np, x_in = ids.cpu().numpy(), xd.cpu().numpy()
        toks = tile_boundary_tokens(ids_np, spec.E, k)
        logits = O.router_logits(x_in, L["w_router"], L["b_router"])
        sel = np.take_along_axis(logits, ids_np.astype(np.int64), 1)
        w_ref = np.exp(sel - sel[:, :1])
        w_ref /= w_ref.sum(1, keepdims=True)
        y64, _, _, _ = O.moe_layer(L, x_in, k, token_idx=toks, ids=ids_np, weights=w_ref)
        err = O.rownorm_rel_err(y.cpu().numpy()[toks], y64).max()
        assert err <= PREFILL_TOL, (li, err)
        nxt = empty((T, D), torch.float32)
        assert moe.moe_rms_renorm(y, T, D, nxt) == 0
        torch.cuda.synchronize()
        assert np.abs(nxt.cpu().numpy().astype(np.float64) - O.rms_renorm(y.cpu().numpy())).max() <= 1e-5
        xd = nxt
        del layer, L
        gc.collect()
        torch.cuda.empty_cache()
