"""Gate and up stored interleaved (one [2F][D] plane per expert, as gpt-oss
stores them) give the layer of the separated planes: bit for bit on the
deterministic rails, within float-atomic reordering on the grouped rails, and
prepacked planes identical byte for byte."""

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from synthetic import interleave_gate_up, make_layer, make_tokens, spec_for
from tests.gpu_helpers import dev, status

pytestmark = pytest.mark.gpu

_PAIRS = {}


def pair(moe, key):
    if key not in _PAIRS:
        spec = spec_for(1, D=192, F=320, E=6, k=3, name="rect") if key == "rect" else spec_for(key)
        L = make_layer(spec, with_tokens=False)
        Li = interleave_gate_up(L)
        assert Li["gu_qs"].shape == (spec.E, 2 * spec.F, spec.D // 2)
        assert np.array_equal(Li["gu_qs"][:, 1::2], L["u_qs"]) and np.array_equal(Li["gu_b"][:, ::2], L["bg"])
        _PAIRS[key] = (spec, L, moe.MoeLayer(L, k=spec.k, packed=True), moe.MoeLayer(Li, k=spec.k, packed=True))
    return _PAIRS[key]


@pytest.mark.parametrize("key,T", [(0, 8), (1, 1), (1, 8), ("rect", 5)])
@pytest.mark.parametrize("rail_name", ["GEMV", "GEMV_Q8", "DECODE_MX"])
def test_interleaved_equals_separate_bit_for_bit(moe, key, T, rail_name):
    spec, L, sep, ilv = pair(moe, key)
    rail = getattr(moe, "MOE_RAIL_" + rail_name)
    x = dev(make_tokens(spec, T=T, seed=300 + T))
    y_sep = sep(x, rail=rail)
    y_ilv = ilv(x, rail=rail)
    torch.cuda.synchronize()
    assert status(moe) == 0
    assert torch.equal(y_sep, y_ilv)


@pytest.mark.parametrize("key,T", [(0, 37), (2, 512), ("rect", 300)])
@pytest.mark.parametrize("rail_name", ["GROUPED_MM", "GROUPED_MX"])
def test_interleaved_equals_separate_on_the_grouped_rails(moe, key, T, rail_name):
    spec, L, sep, ilv = pair(moe, key)
    rail = getattr(moe, "MOE_RAIL_" + rail_name)
    x = dev(make_tokens(spec, T=T, seed=400 + T))
    y_sep = sep(x, rail=rail).cpu().numpy()
    y_ilv = ilv(x, rail=rail).cpu().numpy()
    torch.cuda.synchronize()
    assert status(moe) == 0
    # the same products; only the order of the scatter's float atomics differs
    assert O.rownorm_rel_err(y_ilv, y_sep.astype(np.float64)).max() <= 1e-5


@pytest.mark.parametrize("key", [1, "rect"])
def test_prepack_from_the_interleaved_plane_is_identical(moe, key):
    spec, L, sep, ilv = pair(moe, key)
    for m in ("g_qs", "g_sf", "u_qs", "u_sf", "d_qs", "d_sf"):
        assert torch.equal(sep.packed[m], ilv.packed[m]), m


def test_interleaved_layer_rejects_mixed_planes(moe):
    spec, L, _, _ = pair(moe, 0)
    mixed = dict(interleave_gate_up(L), g_qs=L["g_qs"])
    with pytest.raises(ValueError):
        moe.MoeLayer(mixed, k=spec.k)
