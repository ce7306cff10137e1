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


def _ru(v, a):
    return (v + a - 1) // a * a


def _read_x_terms(moe, layer, spec, T):
    """x as the prefill rail's quantiser left it in the layer workspace: for every
    live bucket row, the sum of its six E2M1 terms, decoded from the activation
    chunks (term-major 8192-byte images of 128 rows, 64-byte swizzle) and the
    scale atoms of the row's segment."""
    E, k, D = spec.E, spec.k, spec.D
    ws = layer.workspace(T, moe.MOE_RAIL_GROUPED_MX4).cpu().numpy()
    mr = _ru(T * k + E * 127, 128)
    ntiles, NK, NT = mr // 128, (D + 127) // 128, 6
    off, parts = 0, {}
    for name, nbytes in (("logits", T * E * 4), ("ids", T * k * 4), ("w", T * k * 4), ("counts", E * 4),
                         ("basep", (E + 1) * 4), ("rows", mr * 4), ("inv", T * k * 4),
                         ("aq", ntiles * NK * NT * 8192), ("asf", ntiles * NK * 2 * NT * 512)):
        parts[name] = ws[off:off + nbytes]
        off = _ru(off + nbytes, 256)
    counts, basep = parts["counts"].view(np.int32), parts["basep"].view(np.int32)
    rows = parts["rows"].view(np.int32)
    aq = parts["aq"].reshape(ntiles, NK, NT, 128, 64)
    asf = parts["asf"].reshape(ntiles, NK, 2, NT, 512)
    got = {}
    for b in range(int(basep[E]) // 128):
        e = int(np.searchsorted(basep, 128 * b, side="right")) - 1
        live = min(128, int(counts[e]) - (128 * b - int(basep[e])))
        for rt in range(live):
            p = 128 * b + rt
            s = (rt >> 6) if live > 96 else 0
            nrows = (64 if s == 0 else live - 64) if live > 96 else live
            rn = _ru(nrows, 16)
            r = rt - 64 * s
            m = max([d for d in range(1, NT + 1) if NT % d == 0 and d * rn <= 192])
            apg = (m * rn + 127) // 128
            blk = np.arange(D // 32)
            j, kb = blk // 4, blk % 4
            col = (16 * (kb ^ ((rt >> 1) & 3)))[:, None] + np.arange(16)[None, :]
            row = np.zeros((D // 32, 32))
            for t in range(NT):
                byts = aq[b, j[:, None], t, rt, col].astype(np.int64)  # [block][16]
                codes = np.concatenate([byts & 15, byts >> 4], axis=1)  # columns 0..15, then 16..31
                nn = (t % m) * rn + r
                ai, n = (t // m) * apg + (nn >> 7), nn & 127
                sc = asf[b, j, s, ai, 16 * (n & 31) + 4 * (n >> 5) + kb].astype(np.int64)
                row += O.E2M1_LUT[codes] * np.exp2(sc - 127.0)[:, None]
            row = row.reshape(D)
            got[p] = (int(rows[p]), row)
    return got


@pytest.mark.parametrize("key,T,seed", [(0, 37, 21), ("rect", 300, 22), (2, 96, 23)])
def test_mx4_x_terms_are_exact(moe, key, T, seed):
    """The quantiser's x operand (six E2M1 terms per value, bucket order, the
    segment-stacked atoms) equals the oracle's split_e2m1_terms(x, 6) bit for bit
    on every live bucket row; single-segment and two-segment tiles both occur."""
    spec, L, layer, _ = packed_layer(moe, key)
    x = make_tokens(spec, T=T, seed=seed)
    layer(dev(x), rail=moe.MOE_RAIL_GROUPED_MX4)
    torch.cuda.synchronize()
    assert status(moe) == 0
    got = _read_x_terms(moe, layer, spec, T)
    ref = O.split_e2m1_terms(x, 6)
    assert len(got) == T * spec.k
    for p, (a, row) in got.items():
        assert a >= 0, p
        assert np.array_equal(row, ref[a // spec.k]), (p, a)
