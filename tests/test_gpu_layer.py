"""GPU parity of the whole layer (moe_ffn_layer, both rails) against the oracle.

The full gpt-oss-shaped workloads run at their real sizes in the same launch
configuration the benchmark times; the oracle then evaluates a sample of the
tokens (it computes one token at a time, dequantising only the experts used).
"""

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from synthetic import make_layer, make_tokens, spec_for
from tests.gpu_helpers import (DECODE_TOL, PREFILL_BF16_TOL, PREFILL_MX_TOL, PREFILL_TOL, dev, empty,
                               status)

pytestmark = pytest.mark.gpu

_CACHE = {}


def layer_for(moe, cfg):
    if cfg not in _CACHE:
        spec = spec_for(cfg)
        L = make_layer(spec, with_tokens=False)
        _CACHE[cfg] = (spec, L, moe.MoeLayer(L, k=spec.k), O.ExpertCache(L))
    return _CACHE[cfg]


def run_layer(moe, layer, x_np, rail, k):
    T = x_np.shape[0]
    ids = empty((T, k), torch.int32)
    w = empty((T, k), torch.float32)
    y = layer(dev(x_np), rail=rail, ids_out=ids, weights_out=w)
    torch.cuda.synchronize()
    assert status(moe) == 0
    return y.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy()


def tile_boundary_tokens(ids, E, k, tile=128):
    """Tokens whose assignments sit at the edges of the grouped GEMM's work: each
    expert's first and last live bucket row, and the first and last live row of
    every 128-row bucket tile (the oracle's CSR of the GPU's own routing)."""
    csr = O.bucket_csr(ids, E, tile)
    rows, basep, counts = csr["rows"], csr["basep"], csr["counts"]
    picks = set()
    for e in range(E):
        n = int(counts[e])
        for lo in range(0, n, tile):
            hi = min(n, lo + tile) - 1
            picks.add(int(rows[basep[e] + lo]) // k)
            picks.add(int(rows[basep[e] + hi]) // k)
    return np.array(sorted(picks), dtype=np.int64)


def check_layer(moe, cfg, T, rail, sample=None, seed=None):
    spec, L, layer, cache = layer_for(moe, cfg)
    if rail == moe.MOE_RAIL_AUTO:  # the canonical planes' automatic choice by T
        rail = (moe.MOE_RAIL_GEMV if T <= moe.MOE_AUTO_GEMV_MAX_T else
                moe.MOE_RAIL_GROUPED_MX if T <= moe.MOE_AUTO_MX_MAX_T else moe.MOE_RAIL_GROUPED_MM)
    x = make_tokens(spec, T=T, seed=seed)
    y, ids, w = run_layer(moe, layer, x, rail, spec.k)
    logits = O.router_logits(x, L["w_router"], L["b_router"])
    ids_ref, _ = O.topk_softmax(logits, spec.k)
    margin = O.routing_margins(logits, spec.k)
    clear = margin > 1e-4 * np.abs(logits).max()
    assert np.array_equal(ids[clear], ids_ref[clear])
    if isinstance(sample, str) and sample == "tiles":
        sample = tile_boundary_tokens(ids, spec.E, spec.k)
        print(f"cfg {cfg} T {T}: {len(sample)} tokens sampled at bucket-tile edges")
    toks = np.arange(T) if sample is None else sample
    # evaluate the oracle on the GPU's routing for the sampled tokens (identical where clear)
    w_ref = np.take_along_axis(logits, ids.astype(np.int64), 1)
    w_ref = np.exp(w_ref - w_ref[:, :1])
    w_ref /= w_ref.sum(1, keepdims=True)
    y64, _, _, _ = O.moe_layer(L, x, spec.k, token_idx=toks, ids=ids, weights=w_ref, cache=cache)
    if rail == moe.MOE_RAIL_GEMV:
        err = O.rownorm_rel_err(y[toks], y64)
        assert err.max() <= DECODE_TOL, err.max()
    elif rail == moe.MOE_RAIL_GROUPED_MX:
        err64 = O.rownorm_rel_err(y[toks], y64)
        ye4, _, _, _ = O.moe_layer(L, x, spec.k, token_idx=toks, ids=ids, weights=w_ref, cache=cache,
                                   operands="e4m3_terms")
        err_e4 = O.rownorm_rel_err(y[toks], ye4)
        print(f"mx rail cfg {cfg} T {T}: rownorm err vs float64 {err64.max():.3e}, "
              f"vs the same E4M3-term operands {err_e4.max():.3e}")
        assert err64.max() <= PREFILL_TOL, err64.max()
        assert err_e4.max() <= PREFILL_MX_TOL, err_e4.max()
    else:
        ybf, _, _, _ = O.moe_layer(L, x, spec.k, token_idx=toks, ids=ids, weights=w_ref, cache=cache,
                                   operands="bf16_split")
        err_bf = O.rownorm_rel_err(y[toks], ybf)
        err64 = O.rownorm_rel_err(y[toks], y64)
        assert err_bf.max() <= PREFILL_BF16_TOL, err_bf.max()
        assert err64.max() <= PREFILL_TOL, err64.max()
    return y, ids


@pytest.mark.parametrize("rail_name", ["GEMV", "GROUPED_MM", "GROUPED_MX"])
def test_tiny_layer_both_rails(moe, rail_name):
    check_layer(moe, 0, 8, getattr(moe, "MOE_RAIL_" + rail_name))


@pytest.mark.parametrize("T", [1, 2, 3, 5, 8])
def test_tiny_layer_gemv_token_counts(moe, T):
    check_layer(moe, 0, T, moe.MOE_RAIL_GEMV, seed=40 + T)


@pytest.mark.parametrize("rail_name", ["GROUPED_MM", "GROUPED_MX"])
@pytest.mark.parametrize("T", [1, 9, 40, 131])
def test_tiny_layer_grouped_token_counts(moe, T, rail_name):
    check_layer(moe, 0, T, getattr(moe, "MOE_RAIL_" + rail_name), seed=50 + T)


def test_decode_T1_full_size(moe):
    # the decode workload the benchmark times (E=32, k=4, D=F=2880, T=1)
    for seed in (1, 2, 3):
        check_layer(moe, 1, 1, moe.MOE_RAIL_AUTO, seed=seed)


def test_decode_T8_full_size(moe):
    check_layer(moe, 1, 8, moe.MOE_RAIL_GEMV, seed=9)


def test_prefill_T512_full_size_sampled(moe):
    # the prefill workload (T=512): the first and last token, and every token at
    # an edge of a bucket tile (each expert's first and last live row, each
    # 128-row tile's first and last), through the oracle
    y, ids = check_layer(moe, 2, 512, moe.MOE_RAIL_GROUPED_MM, sample="tiles")


def test_prefill_T512_full_size_sampled_mx(moe):
    check_layer(moe, 2, 512, moe.MOE_RAIL_GROUPED_MX, sample="tiles")


def test_prefill_T512_auto_rail(moe):
    check_layer(moe, 2, 512, moe.MOE_RAIL_AUTO, sample=np.array([0, 1, 255, 511]))


@pytest.mark.parametrize("rail_name", ["GROUPED_MM", "GROUPED_MX"])
def test_skew_T4096_full_size_sampled(moe, rail_name):
    spec, L, layer, cache = layer_for(moe, 4)
    y, ids = check_layer(moe, 4, 4096, getattr(moe, "MOE_RAIL_" + rail_name), sample="tiles")
    counts = np.bincount(ids.reshape(-1), minlength=spec.E)
    # the stated shape of the skewed workload: about half of the assignments on the
    # two hot experts, several experts nearly empty
    assert 0.45 <= (counts[0] + counts[1]) / ids.size <= 0.55
    assert (counts <= 3).sum() >= 3


def test_rails_agree_on_routing_and_values(moe):
    spec, L, layer, _ = layer_for(moe, 1)
    x = make_tokens(spec, T=8, seed=77)
    yg, idg, wg = run_layer(moe, layer, x, moe.MOE_RAIL_GEMV, spec.k)
    ym, idm, wm = run_layer(moe, layer, x, moe.MOE_RAIL_GROUPED_MM, spec.k)
    assert np.array_equal(idg, idm) and np.array_equal(wg, wm)
    assert O.rownorm_rel_err(ym, yg).max() <= PREFILL_TOL


def test_gemv_rail_is_deterministic(moe):
    spec, L, layer, _ = layer_for(moe, 1)
    x = dev(make_tokens(spec, T=1, seed=5))
    ys = [layer(x, rail=moe.MOE_RAIL_GEMV).clone() for _ in range(5)]
    for y in ys[1:]:
        assert torch.equal(y, ys[0])


def test_fused_chain_matches_unfused_entry_points(moe):
    """Fused GEMV rail vs the per-op composition of the exported entry points
    (route, gate GEMV, up GEMV, swiglu, down GEMV), combined in slot order."""
    spec, L, layer, _ = layer_for(moe, 1)
    T, k, D, F, E = 2, spec.k, spec.D, spec.F, spec.E
    x_np = make_tokens(spec, T=T, seed=31)
    y_fused, ids_f, w_f = run_layer(moe, layer, x_np, moe.MOE_RAIL_GEMV, k)
    W = layer.w
    x = dev(x_np)
    logits, ids, w = empty((T, E), torch.float32), empty((T, k), torch.int32), empty((T, k), torch.float32)
    assert moe.moe_route_topk(x, T, D, W["w_router"], W["b_router"], E, k, logits, ids, w) == 0
    flat = ids.reshape(-1).contiguous()
    xr = x.repeat_interleave(k, dim=0).contiguous()
    g, u = empty((T * k, F), torch.float32), empty((T * k, F), torch.float32)
    assert moe.moe_mxfp4_gemv(W["g_qs"], W["g_sc"], E, F, D, flat, T * k, xr, D, W["bg"], g) == 0
    assert moe.moe_mxfp4_gemv(W["u_qs"], W["u_sc"], E, F, D, flat, T * k, xr, D, W["bu"], u) == 0
    h = empty((T * k, F), torch.float32)
    assert moe.moe_swiglu_oai(g, u, h, T * k * F, moe.MOE_DTYPE_F32) == 0
    o = empty((T * k, D), torch.float32)
    assert moe.moe_mxfp4_gemv(W["d_qs"], W["d_sc"], E, D, F, flat, T * k, h, F, W["bd"], o) == 0
    torch.cuda.synchronize()
    o = o.cpu().numpy().reshape(T, k, D)
    wn = w.cpu().numpy()
    y_unf = np.zeros((T, D), np.float32)
    for j in range(k):  # slot order
        y_unf += wn[:, j:j + 1] * o[:, j]
    assert np.array_equal(ids.cpu().numpy(), ids_f) and np.array_equal(wn, w_f)
    assert O.rownorm_rel_err(y_fused, y_unf).max() <= 1e-5


def test_routing_ids_stable_across_runs(moe):
    spec, L, layer, _ = layer_for(moe, 2)
    x = dev(make_tokens(spec, T=512, seed=3))
    first = None
    for _ in range(10):
        ids = empty((512, spec.k), torch.int32)
        layer(x, ids_out=ids)
        if first is None:
            first = ids.clone()
        assert torch.equal(ids, first)


def test_layer_T0_is_noop(moe):
    spec, L, layer, _ = layer_for(moe, 0)
    y = torch.full((1, spec.D), 3.0, device="cuda")
    rc = moe.moe_ffn_layer(None, 0, spec.D, spec.F, spec.E, spec.k, None, None, None, None, None, None,
                           None, None, None, None, None, 0, None, 0, y)
    assert rc == 0
    assert torch.all(y == 3.0)


def test_layer_without_biases(moe):
    spec = spec_for(0)
    L = dict(make_layer(spec, layer=5))
    for key in ("b_router", "bg", "bu", "bd"):
        L[key] = None
    layer = moe.MoeLayer(L, k=spec.k)
    x = make_tokens(spec, T=8, seed=8)
    L0 = dict(L, b_router=np.zeros(spec.E, np.float32), bg=np.zeros((spec.E, spec.F), np.float32),
              bu=np.zeros((spec.E, spec.F), np.float32), bd=np.zeros((spec.E, spec.D), np.float32))
    y64, ids64, _, _ = O.moe_layer(L0, x, spec.k)
    ybf, _, _, _ = O.moe_layer(L0, x, spec.k, operands="bf16_split")
    for rail, ref, tol in ((moe.MOE_RAIL_GEMV, y64, DECODE_TOL), (moe.MOE_RAIL_GROUPED_MM, ybf, PREFILL_BF16_TOL),
                           (moe.MOE_RAIL_GROUPED_MX, y64, PREFILL_TOL)):
        y, ids, _ = run_layer(moe, layer, x, rail, spec.k)
        assert np.array_equal(ids, ids64)
        assert O.rownorm_rel_err(y, ref).max() <= tol


@pytest.mark.parametrize("T", [1, 3, 8])
def test_decode_stage_entry_points_match_the_layer(moe, T):
    """moe_route_topk -> moe_expert_gateup_swiglu -> moe_expert_down_combine (ids given)
    equals the layer's GEMV rail (top-k taken inside the expert kernels), and the oracle."""
    spec, L, layer, cache = layer_for(moe, 1)
    E, k, D, F = spec.E, spec.k, spec.D, spec.F
    x_np = make_tokens(spec, T=T, seed=60 + T)
    y_layer, ids_l, w_l = run_layer(moe, layer, x_np, moe.MOE_RAIL_GEMV, k)
    W = layer.w
    x = dev(x_np)
    logits, ids, w = empty((T, E), torch.float32), empty((T, k), torch.int32), empty((T, k), torch.float32)
    assert moe.moe_route_topk(x, T, D, W["w_router"], W["b_router"], E, k, logits, ids, w) == 0
    h = empty((T * k, F), torch.float32)
    assert moe.moe_expert_gateup_swiglu(W["g_qs"], W["g_sc"], W["bg"], W["u_qs"], W["u_sc"], W["bu"], E, F, D,
                                        T, k, x, ids, 1.702, 7.0, h) == 0
    y = empty((T, D), torch.float32)
    assert moe.moe_expert_down_combine(W["d_qs"], W["d_sc"], W["bd"], E, D, F, T, k, h, ids, w, y) == 0
    torch.cuda.synchronize()
    assert status(moe) == 0
    assert np.array_equal(ids.cpu().numpy(), ids_l) and np.array_equal(w.cpu().numpy(), w_l)
    assert torch.equal(y.cpu(), torch.from_numpy(y_layer))
    y64, _, _, _ = O.moe_layer(L, x_np, k, ids=ids_l, weights=w_l.astype(np.float64), cache=cache)
    assert O.rownorm_rel_err(y_layer, y64).max() <= DECODE_TOL


@pytest.mark.parametrize("cfg,T,rail", [(1, 1, "GEMV"), (1, 3, "GEMV"), (0, 8, "GEMV"), (0, 8, "GROUPED_MM"),
                                        (0, 8, "GROUPED_MX")])
def test_forward_host_matches_forward(moe, cfg, T, rail):
    """moe_ffn_layer_hostio (host x in, host y out, one call) gives the same bits as
    moe_ffn_layer on device buffers, for two calls in a row on one stream."""
    spec, L, layer, _ = layer_for(moe, cfg)
    r = getattr(moe, f"MOE_RAIL_{rail}")
    for rep in range(2):
        x_np = make_tokens(spec, T=T, seed=300 + 10 * cfg + T + rep)
        y_dev = layer(dev(x_np), rail=r)
        x_host = torch.from_numpy(x_np).pin_memory()
        y_host = layer.forward_host(x_host, rail=r)
        torch.cuda.synchronize()
        assert status(moe) == 0
        assert torch.equal(y_host, y_dev.cpu())


def test_forward_host_pinned_and_pageable(moe):
    """Host-I/O decode with pinned buffers (the kernels read x and write y in host
    memory, no copies) and with pageable ones (copied through the staging
    buffers): every result equals the device-buffer call bit for bit."""
    spec, L, layer, _ = layer_for(moe, 1)
    rail = moe.MOE_RAIL_GEMV
    xs = [torch.from_numpy(make_tokens(spec, T=1, seed=400 + i)).pin_memory() for i in range(3)]
    ys = [torch.full((1, spec.D), float("nan")).pin_memory() for _ in range(3)]
    for x, y in zip(xs, ys):
        layer.forward_host(x, y, rail=rail)
    xp = torch.from_numpy(make_tokens(spec, T=1, seed=403))
    yp = torch.full((1, spec.D), float("nan"))
    layer.forward_host(xp, yp, rail=rail)
    torch.cuda.synchronize()
    assert status(moe) == 0
    for x, y in zip(xs + [xp], ys + [yp]):
        assert torch.equal(y, layer(dev(x.numpy()), rail=rail).cpu())


def test_forward_host_rejects_mismatched_buffers(moe):
    """Host buffers whose shape, dtype, layout or device do not fit the layer are
    refused before anything is enqueued (a short y would otherwise be written
    past its end)."""
    spec, L, layer, _ = layer_for(moe, 1)
    x = torch.from_numpy(make_tokens(spec, T=2, seed=410)).pin_memory()
    bad = [
        (x, torch.empty((1, spec.D)).pin_memory()),                 # y too short
        (x, torch.empty((2, spec.D + 32)).pin_memory()),            # y too wide
        (x, torch.empty((2, spec.D), dtype=torch.float64)),         # y not float32
        (x, torch.empty((spec.D, 2)).t()),                          # y not contiguous
        (x[:, :64].contiguous(), torch.empty((2, 64))),             # x of the wrong width
        (x.cuda(), torch.empty((2, spec.D))),                       # x on the device
    ]
    for xb, yb in bad:
        with pytest.raises(ValueError):
            layer.forward_host(xb, yb, rail=moe.MOE_RAIL_GEMV)
    torch.cuda.synchronize()
    assert status(moe) == 0


def _e4m3_values():
    vals = np.empty(256)
    for c in range(256):
        s = -1.0 if c & 0x80 else 1.0
        e, m = (c >> 3) & 15, c & 7
        vals[c] = np.nan if (e == 15 and m == 7) else (s * (m / 8.0) * 2.0 ** -6 if e == 0 else
                                                       s * (1 + m / 8.0) * 2.0 ** (e - 7))
    return vals


@pytest.mark.parametrize("cfg,T", [(0, 40), (2, 48)])
def test_mx_activation_terms_are_exact(moe, cfg, T):
    """The block-scaled rail's x operand, read back from the layer workspace (three
    E4M3 terms per bucket row in the MMA's per-block column order, E8M0 words per
    stage of four blocks), equals the oracle's split_e4m3_terms(x, 3) bit for bit."""
    spec, L, layer, _ = layer_for(moe, cfg)
    E, k, D = spec.E, spec.k, spec.D
    rail = moe.MOE_RAIL_GROUPED_MX
    x = make_tokens(spec, T=T, seed=500 + cfg)
    layer(dev(x), rail=rail)
    torch.cuda.synchronize()
    assert status(moe) == 0
    ws = layer.workspace(T, rail).cpu().numpy()
    ru = lambda v, a: (v + a - 1) // a * a
    mr = ru(T * k + E * 127, 128)
    nd = (D // 32 + 3) // 4
    off, parts = 0, {}
    # the grouped rails' workspace: logits, the split router's partial dots (32 slices at most), the route
    for name, nbytes in (("logits", T * E * 4), ("rpart", 32 * T * E * 4), ("ids", T * k * 4), ("w", T * k * 4),
                         ("counts", E * 4),
                         ("basep", (E + 1) * 4), ("rows", mr * 4), ("inv", T * k * 4),
                         ("xq", 3 * mr * D), ("xs", 3 * nd * mr * 4)):
        parts[name] = ws[off:off + nbytes]
        off = ru(off + nbytes, 256)
    basep = parts["basep"].view(np.int32)
    rows = parts["rows"].view(np.int32)
    xq = parts["xq"].reshape(3, mr, D)
    xs = parts["xs"].view(np.uint32).reshape(3, nd, mr)
    vals = _e4m3_values()
    pos = np.array([2 * (c % 16) + c // 16 for c in range(32)])
    ref = O.split_e4m3_terms(x, 3)
    checked = 0
    for p in range(int(basep[E])):
        a = int(rows[p])
        if a < 0:
            continue
        got = np.zeros(D)
        for t in range(3):
            for b in range(D // 32):
                code = (int(xs[t, b // 4, p]) >> (8 * (b % 4))) & 0xFF
                got[32 * b:32 * b + 32] += vals[xq[t, p, 32 * b + pos]] * 2.0 ** (code - 127)
        assert np.array_equal(got, ref[a // k]), (p, a)
        checked += 1
    assert checked == T * k


@pytest.mark.parametrize("T,rail_name", [(8, "GEMV"), (50, "GROUPED_MM"), (50, "GROUPED_MX"),
                                         (300, "GROUPED_MM"), (300, "GROUPED_MX")])
def test_rectangular_layer(moe, T, rail_name):
    """D != F and neither a multiple of 128 (D = 192, F = 320): ragged last K stages
    on both projections and ragged weight-row tiles; T = 300 fills whole 128-row
    bucket tiles."""
    spec = spec_for(0, name="rectangular", E=6, k=2, D=192, F=320, seed=4242)
    L = make_layer(spec, with_tokens=False)
    layer = moe.MoeLayer(L, k=spec.k)
    rail = getattr(moe, "MOE_RAIL_" + rail_name)
    x = make_tokens(spec, T=T, seed=77)
    y, ids, _ = run_layer(moe, layer, x, rail, spec.k)
    logits = O.router_logits(x, L["w_router"], L["b_router"])
    ids_ref, _ = O.topk_softmax(logits, spec.k)
    clear = O.routing_margins(logits, spec.k) > 1e-4 * np.abs(logits).max()
    assert np.array_equal(ids[clear], ids_ref[clear])
    w_ref = np.take_along_axis(logits, ids.astype(np.int64), 1)
    w_ref = np.exp(w_ref - w_ref[:, :1])
    w_ref /= w_ref.sum(1, keepdims=True)
    y64, _, _, _ = O.moe_layer(L, x, spec.k, ids=ids, weights=w_ref)
    err64 = O.rownorm_rel_err(y, y64).max()
    if rail == moe.MOE_RAIL_GEMV:
        assert err64 <= DECODE_TOL, err64
        return
    assert err64 <= PREFILL_TOL, err64
    operands, tol = (("bf16_split", PREFILL_BF16_TOL) if rail == moe.MOE_RAIL_GROUPED_MM
                     else ("e4m3_terms", PREFILL_MX_TOL))
    ymod, _, _, _ = O.moe_layer(L, x, spec.k, ids=ids, weights=w_ref, operands=operands)
    err = O.rownorm_rel_err(y, ymod).max()
    assert err <= tol, (operands, err)
