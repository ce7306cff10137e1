"""GPU parity of the block-scaled decode rail (prepacked weights, T <= 8).

The prepack is checked byte for byte against the layout restated from the
header; the x operand the prologue writes bit for bit against the oracle's
E2M1-term split; the layer against the float64 oracle (the decode bound, 1e-4
row-normwise) and against the oracle's model of the rail's operands (x and w*h
as eight E2M1 terms), with routing ids bit-exact wherever the logits have a
clear margin.
"""

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from synthetic import make_layer, make_tokens, spec_for
from tests.gpu_helpers import DECODE_TOL, dev, empty, status

pytestmark = pytest.mark.gpu

# Against the oracle's model of the rail's operands (x and w*h as eight E2M1 terms) the remaining
# difference is fp32 accumulation in the tensor cores against float64. With short reductions
# (D, F <= 512) that is small and the model is held tightly; at the gpt-oss width (2880) the
# gate/up pre-activations reach 1e4..1e5 at these E8M0 scales, fp32 accumulation moves them by
# ~1e-2, the swiglu passes that on (gain up to 8) to an h whose row maximum is ~56, and y, which
# sums many such h, is held to the decode bound like the float64 comparison.
def model_tolerances(D):
    return (2e-5, 5e-4) if D <= 512 else (DECODE_TOL, 1e-3)  # (y, h)


def prepack_reference(qs, sc):
    """The prepacked planes of the header, restated: qs_p tile by tile as 64-byte-swizzled
    chunk images, sf_p [E][NT][NK][512] atoms."""
    E, R, half = qs.shape
    C = 2 * half
    NK, NT, nb = (C + 127) // 128, (R + 127) // 128, C // 32
    blocks = np.zeros((E, R, 4 * NK, 16), np.uint8)
    blocks[:, :, :nb] = qs.reshape(E, R, nb, 16)
    qs_p = np.zeros(E * R * NK * 64, np.uint8)
    for e in range(E):
        for t in range(NT):
            rows_t = min(128, R - 128 * t)
            m = np.arange(rows_t)
            for j in range(NK):
                base = (e * R + 128 * t) * NK * 64 + rows_t * 64 * j
                for kb in range(4):
                    dst = base + m * 64 + 16 * (kb ^ ((m >> 1) & 3))
                    qs_p[dst[:, None] + np.arange(16)] = blocks[e, 128 * t + m, 4 * j + kb]
    sf_p = np.full((E, NT, NK, 512), 127, np.uint8)
    for m in range(128):
        for kb in range(4):
            rows = np.arange(NT) * 128 + m
            ok_r = rows < R
            for j in range(NK):
                b = 4 * j + kb
                if b < nb:
                    sf_p[:, ok_r, j, 16 * (m % 32) + 4 * (m // 32) + kb] = sc[:, rows[ok_r], b]
    return qs_p, sf_p.reshape(-1)


@pytest.mark.parametrize("E,R,C", [(3, 192, 320), (2, 64, 64), (2, 2880, 2880)])
def test_prepack_matches_the_documented_layout(moe, E, R, C):
    rng = np.random.default_rng(R + C)
    qs = rng.integers(0, 256, size=(E, R, C // 2), dtype=np.uint8)
    sc = rng.integers(0, 256, size=(E, R, C // 32), dtype=np.uint8)
    nq, ns = moe.moe_mxfp4_packed_qs_bytes(E, R, C), moe.moe_mxfp4_packed_sf_bytes(E, R, C)
    qs_p = torch.full((nq,), 0xEE, dtype=torch.uint8, device="cuda")
    sf_p = torch.full((ns,), 0xEE, dtype=torch.uint8, device="cuda")
    assert moe.moe_mxfp4_prepack(dev(qs), dev(sc), E, R, C, qs_p, sf_p) == 0
    ref_q, ref_s = prepack_reference(qs, sc)
    assert nq == ref_q.size and ns == ref_s.size
    assert np.array_equal(qs_p.cpu().numpy(), ref_q)
    assert np.array_equal(sf_p.cpu().numpy(), ref_s)


def test_prepack_rejects_bad_shapes(moe):
    assert moe.moe_mxfp4_packed_qs_bytes(2, 100, 64) == 0   # R not a multiple of 64
    assert moe.moe_mxfp4_prepack(1 << 20, 1 << 20, 2, 100, 64, 1 << 20, 1 << 20, stream=0) == moe.MOE_EINVAL
    assert moe.moe_mxfp4_prepack(1 << 20, 1 << 20, 2, 64, 48, 1 << 20, 1 << 20, stream=0) == moe.MOE_EINVAL
    assert moe.moe_mxfp4_prepack(1 << 20, 1 << 20, 2, 64, 64, (1 << 20) + 16, 1 << 20, stream=0) == moe.MOE_EINVAL


_LAYERS = {}


def packed_layer(moe, key):
    if key not in _LAYERS:
        if key == "rect":
            spec = spec_for(1, D=192, F=320, E=6, k=3, name="rect")
        else:
            spec = spec_for(key)
        L = make_layer(spec, with_tokens=False)
        _LAYERS[key] = (spec, L, moe.MoeLayer(L, k=spec.k, packed=True), O.ExpertCache(L))
    return _LAYERS[key]


def run_packed(moe, layer, x, k, F):
    T = x.shape[0]
    ids = empty((T, k), torch.int32)
    w = empty((T, k), torch.float32)
    h = torch.full((T * k, F), float("nan"), device="cuda")
    y = layer(dev(x), rail=moe.MOE_RAIL_DECODE_MX, ids_out=ids, weights_out=w, h_out=h)
    torch.cuda.synchronize()
    assert status(moe) == 0
    return y.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy(), h.cpu().numpy().reshape(T, k, F)


def check_decode_mx(moe, key, T, seed):
    spec, L, layer, cache = packed_layer(moe, key)
    x = make_tokens(spec, T=T, seed=seed)
    y, ids, w, h = run_packed(moe, layer, x, spec.k, spec.F)
    logits = O.router_logits(x, L["w_router"], L["b_router"])
    y64, ids_ref, w_ref, _ = O.moe_layer(L, x, spec.k, cache=cache)
    clear = O.routing_margins(logits, spec.k) > 1e-4 * np.abs(logits).max()
    assert clear.all(), "seeded tokens are expected to route with a clear margin"
    assert np.array_equal(ids, ids_ref)
    assert np.max(np.abs(w - w_ref)) <= 1e-5
    err = O.rownorm_rel_err(y, y64)
    assert err.max() <= DECODE_TOL, err.max()
    ym, _, _, hm = O.moe_layer_decode_terms(L, x, spec.k, cache=cache)
    tol_y, tol_h = model_tolerances(spec.D)
    err_m = O.rownorm_rel_err(y, ym)
    assert err_m.max() <= tol_y, err_m.max()
    err_h = O.rownorm_rel_err(h.reshape(T * spec.k, -1), hm.reshape(T * spec.k, -1))
    assert err_h.max() <= tol_h, err_h.max()
    print(f"decode_mx {key} T={T}: y vs float64 {err.max():.2e}, vs operand model {err_m.max():.2e}, "
          f"h vs model {err_h.max():.2e}")
    return err.max()


@pytest.mark.parametrize("key,T,seed", [(0, 1, 1), (0, 3, 2), (0, 8, 3), ("rect", 1, 4), ("rect", 4, 5),
                                        ("rect", 8, 6), (1, 1, 7), (1, 1, 8), (1, 1, 9), (1, 2, 10),
                                        (1, 5, 11), (1, 8, 12)])
def test_decode_mx_layer_parity(moe, key, T, seed):
    check_decode_mx(moe, key, T, seed)


def test_decode_mx_is_deterministic(moe):
    spec, L, layer, _ = packed_layer(moe, 1)
    x = dev(make_tokens(spec, T=3, seed=77))
    ys = []
    for _ in range(5):
        ys.append(layer(x, rail=moe.MOE_RAIL_DECODE_MX).clone())
    torch.cuda.synchronize()
    for y in ys[1:]:
        assert torch.equal(y, ys[0])


def test_decode_mx_rail_and_gemv_rail_agree(moe):
    spec, L, layer, _ = packed_layer(moe, 1)
    x = dev(make_tokens(spec, T=2, seed=78))
    y_mx = layer(x, rail=moe.MOE_RAIL_DECODE_MX)
    y_gemv = layer(x, rail=moe.MOE_RAIL_GEMV)
    y_auto = layer(x)  # both sets of planes, T = 2: the automatic choice is the block-scaled decode rail
    x1 = x[:1]
    y1_auto, y1_gemv = layer(x1), layer(x1, rail=moe.MOE_RAIL_GEMV)  # T = 1: the CUDA-core GEMV rail
    torch.cuda.synchronize()
    assert O.rownorm_rel_err(y_mx.cpu().numpy(), y_gemv.cpu().numpy()).max() <= 2 * DECODE_TOL
    assert torch.equal(y_auto, y_mx)
    assert torch.equal(y1_auto, y1_gemv)


@pytest.mark.parametrize("pinned", [True, False])
def test_decode_mx_host_io(moe, pinned):
    spec, L, layer, cache = packed_layer(moe, 1)
    x = make_tokens(spec, T=1, seed=79)
    xh = torch.from_numpy(x)
    yh = torch.full((1, spec.D), float("nan"))
    if pinned:
        xh, yh = xh.pin_memory(), yh.pin_memory()
    stream = torch.cuda.current_stream()
    for _ in range(2):
        layer.forward_host(xh, yh, rail=moe.MOE_RAIL_DECODE_MX, stream=stream)
    stream.synchronize()
    assert status(moe) == 0
    y64, _, _, _ = O.moe_layer(L, x, spec.k, cache=cache)
    assert O.rownorm_rel_err(yh.numpy(), y64).max() <= DECODE_TOL


def test_decode_mx_workspace_and_rail_limits(moe):
    spec, L, layer, _ = packed_layer(moe, 0)
    assert moe.moe_ffn_packed_workspace_bytes(9, 64, 64, 4, 2, moe.MOE_RAIL_DECODE_MX) == 0  # decode sizes only
    ws = layer.workspace(1, moe.MOE_RAIL_DECODE_MX)
    x = dev(make_tokens(spec, T=1, seed=1))
    y = empty((1, spec.D), torch.float32)
    rc = moe.moe_ffn_layer_packed(layer.packed_struct, x, 1, moe.MOE_RAIL_DECODE_MX, ws, 16, y)
    assert rc == moe.MOE_EINVAL  # workspace too small, rejected before anything is enqueued
    rc = moe.moe_ffn_layer_packed(layer.packed_struct, x, 9, moe.MOE_RAIL_DECODE_MX, ws, ws.numel(), y)
    assert rc == moe.MOE_EUNSUPPORTED


def test_decode_mx_stages_one_call_at_a_time_equal_the_layer(moe):
    spec, L, layer, _ = packed_layer(moe, 1)
    T = 2
    x = dev(make_tokens(spec, T=T, seed=80))
    y_ref = layer(x, rail=moe.MOE_RAIL_DECODE_MX)
    ws = layer.workspace(T, moe.MOE_RAIL_DECODE_MX)
    y = torch.full((T, spec.D), float("nan"), device="cuda")
    for st in (moe.MOE_STAGE_PROLOGUE, moe.MOE_STAGE_GATEUP, moe.MOE_STAGE_DOWN):
        assert moe.moe_ffn_layer_packed_stage(layer.packed_struct, x, T, ws, ws.numel(), st, y) == 0
    torch.cuda.synchronize()
    assert status(moe) == 0
    assert torch.equal(y, y_ref)


def _e2m1_values(codes):
    table = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0.0, -.5, -1, -1.5, -2, -3, -4, -6])
    return table[codes]


def test_decode_mx_x_terms_are_exact(moe):
    """The prologue's x operand (eight E2M1 terms per value) read back from the
    workspace equals the oracle's split bit for bit. Workspace layout of the
    rail: logits [T][E] f32, then x chunks [NK][npad][64] and their scale atoms
    [NK][512], each region 256-byte aligned."""
    spec, L, layer, _ = packed_layer(moe, 1)
    T, D, E = 3, spec.D, spec.E
    x = make_tokens(spec, T=T, seed=81)
    ws = layer.workspace(T, moe.MOE_RAIL_DECODE_MX)
    assert moe.moe_ffn_layer_packed_stage(layer.packed_struct, dev(x), T, ws, ws.numel(), moe.MOE_STAGE_PROLOGUE) == 0
    torch.cuda.synchronize()
    raw = ws.cpu().numpy()
    rnd = lambda v: (v + 255) // 256 * 256  # noqa: E731
    NK, npad, nterm = (D + 127) // 128, 16 * ((T * 8 + 15) // 16), 8
    off_q = rnd(T * E * 4)
    off_s = off_q + rnd(NK * npad * 64)
    xq = raw[off_q:off_q + NK * npad * 64].reshape(NK, npad, 4, 16)
    xs = raw[off_s:off_s + NK * 512].reshape(NK, 512)
    got = np.zeros((T, D))
    for t in range(T):
        for term in range(nterm):
            n = t * nterm + term
            for j in range(NK):
                for kb in range(4):
                    b = 4 * j + kb
                    if b >= D // 32:
                        continue
                    bytes_ = xq[j, n, kb ^ ((n >> 1) & 3)]
                    codes = np.concatenate([bytes_ & 15, bytes_ >> 4])
                    scale = 2.0 ** (int(xs[j, 16 * (n % 32) + 4 * (n // 32) + kb]) - 127)
                    got[t, 32 * b:32 * b + 32] += _e2m1_values(codes) * scale
    ref = O.split_e2m1_terms(x, nterm)
    assert np.array_equal(got, ref)
