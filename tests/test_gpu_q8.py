"""GPU parity of the Q8 activation rail: the 32-block requant and the MXFP4 x Q8
integer-dot GEMV bit for bit against the oracle, and the layer on the Q8 rail
against the float64 layer and against the oracle on the same Q8 operands."""

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from synthetic import make_layer, make_tokens, spec_for
from tests.gpu_helpers import dev, empty, status
from tests.test_gpu_layer import layer_for

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,C", [(1, 32), (5, 2880), (3, 4096), (17, 64)])
def test_quantize_q8_bit_exact(moe, rows, C):
    rng = np.random.default_rng(rows * 13 + C)
    x = (rng.standard_normal((rows, C)) * rng.uniform(1e-4, 1e4, (rows, 1))).astype(np.float32)
    x[0, :32] = 0.0                       # an all-zero block
    if C >= 64:
        x[0, 32:36] = [127.0, -63.5, 0.5, 1.5]  # ties to even at scale 1
        x[0, 36:64] = 0.25
    q = empty((rows, C), torch.int8)
    d = empty((rows, C // 32), torch.float32)
    assert moe.moe_quantize_q8(dev(x), rows, C, q, d) == 0
    q_ref, d_ref = O.quantize_q8(x)
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(d.cpu().numpy().view(np.uint32), d_ref.view(np.uint32))
    assert status(moe) == 0


@pytest.mark.parametrize("E,R,C,n,act_div", [(4, 64, 64, 3, 1), (3, 200, 2880, 6, 2), (2, 131, 4096, 2, 1),
                                             (6, 8, 1024, 8, 4)])
def test_gemv_q8_bit_exact(moe, E, R, C, n, act_div):
    rng = np.random.default_rng(E * 100 + R + C)
    qs = rng.integers(0, 256, (E, R, C // 2), dtype=np.uint8)
    sc = rng.integers(110, 136, (E, R, C // 32), dtype=np.uint8)
    sc[0, 0, :] = np.arange(C // 32) % 255  # scales from 0 (2^-127, subnormal products) upwards
    bias = rng.standard_normal((E, R)).astype(np.float32)
    experts = rng.integers(0, E, n).astype(np.int32)
    experts[0] = 0
    na = (n + act_div - 1) // act_div
    x = rng.standard_normal((na, C)).astype(np.float32)
    q, d = O.quantize_q8(x)
    out = empty((n, R), torch.float32)
    assert moe.moe_mxfp4_gemv_q8(dev(qs), dev(sc), E, R, C, dev(experts), n, act_div, dev(q), dev(d), dev(bias),
                                 out) == 0
    got = out.cpu().numpy()
    for i in range(n):
        e, a = int(experts[i]), i // act_div
        ref = O.mxfp4_gemv_q8(qs[e], sc[e], q[a], d[a], bias[e])
        assert np.array_equal(got[i].view(np.uint32), ref.view(np.uint32)), (i, np.abs(got[i] - ref).max())
    assert status(moe) == 0


def test_gemv_q8_bad_expert_gives_a_zero_row(moe):
    rng = np.random.default_rng(3)
    E, R, C = 2, 16, 64
    qs = rng.integers(0, 256, (E, R, C // 2), dtype=np.uint8)
    sc = np.full((E, R, C // 32), 127, np.uint8)
    q, d = O.quantize_q8(rng.standard_normal((1, C)).astype(np.float32))
    out = torch.full((2, R), float("nan"), device="cuda")
    experts = np.array([1, 7], np.int32)
    assert moe.moe_mxfp4_gemv_q8(dev(qs), dev(sc), E, R, C, dev(experts), 2, 2, dev(q), dev(d), None, out) == 0
    torch.cuda.synchronize()
    rc, st = moe.moe_get_status()
    assert st & moe.MOE_STATUS_BAD_EXPERT_ID
    o = out.cpu().numpy()
    assert np.array_equal(o[0], O.mxfp4_gemv_q8(qs[1], sc[1], q[0], d[0], None)) and not o[1].any()


@pytest.mark.parametrize("cfg,T", [(0, 8), (0, 1), (1, 1), (1, 8)])
def test_layer_q8_rail(moe, cfg, T):
    spec, L, layer, cache = layer_for(moe, cfg)
    x = make_tokens(spec, T=T, seed=60 + T)
    k = spec.k
    ids = empty((T, k), torch.int32)
    w = empty((T, k), torch.float32)
    y = layer(dev(x), rail=moe.MOE_RAIL_GEMV_Q8, ids_out=ids, weights_out=w)
    torch.cuda.synchronize()
    assert status(moe) == 0
    y, ids = y.cpu().numpy(), ids.cpu().numpy()
    logits = O.router_logits(x, L["w_router"], L["b_router"])
    margin = O.routing_margins(logits, k)
    clear = margin > 1e-4 * np.abs(logits).max()
    ids_ref, _ = O.topk_softmax(logits, k)
    assert np.array_equal(ids[clear], ids_ref[clear])
    sel = np.take_along_axis(logits, ids.astype(np.int64), 1)
    w_ref = np.exp(sel - sel[:, :1])
    w_ref /= w_ref.sum(1, keepdims=True)
    y64, _, _, _ = O.moe_layer(L, x, k, ids=ids, weights=w_ref, cache=cache)
    yq8, _, _, _ = O.moe_layer(L, x, k, ids=ids, weights=w_ref, cache=cache, operands="q8")
    err64 = O.rownorm_rel_err(y, y64).max()
    errq8 = O.rownorm_rel_err(y, yq8).max()
    model64 = O.rownorm_rel_err(yq8, y64).max()  # the requant's own distance from the float64 layer
    print(f"q8 rail cfg {cfg} T {T}: rownorm err vs float64 {err64:.3e} (the Q8 operands themselves "
          f"{model64:.3e}), vs the same Q8 operands {errq8:.3e}")
    # the kernels compute the Q8 operand model (float32 sums, float32 swiglu): whatever distance from
    # float64 remains is the format's, not the kernels'
    assert errq8 <= 1e-5
    assert abs(err64 - model64) <= 1e-5 * max(1.0, model64)


def test_layer_q8_rail_is_deterministic(moe):
    spec, L, layer, _ = layer_for(moe, 1)
    x = dev(make_tokens(spec, T=4, seed=91))
    ys = [layer(x, rail=moe.MOE_RAIL_GEMV_Q8).clone() for _ in range(3)]
    torch.cuda.synchronize()
    assert all(torch.equal(ys[0], yy) for yy in ys[1:])
