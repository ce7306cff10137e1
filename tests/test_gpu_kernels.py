"""GPU parity of each C-ABI entry point against the CPU oracle, element by element.

Sizes span several tiles with ragged tails; tolerances are the ones the layer
is specified with (bit-exact for ids and the CSR, 1e-4 row-normwise for the
fp32 GEMV, bf16 rounding bounds for the tensor-core path).
"""

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from synthetic import make_layer, spec_for
from tests.gpu_helpers import (DECODE_TOL, PREFILL_TOL, bf16_bits_to_f64, dev, empty, routing_check,
                               status)

pytestmark = pytest.mark.gpu


# ---------------------------------------------------------------------------
# router
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("cfg,T", [(0, 8), (1, 1), (1, 3), (2, 512), (4, 4096), (0, 37)])
def test_route_topk_parity(moe, cfg, T):
    spec = spec_for(cfg)
    L = make_layer(spec, with_tokens=False)
    x = np.random.default_rng(100 + T).standard_normal((T, spec.D), dtype=np.float32)
    E, k = spec.E, spec.k
    logits = empty((T, E), torch.float32)
    ids = empty((T, k), torch.int32)
    w = empty((T, k), torch.float32)
    rc = moe.moe_route_topk(dev(x), T, spec.D, dev(L["w_router"]), dev(L["b_router"]), E, k, logits, ids, w)
    assert rc == 0
    torch.cuda.synchronize()
    ref = O.router_logits(x, L["w_router"], L["b_router"])
    routing_check(logits.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy(), ref, k)
    assert status(moe) == 0


def test_route_topk_exact_ties_pick_lower_index(moe):
    # All-zero router: every logit ties; slots must be experts 0..k-1 with equal weights.
    T, D, E, k = 5, 64, 8, 3
    x = np.random.default_rng(0).standard_normal((T, D), dtype=np.float32)
    ids = empty((T, k), torch.int32)
    w = empty((T, k), torch.float32)
    logits = empty((T, E), torch.float32)
    rc = moe.moe_route_topk(dev(x), T, D, dev(np.zeros((E, D), np.float32)), None, E, k, logits, ids, w)
    assert rc == 0
    assert np.array_equal(ids.cpu().numpy(), np.tile(np.arange(k), (T, 1)))
    assert np.allclose(w.cpu().numpy(), 1.0 / k, rtol=0, atol=1e-7)


# ---------------------------------------------------------------------------
# bucket
# ---------------------------------------------------------------------------
def _ids(rng, T, k, E, hot=None):
    rows = []
    for _ in range(T):
        if hot is not None and rng.random() < 0.6:
            rest = [e for e in range(E) if e not in hot]
            rows.append(list(hot[:min(k, len(hot))]) + list(rng.choice(rest, size=k - min(k, len(hot)),
                                                                       replace=False)))
        else:
            rows.append(list(rng.choice(E, size=k, replace=False)))
    return np.array(rows, dtype=np.int32).reshape(T, k)


BUCKET_CASES = [
    # T, k, E, tile, hot experts
    (1, 4, 32, 128, None),
    (8, 2, 4, 128, None),
    (8, 2, 4, 4, None),
    (512, 4, 32, 128, None),
    (4096, 4, 32, 128, (0, 1)),
    (300, 4, 32, 16, (3,)),
    (33, 3, 40, 1, None),
    (127, 1, 2, 128, None),     # one bucket just under the tile, the other just over half
    (257, 1, 2, 128, (0,)),     # bucket sizes crossing 128 and 256
    (1000, 2, 300, 128, None),  # more experts than bucket threads' warps, many empty buckets
]


@pytest.mark.parametrize("T,k,E,tile,hot", BUCKET_CASES)
def test_bucket_bit_exact(moe, T, k, E, tile, hot):
    rng = np.random.default_rng(T * 7 + E)
    ids = _ids(rng, T, k, E, hot)
    mr = moe.moe_bucket_max_rows(T, k, E, tile)
    counts = empty((E,), torch.int32)
    basep = empty((E + 1,), torch.int32)
    rows = torch.full((mr,), 12345, dtype=torch.int32, device="cuda")
    inv = empty((T * k,), torch.int32)
    assert moe.moe_bucket(dev(ids), T, k, E, tile, counts, basep, rows, inv) == 0
    ref = O.bucket_csr(ids, E, tile)
    assert np.array_equal(counts.cpu().numpy(), ref["counts"])
    assert np.array_equal(basep.cpu().numpy(), ref["basep"])
    assert np.array_equal(rows.cpu().numpy(), ref["rows"])
    assert np.array_equal(inv.cpu().numpy(), ref["inv"])
    assert status(moe) == 0


def test_bucket_empty_input(moe):
    E, k, tile = 6, 2, 8
    mr = moe.moe_bucket_max_rows(0, k, E, tile)
    counts = empty((E,), torch.int32)
    basep = empty((E + 1,), torch.int32)
    rows = torch.full((mr,), 7, dtype=torch.int32, device="cuda")
    assert moe.moe_bucket(None, 0, k, E, tile, counts, basep, rows, None) == 0
    assert counts.cpu().numpy().tolist() == [0] * E
    assert basep.cpu().numpy().tolist() == [0] * (E + 1)
    assert np.all(rows.cpu().numpy() == -1)


def test_bucket_flags_out_of_range_ids(moe):
    T, k, E, tile = 6, 2, 4, 4
    ids = np.array([[0, 1], [2, -1], [3, 4], [1, 0], [9, 2], [3, 1]], np.int32)
    mr = moe.moe_bucket_max_rows(T, k, E, tile)
    counts = empty((E,), torch.int32)
    basep = empty((E + 1,), torch.int32)
    rows = empty((mr,), torch.int32)
    inv = empty((T * k,), torch.int32)
    assert moe.moe_bucket(dev(ids), T, k, E, tile, counts, basep, rows, inv) == 0
    assert status(moe) & moe.MOE_STATUS_BAD_EXPERT_ID
    ref = O.bucket_csr(ids, E, tile)  # the oracle skips out-of-range ids the same way
    assert np.array_equal(counts.cpu().numpy(), ref["counts"])
    assert np.array_equal(rows.cpu().numpy(), ref["rows"])
    assert np.array_equal(inv.cpu().numpy(), ref["inv"])
    assert status(moe) == 0  # reading cleared it


def test_bucket_is_deterministic(moe):
    rng = np.random.default_rng(5)
    T, k, E, tile = 4096, 4, 32, 128
    ids = dev(_ids(rng, T, k, E, (0, 1)))
    mr = moe.moe_bucket_max_rows(T, k, E, tile)
    outs = []
    for _ in range(10):
        counts, basep = empty((E,), torch.int32), empty((E + 1,), torch.int32)
        rows, inv = empty((mr,), torch.int32), empty((T * k,), torch.int32)
        assert moe.moe_bucket(ids, T, k, E, tile, counts, basep, rows, inv) == 0
        outs.append(torch.cat([counts, basep, rows, inv]).cpu())
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


# ---------------------------------------------------------------------------
# MXFP4 GEMV
# ---------------------------------------------------------------------------
GEMV_CASES = [
    # E, R, C, n, x_stride_is_zero, bias
    (3, 40, 96, 5, False, True),
    (4, 33, 32, 3, True, False),
    (2, 17, 4096, 2, False, True),
    (32, 2880, 2880, 4, False, True),
    (5, 64, 1024, 7, True, True),
]


@pytest.mark.parametrize("E,R,C,n,shared_x,with_bias", GEMV_CASES)
def test_mxfp4_gemv_parity(moe, E, R, C, n, shared_x, with_bias):
    rng = np.random.default_rng(E * 1000 + C)
    qs = rng.integers(0, 256, size=(E, R, C // 2), dtype=np.uint8)
    sc = rng.integers(110, 136, size=(E, R, C // 32), dtype=np.uint8)
    bias = (rng.standard_normal((E, R)) * 0.02).astype(np.float32) if with_bias else None
    experts = rng.integers(0, E, size=n).astype(np.int32)
    x = rng.standard_normal((1 if shared_x else n, C), dtype=np.float32)
    out = empty((n, R), torch.float32)
    rc = moe.moe_mxfp4_gemv(dev(qs), dev(sc), E, R, C, dev(experts), n, dev(x), 0 if shared_x else C,
                            None if bias is None else dev(bias), out)
    assert rc == 0
    got = out.cpu().numpy()
    for i in range(n):
        e = experts[i]
        ref = O.mxfp4_gemv(qs[e], sc[e], x[0 if shared_x else i], None if bias is None else bias[e])
        assert O.rownorm_rel_err(got[i], ref) <= DECODE_TOL
    assert status(moe) == 0


def test_mxfp4_gemv_extreme_scales(moe):
    # Every E8M0 byte 0..254 appears: denormal 2^-127 through 2^127 scales decode exactly.
    rng = np.random.default_rng(3)
    E, R, C = 1, 255, 64
    qs = rng.integers(0, 256, size=(E, R, C // 2), dtype=np.uint8)
    sc = np.stack([np.full(C // 32, s, np.uint8) for s in range(255)])[None]
    x = rng.standard_normal((1, C), dtype=np.float32) * 1e-3
    out = empty((1, R), torch.float32)
    assert moe.moe_mxfp4_gemv(dev(qs), dev(sc), E, R, C, dev(np.zeros(1, np.int32)), 1, dev(x), 0, None, out) == 0
    got = out.cpu().numpy()[0].astype(np.float64)
    ref = O.mxfp4_gemv(qs[0], sc[0], x[0], None)
    finite = np.isfinite(ref) & (np.abs(ref) < 3e38) & (np.abs(ref) > 1e-36)
    rel = np.abs(got[finite] - ref[finite]) / np.abs(ref[finite])
    assert np.all(rel < 1e-4)


def test_mxfp4_gemv_bad_expert_sets_status(moe):
    E, R, C = 2, 16, 64
    qs = np.zeros((E, R, C // 2), np.uint8)
    sc = np.full((E, R, C // 32), 127, np.uint8)
    out = torch.full((2, R), 5.0, device="cuda")
    rc = moe.moe_mxfp4_gemv(dev(qs), dev(sc), E, R, C, dev(np.array([1, 7], np.int32)), 2,
                            dev(np.ones((1, C), np.float32)), 0, None, out)
    assert rc == 0
    assert status(moe) & moe.MOE_STATUS_BAD_EXPERT_ID
    assert torch.all(out[1] == 0)


# ---------------------------------------------------------------------------
# swiglu
# ---------------------------------------------------------------------------
def test_swiglu_parity(moe):
    rng = np.random.default_rng(11)
    n = 100003
    g = (rng.standard_normal(n) * 6).astype(np.float32)
    u = (rng.standard_normal(n) * 6).astype(np.float32)
    g[:6] = [1e4, -1e4, 0.0, 7.0, -80.0, 3.0]
    u[:6] = [0.5, 2.0, 1.0, -1.0, 100.0, -100.0]
    ref = O.swiglu_oai(g, u)
    h = empty((n,), torch.float32)
    assert moe.moe_swiglu_oai(dev(g), dev(u), h, n, moe.MOE_DTYPE_F32) == 0
    got = h.cpu().numpy().astype(np.float64)
    assert not np.any(np.isnan(got))
    assert np.all(np.abs(got - ref) <= 2e-6 * np.maximum(np.abs(ref), 1.0))
    hb = empty((n,), torch.bfloat16)
    assert moe.moe_swiglu_oai(dev(g), dev(u), hb, n, moe.MOE_DTYPE_BF16) == 0
    gotb = hb.float().cpu().numpy().astype(np.float64)
    # within one bf16 ulp of the correctly rounded value
    assert np.all(np.abs(gotb - O.round_bf16(ref)) <= 2.0 ** -7 * np.abs(ref) + 1e-30)


@pytest.mark.parametrize("T,D", [(1, 2880), (6, 2880), (3, 64), (2, 1000)])
def test_rms_renorm_parity(moe, T, D):
    rng = np.random.default_rng(T * 7 + D)
    scale = np.array([1e-3, 1.0, 30.0, 1e4, 0.5, 2.0])[:T, None]
    x = (rng.standard_normal((T, D)) * scale).astype(np.float32)
    if T > 1:
        x[T - 1] = 0.0  # a zero row stays zero
    ref = O.rms_renorm(x)
    y = empty((T, D), torch.float32)
    assert moe.moe_rms_renorm(dev(x), T, D, y) == 0
    got = y.cpu().numpy().astype(np.float64)
    # fp32 sum of squares and one division per element: a few ulp of 1
    assert np.all(np.abs(got - ref) <= 4e-6 * np.maximum(np.abs(ref), 1e-3))
    xi = dev(x)
    assert moe.moe_rms_renorm(xi, T, D, xi) == 0  # in place
    assert np.array_equal(xi.cpu().numpy(), y.cpu().numpy())
    assert status(moe) == 0


# ---------------------------------------------------------------------------
# gather + grouped GEMM (tcgen05)
# ---------------------------------------------------------------------------
def _bucket_on_gpu(moe, ids, E, tile=128):
    T, k = ids.shape
    mr = moe.moe_bucket_max_rows(T, k, E, tile)
    counts, basep = empty((E,), torch.int32), empty((E + 1,), torch.int32)
    rows, inv = empty((mr,), torch.int32), empty((T * k,), torch.int32)
    assert moe.moe_bucket(dev(ids), T, k, E, tile, counts, basep, rows, inv) == 0
    return counts, basep, rows, inv, mr


def test_gather_rows_bf16(moe):
    rng = np.random.default_rng(2)
    T, k, E, D = 50, 3, 7, 192
    ids = _ids(rng, T, k, E)
    x = rng.standard_normal((T, D), dtype=np.float32)
    counts, basep, rows, inv, mr = _bucket_on_gpu(moe, ids, E)
    xg = torch.full((mr, D), -1, dtype=torch.int16, device="cuda")
    y = torch.full((T, D), 3.0, device="cuda")
    xlo = torch.full((mr, D), -1, dtype=torch.int16, device="cuda")
    assert moe.moe_gather_rows_bf16(dev(x), T, D, k, rows, basep, E, mr, xg, xlo, y) == 0
    ref = O.bucket_csr(ids, E, 128)
    got = bf16_bits_to_f64(xg)
    got_lo = bf16_bits_to_f64(xlo)
    mpad = ref["basep"][E]
    for p in range(mpad):
        a = ref["rows"][p]
        hi = O.round_bf16(x[a // k]) if a >= 0 else np.zeros(D)
        lo = O.round_bf16(x[a // k].astype(np.float64) - hi) if a >= 0 else np.zeros(D)
        assert np.array_equal(got[p], hi), p
        assert np.array_equal(got_lo[p], lo), p
    assert torch.all(y == 0)


def _mm_case(rng, E, R, C, counts_wanted, k=1):
    """Token rows routed so that expert e receives counts_wanted[e] rows (k = 1)."""
    ids = np.concatenate([np.full(c, e, np.int32) for e, c in enumerate(counts_wanted)])
    rng.shuffle(ids)
    T = len(ids)
    ids = ids.reshape(T, 1)
    qs = rng.integers(0, 256, size=(E, R, C // 2), dtype=np.uint8)
    sc = rng.integers(110, 136, size=(E, R, C // 32), dtype=np.uint8)
    x = rng.standard_normal((T, C), dtype=np.float32)
    bias = (rng.standard_normal((E, R)) * 0.5).astype(np.float32)
    return ids, qs, sc, x, bias


MM_CASES = [
    # E, R, C, counts per expert
    (4, 64, 64, [3, 0, 5, 1]),
    (3, 264, 192, [127, 128, 129]),
    (4, 128, 256, [0, 300, 1, 64]),
    (2, 2880, 2880, [70, 130]),
]


def split_operand(x):
    hi = O.round_bf16(x)
    return hi + O.round_bf16(np.asarray(x, np.float64) - hi)


@pytest.mark.parametrize("E,R,C,cnt", MM_CASES)
@pytest.mark.parametrize("with_bias,split", [(True, False), (False, False), (True, True)])
def test_grouped_mm_store_parity(moe, E, R, C, cnt, with_bias, split):
    rng = np.random.default_rng(R + C + E)
    ids, qs, sc, x, bias = _mm_case(rng, E, R, C, cnt)
    T = ids.shape[0]
    counts, basep, rows, inv, mr = _bucket_on_gpu(moe, ids, E)
    xg = empty((mr, C), torch.int16)
    xlo = empty((mr, C), torch.int16)
    assert moe.moe_gather_rows_bf16(dev(x), T, C, 1, rows, basep, E, mr, xg, xlo if split else None) == 0
    out = torch.full((mr, R), 0, dtype=torch.int16, device="cuda")
    rc = moe.moe_mxfp4_grouped_mm(dev(qs), dev(sc), dev(bias) if with_bias else None, None, None, None,
                                  E, R, C, xg, xlo if split else None, counts, basep, rows, mr, 1, None,
                                  moe.MOE_EPI_STORE_BF16, 1.702, 7.0, out, R)
    assert rc == 0
    torch.cuda.synchronize()
    assert status(moe) == 0
    ref_b = O.bucket_csr(ids, E, 128)
    got = bf16_bits_to_f64(out)
    xb = split_operand(x) if split else O.round_bf16(x)
    for e in range(E):
        if cnt[e] == 0:
            continue
        W = O.dequant_mxfp4(qs[e], sc[e])
        p0 = ref_b["basep"][e]
        toks = ref_b["rows"][p0:p0 + cnt[e]]
        acc = xb[toks] @ W.T + (bias[e] if with_bias else 0.0)
        assert np.max(O.rownorm_rel_err(got[p0:p0 + cnt[e]], O.round_bf16(acc))) <= 8e-3, e


def _fp32_projection(moe, qs, sc, bias, E, R, C, xg, xlo, counts, basep, rows, mr, T):
    """One grouped GEMM's fp32 accumulators per token, read through the scatter
    epilogue with k = 1 and weight 1 (a single atomic add onto zero is exact)."""
    y = torch.zeros((T, R), dtype=torch.float32, device="cuda")
    ones = torch.ones((T,), dtype=torch.float32, device="cuda")
    rc = moe.moe_mxfp4_grouped_mm(dev(qs), dev(sc), dev(bias), None, None, None, E, R, C, xg, xlo, counts, basep,
                                  rows, mr, 1, ones, moe.MOE_EPI_SCATTER_WEIGHTED, 1.702, 7.0, y, R)
    assert rc == 0
    return y.cpu().numpy().astype(np.float64)


def _bf16_ulp(v):
    """Spacing of bfloat16 values at |v| (normal range)."""
    a = np.maximum(np.abs(v), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


@pytest.mark.parametrize("E,R,C,cnt", MM_CASES)
@pytest.mark.parametrize("split", [False, True])
def test_grouped_mm_swiglu_parity(moe, E, R, C, cnt, split):
    rng = np.random.default_rng(7 * R + C)
    ids, qs, sc, x, bias = _mm_case(rng, E, R, C, cnt)
    qs2 = rng.integers(0, 256, size=qs.shape, dtype=np.uint8)
    sc2 = rng.integers(110, 136, size=sc.shape, dtype=np.uint8)
    bias2 = (rng.standard_normal((E, R)) * 0.5).astype(np.float32)
    T = ids.shape[0]
    counts, basep, rows, inv, mr = _bucket_on_gpu(moe, ids, E)
    xg = empty((mr, C), torch.int16)
    xlo = empty((mr, C), torch.int16)
    lo = xlo if split else None
    assert moe.moe_gather_rows_bf16(dev(x), T, C, 1, rows, basep, E, mr, xg, lo) == 0
    out = empty((mr, R), torch.int16)
    rc = moe.moe_mxfp4_grouped_mm(dev(qs), dev(sc), dev(bias), dev(qs2), dev(sc2), dev(bias2), E, R, C,
                                  xg, lo, counts, basep, rows, mr, 1, None,
                                  moe.MOE_EPI_SWIGLU_BF16, 1.702, 7.0, out, R)
    assert rc == 0
    # the same two GEMMs with their fp32 accumulators read out (one token per row, k = 1)
    g_gpu = _fp32_projection(moe, qs, sc, bias, E, R, C, xg, lo, counts, basep, rows, mr, T)
    u_gpu = _fp32_projection(moe, qs2, sc2, bias2, E, R, C, xg, lo, counts, basep, rows, mr, T)
    assert status(moe) == 0
    ref_b = O.bucket_csr(ids, E, 128)
    got = bf16_bits_to_f64(out)
    xb = split_operand(x) if split else O.round_bf16(x)
    for e in range(E):
        if cnt[e] == 0:
            continue
        p0 = ref_b["basep"][e]
        toks = ref_b["rows"][p0:p0 + cnt[e]]
        # The epilogue alone: swiglu_oai of the GPU's own fp32 g and u, rounded to
        # bf16, within one bf16 ulp (its sigmoid uses the fast exponential).
        h_own = O.round_bf16(O.swiglu_oai(g_gpu[toks], u_gpu[toks]))
        diff = np.abs(got[p0:p0 + cnt[e]] - h_own)
        assert np.all(diff <= _bf16_ulp(h_own) + 1e-30), (e, diff.max())
        # The whole fused GEMM against float64 accumulation of the same operands:
        # the prefill bound (a row of g or u reaches ~5e4 at these E8M0 scales, so
        # fp32 accumulation moves single features by tenths, which the swiglu
        # passes on with a gain up to 8).
        g = xb[toks] @ O.dequant_mxfp4(qs[e], sc[e]).T + bias[e]
        u = xb[toks] @ O.dequant_mxfp4(qs2[e], sc2[e]).T + bias2[e]
        h = O.swiglu_oai(g, u)
        assert np.max(O.rownorm_rel_err(got[p0:p0 + cnt[e]], h)) <= PREFILL_TOL, e


@pytest.mark.parametrize("E,R,C,cnt,k", [(4, 64, 64, [3, 0, 5, 1], 1), (5, 136, 128, [40, 0, 129, 7, 80], 2),
                                         (2, 2880, 2880, [70, 130], 2)])
def test_grouped_mm_scatter_parity(moe, E, R, C, cnt, k):
    rng = np.random.default_rng(13 * R + C)
    ids1, qs, sc, h, bias = _mm_case(rng, E, R, C, cnt)
    n = ids1.shape[0]
    if n % k:
        pytest.skip("assignment count not divisible by k")
    T = n // k
    ids = ids1.reshape(T, k)
    # distinct experts per token are not needed by the kernel; weights are arbitrary
    w = rng.random((T, k)).astype(np.float32)
    counts, basep, rows, inv, mr = _bucket_on_gpu(moe, ids, E)
    ref_b = O.bucket_csr(ids, E, 128)
    # the A operand is already in bucket order here: row p holds h of assignment rows[p]
    a = np.zeros((mr, C), np.float32)
    live = ref_b["rows"] >= 0
    a[live] = h[ref_b["rows"][live]]
    a_bits = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).to("cuda")
    y = torch.zeros((T, R), dtype=torch.float32, device="cuda")
    rc = moe.moe_mxfp4_grouped_mm(dev(qs), dev(sc), dev(bias), None, None, None, E, R, C, a_bits, None,
                                  counts, basep, rows, mr, k, dev(w), moe.MOE_EPI_SCATTER_WEIGHTED, 1.702, 7.0,
                                  y, R)
    assert rc == 0
    assert status(moe) == 0
    hb = O.round_bf16(h)
    ref = np.zeros((T, R))
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            ref[t] += w[t, j] * (O.dequant_mxfp4(qs[e], sc[e]) @ hb[t * k + j] + bias[e])
    assert np.max(O.rownorm_rel_err(y.cpu().numpy(), ref)) <= 1e-4
