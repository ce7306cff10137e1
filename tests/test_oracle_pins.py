"""Pins of the CPU oracle against things other than itself.

Each check is a plain function taking the oracle functions it exercises as
arguments, so tests/test_oracle_mutations.py can hand it a copy with a planted
mistake and see it fail.
"""

import math
import os

import numpy as np
import pytest

from oracle import brute
from oracle import moe_oracle as O
from synthetic import make_layer, spec_for

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load_e2m1_golden():
    vals = {}
    with open(os.path.join(GOLDEN, "e2m1_table.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            c, v = line.split()
            vals[int(c)] = float(v)
    assert sorted(vals) == list(range(16))
    return vals


def tiny_planes(rng, R, C, s_lo=120, s_hi=130):
    qs = rng.integers(0, 256, size=(R, C // 2), dtype=np.uint8)
    sc = rng.integers(s_lo, s_hi + 1, size=(R, C // 32), dtype=np.uint8)
    return qs, sc


# ---------------------------------------------------------------------------
# reusable checks (return True when the pin holds)
# ---------------------------------------------------------------------------

def check_e2m1(e2m1_value):
    gold = load_e2m1_golden()
    for c in range(16):
        v = e2m1_value(c)
        if v != gold[c] or math.copysign(1.0, v) != math.copysign(1.0, gold[c]):
            return False
    return True


def check_dequant_vs_brute(dequant, seed=0):
    rng = np.random.default_rng(seed)
    for R, C in [(3, 32), (5, 64), (2, 96)]:
        qs, sc = tiny_planes(rng, R, C)
        ref = np.array(brute.dequant(qs.tolist(), sc.tolist()))
        got = dequant(qs, sc)
        if got.shape != ref.shape or not np.array_equal(got, ref):
            return False
    return True


def check_topk_vs_brute(topk_softmax, seed=1):
    rng = np.random.default_rng(seed)
    for E, k in [(4, 2), (6, 3), (5, 5), (8, 1)]:
        # integer-valued logits make exact ties frequent
        logits = rng.integers(-3, 4, size=(40, E)).astype(np.float64)
        logits[::3] += rng.standard_normal((len(logits[::3]), E))
        ids, w = topk_softmax(logits, k)
        for t in range(len(logits)):
            bid, bw = brute.topk(logits[t].tolist(), k)
            if list(ids[t]) != bid or not np.allclose(w[t], bw, rtol=1e-14, atol=0):
                return False
    return True


def check_bucket_vs_brute(bucket_csr, seed=2):
    rng = np.random.default_rng(seed)
    for T, k, E, tile in [(8, 2, 4, 4), (13, 3, 5, 16), (1, 4, 32, 128), (40, 4, 6, 1), (0, 2, 3, 4)]:
        ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]) if T else \
            np.zeros((0, k), np.int64)
        got = bucket_csr(ids, E, tile)
        counts, basep, rows, inv = brute.bucket(ids.tolist(), E, tile, k=k)
        mpad = basep[-1]
        if list(got["counts"]) != counts or list(got["basep"]) != basep:
            return False
        if list(got["rows"][:mpad]) != rows or not np.all(got["rows"][mpad:] == -1):
            return False
        if list(got["inv"]) != inv:
            return False
    return True


def check_swiglu_points(swiglu_oai):
    a = O.SWIGLU_ALPHA
    sig = lambda z: 1.0 / (1.0 + math.exp(-z))  # noqa: E731  (z >= 0 here)
    cases = [
        # (g, u, expected)
        (9.0, 0.5, 7.0 * sig(7.0 * a) * 1.5),        # g clamped at 7 from above
        (7.0, 100.0, 7.0 * sig(7.0 * a) * 8.0),      # u clamped at +7
        (0.0, 3.0, 0.0),                              # g = 0 -> 0
        (2.5, -1.0, 0.0),                             # u = -1 -> 0
        (1.0, -50.0, 1.0 * sig(a) * -6.0),           # u clamped at -7 -> factor -6
        (1.0, 0.0, sig(a)),                           # plain point
        (-0.5, 2.0, -0.5 * (1.0 - sig(0.5 * a)) * 3.0),
    ]
    for g, u, exp in cases:
        got = float(swiglu_oai(np.array([g]), np.array([u]))[0])
        if not math.isclose(got, exp, rel_tol=1e-14, abs_tol=1e-300):
            return False
    # very negative g: tends to -0, never NaN
    got = swiglu_oai(np.array([-1e4, -800.0]), np.array([0.0, 5.0]))
    if np.any(np.isnan(got)) or np.any(np.abs(got) > 1e-300):
        return False
    return True


def check_layer_vs_brute(moe_layer, seed_layer=0):
    spec = spec_for(0)
    L = make_layer(spec, layer=seed_layer)
    y, ids, w, _ = moe_layer(L, L["x"], spec.k)
    by, bids, bw = brute.layer(L, L["x"], spec.k)
    if [list(r) for r in ids] != bids:
        return False
    by = np.array(by)
    return bool(np.max(O.rownorm_rel_err(y, by, floor=1e-300)) < 1e-12)


def check_bias_linearity(moe_layer):
    spec = spec_for(0)
    L = make_layer(spec, layer=3)
    L0 = dict(L)
    L0["bd"] = np.zeros_like(L["bd"])
    y1, ids, w, _ = moe_layer(L, L["x"], spec.k)
    y0, _, _, _ = moe_layer(L0, L["x"], spec.k)
    expect = np.einsum("tj,tjd->td", w, L["bd"].astype(np.float64)[ids])
    return bool(np.allclose(y1 - y0, expect, rtol=1e-9, atol=1e-12 * np.abs(y1).max()))



def check_routing_margins(routing_margins):
    """Hand-written logits whose smallest top-(k+1) gap is known."""
    cases = [
        # (logits [T, E], k, expected per-token margin)
        ([[5.0, 3.0, 2.5, 1.0, 0.0]], 2, [0.5]),          # the k / k+1 gap (3 vs 2.5) is the smallest
        ([[4.0, 3.9, 1.0, 0.0]], 2, [0.1]),               # a gap between selected slots is smaller
        ([[1.0, 2.0, 2.0, 0.0]], 1, [0.0]),               # exact tie at the k / k+1 boundary
        ([[1.0, 3.0, 2.0]], 3, [1.0]),                    # k = E: only the gaps between the k selected
        ([[7.0]], 1, [math.inf]),                         # k = E = 1: nothing to separate
        ([[0.0, -2.0, 9.0, -1.0, 4.0],                    # tokens are rows: 9, 4, 0 -> 4;
          [0.0, 1.0, 2.0, 3.0, 10.0]], 2, [4.0, 1.0]),     # 10, 3, 2 -> 1
        ([[-3.0, -1.0, -6.0, -1.25]], 2, [0.25]),         # negative logits, unsorted input
        ([[2.0, 8.0, 5.0, 7.5, 6.0]], 3, [0.5]),          # 8, 7.5, 6, 5: gaps 0.5, 1.5, 1
    ]
    for logits, k, exp in cases:
        got = np.asarray(routing_margins(np.array(logits, dtype=np.float64), k), np.float64)
        if got.shape != (len(exp),) or not np.allclose(got, exp, rtol=0, atol=1e-12):
            return False
    return True


def check_rownorm_rel_err(rownorm_rel_err):
    """Per-row max abs error over the reference row's max magnitude, floored."""
    cases = [
        # (y, y_ref, floor, expected per-row error)
        ([[1.5, -4.0, 2.0]], [[1.0, -4.0, 2.0]], 1e-3, [0.125]),   # 0.5 / 4
        ([[4.0]], [[2.0]], 1e-3, [1.0]),                           # relative to the reference, not to y
        ([[1.0, 1.0, 1.0, 1.4]], [[1.0, 1.0, 1.0, 1.0]], 1e-3, [0.4]),  # the max error, not the mean
        ([[101.0, 0.0], [1.0, 0.5]], [[100.0, 0.0], [1.0, 0.0]], 1e-3, [0.01, 0.5]),  # rows scaled separately
        ([[1e-4, 0.0]], [[0.0, 0.0]], 1e-3, [0.1]),                # the floor replaces a zero row's scale
        ([[2e-4, 0.0]], [[5e-4, 0.0]], 1e-3, [0.3]),               # ... and a row smaller than the floor
        ([[2e-4, 0.0]], [[5e-4, 0.0]], 1e-6, [0.6]),               # the floor argument is used
    ]
    for y, y_ref, floor, exp in cases:
        got = np.asarray(rownorm_rel_err(np.array(y), np.array(y_ref), floor=floor), np.float64)
        if got.shape != (len(exp),) or not np.allclose(got, exp, rtol=1e-12, atol=0):
            return False
    return True


def check_bucket_max_rows(bucket_max_rows):
    """Hand values of T*k + E*(tile-1) rounded up to a whole tile, and the bound over every routing."""
    cases = [
        ((1, 4, 32, 1), 4),          # tile 1: no padding at all
        ((512, 4, 32, 128), 6144),   # 2048 + 32*127 = 6112 -> 48 tiles
        ((8, 2, 4, 16), 80),         # 16 + 60 = 76 -> 5 tiles
        ((0, 4, 32, 128), 4096),     # no tokens: every expert could still own a padded tile
        ((3, 1, 2, 4), 12),          # 3 + 6 = 9 -> 3 tiles
        ((4096, 4, 32, 128), 20480), # 16384 + 4064 = 20448 -> 160 tiles
    ]
    for args, exp in cases:
        if int(bucket_max_rows(*args)) != exp:
            return False
    # every assignment of ids in tiny cases fits under the bound; with k = 1 the
    # worst one (one token per expert) reaches it exactly
    import itertools
    for T, k, E, tile, tight in [(3, 1, 3, 2, True), (3, 2, 3, 2, False), (2, 2, 2, 3, False)]:
        bound = int(bucket_max_rows(T, k, E, tile))
        worst = 0
        for choice in itertools.product(range(E), repeat=T * k):
            counts = np.bincount(np.array(choice), minlength=E)
            worst = max(worst, int(sum(-(-c // tile) * tile for c in counts)))
        if worst > bound or (tight and worst != bound):
            return False
    return True



def check_decode_terms_layer(layer_fn):
    """With enough terms to hold every bit of the float32 operands the decode
    rail's operand model is the layer itself (the router weight distributes over
    the down projection); with five terms it stays within its 2^-20 bound."""
    spec = spec_for(0)
    L = make_layer(spec, layer=5)
    y_ref, ids_ref, w_ref, _ = O.moe_layer(L, L["x"], spec.k)
    y8, ids, w, h8 = layer_fn(L, L["x"], spec.k, x_terms=13, h_terms=13)  # 13 E2M1 terms hold a float32
    if not np.array_equal(ids, ids_ref) or np.max(O.rownorm_rel_err(y8, y_ref, floor=1e-300)) > 1e-6:
        return False
    # h of each slot against the float64 expert (x in eight terms is x itself)
    for t in range(L["x"].shape[0]):
        for j in range(spec.k):
            e = int(ids[t, j])
            g = L["x"][t].astype(np.float64) @ O.dequant_mxfp4(L["g_qs"][e], L["g_sc"][e]).T + L["bg"][e]
            u = L["x"][t].astype(np.float64) @ O.dequant_mxfp4(L["u_qs"][e], L["u_sc"][e]).T + L["bu"][e]
            if np.max(np.abs(h8[t, j] - O.swiglu_oai(g, u))) > 1e-9 * max(1.0, np.abs(h8[t, j]).max()):
                return False
    y5, _, _, _ = layer_fn(L, L["x"], spec.k)
    return bool(np.max(O.rownorm_rel_err(y5, y_ref)) < 1e-4)



def e2m1_magnitudes():
    """The 8 non-negative E2M1 magnitudes by code, from the printed table."""
    gold = load_e2m1_golden()
    return [gold[c] for c in range(8)]


def brute_round_e2m1(v):
    """Nearest E2M1 value by exhaustive search over the 16 codes, ties to the code with mantissa bit 0."""
    gold = load_e2m1_golden()
    best = None
    for c in range(16):
        val = gold[c]
        if (val < 0) != (v < 0 or (v == 0 and math.copysign(1.0, v) < 0)) and val != 0:
            continue
        d = abs(v - val)
        key = (d, c & 1)  # nearer first, then even mantissa
        if best is None or key < best[0]:
            best = (key, val)
    mag = min(abs(best[1]), 6.0)
    return math.copysign(mag, v)


def e2m1_probe_values():
    vals = [0.0, 0.1, 0.24, 0.25, 0.26, 0.5, 0.74, 0.75, 0.76, 1.0, 1.25, 1.3, 1.5, 1.75, 1.8, 2.0, 2.49,
            2.5, 2.51, 3.0, 3.5, 3.9, 4.0, 4.9, 5.0, 5.1, 6.0, 6.9, 7.0, 100.0]
    return np.array(vals + [-v for v in vals if v != 0.0])


def check_round_e2m1(round_e2m1):
    v = e2m1_probe_values()
    got = np.asarray(round_e2m1(v), np.float64)
    ref = np.array([brute_round_e2m1(float(a)) for a in v])
    return bool(np.array_equal(got, ref))


def brute_split_e2m1_terms(block, nterms):
    """Pure-Python split of one block of 32 into E2M1 terms: the smallest power of two 2^e with
    max|r| <= 6 * 2^e, found by counting, and the exhaustive nearest-value search above."""
    r = [float(np.float32(b)) for b in block]
    total = [0.0] * 32
    for _ in range(nterms):
        amax = max(abs(a) for a in r)
        e = -127
        while e < 127 and amax > 6.0 * 2.0 ** e:
            e += 1
        terms = [brute_round_e2m1(a / 2.0 ** e) * 2.0 ** e for a in r]
        total = [t0 + t1 for t0, t1 in zip(total, terms)]
        r = [a - t for a, t in zip(r, terms)]
    return total


def check_split_e2m1_vs_brute(split_e2m1_terms, seed=8):
    rng = np.random.default_rng(seed)
    for scale in (1e-30, 1e-3, 1.0, 37.0, 3e4):
        blocks = (rng.standard_normal((3, 32)) * scale).astype(np.float32)
        blocks[1, 5] = 0.0
        for n in (1, 2, 4, 8):
            got = split_e2m1_terms(blocks, n)
            ref = np.array([brute_split_e2m1_terms(b, n) for b in blocks])
            if not np.array_equal(got, ref):
                return False
    return True


# ---------------------------------------------------------------------------
# tests
# ---------------------------------------------------------------------------

def test_e2m1_matches_printed_table():
    assert check_e2m1(O.e2m1_value)
    assert np.array_equal(O.E2M1_LUT, np.array([load_e2m1_golden()[c] for c in range(16)]))


def test_e8m0_exhaustive():
    # 2**(s-127) against math.ldexp, and against the float32 exponent-field bitcast
    # (s << 23) that the pages' ALU decode uses, for every byte 1..254; byte 0 is
    # the float32 denormal 2**-127 (bit pattern 0x00400000); 255 is NaN.
    for s in range(255):
        v = O.e8m0_value(s)
        assert v == math.ldexp(1.0, s - 127)
        bits = (s << 23) if s >= 1 else 0x00400000
        f32 = np.array([bits], dtype=np.uint32).view(np.float32)[0]
        assert float(f32) == v
    assert math.isnan(O.e8m0_value(255))


def test_dequant_matches_brute_force():
    assert check_dequant_vs_brute(O.dequant_mxfp4)


def test_dequant_nibble_layout_closed_form():
    # One row, one block: byte i = (code_hi << 4) | code_lo with chosen codes.
    qs = np.zeros((1, 16), np.uint8)
    qs[0, 0] = (7 << 4) | 1      # col 0 -> 0.5, col 16 -> 6
    qs[0, 5] = (10 << 4) | 3     # col 5 -> 1.5, col 21 -> -1
    qs[0, 15] = (0 << 4) | 15    # col 15 -> -6, col 31 -> 0
    sc = np.array([[128]], np.uint8)   # scale 2
    W = O.dequant_mxfp4(qs, sc)[0]
    expect = np.zeros(32)
    expect[0], expect[16] = 1.0, 12.0
    expect[5], expect[21] = 3.0, -2.0
    expect[15], expect[31] = -12.0, 0.0
    assert np.array_equal(W, expect)


def test_router_logits_match_loops():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, 7)).astype(np.float32)
    wr = rng.standard_normal((4, 7)).astype(np.float32)
    br = rng.standard_normal(4).astype(np.float32)
    got = O.router_logits(x, wr, br)
    for t in range(3):
        for e in range(4):
            ref = sum(float(x[t, i]) * float(wr[e, i]) for i in range(7)) + float(br[e])
            assert math.isclose(got[t, e], ref, rel_tol=1e-13, abs_tol=1e-13)


def test_topk_matches_brute_force():
    assert check_topk_vs_brute(O.topk_softmax)


def test_topk_invariants():
    rng = np.random.default_rng(6)
    logits = rng.standard_normal((200, 32)) * 5
    ids, w = O.topk_softmax(logits, 4)
    assert np.allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-15)
    assert np.all(np.diff(w, axis=1) <= 0)
    assert all(len(set(r)) == 4 for r in ids.tolist())
    # the chosen logits are the 4 largest
    assert np.allclose(np.sort(logits, axis=1)[:, ::-1][:, :4], np.take_along_axis(logits, ids, 1))


def test_topk_all_equal_k_equals_E():
    ids, w = O.topk_softmax(np.zeros((3, 5)), 5)
    assert np.array_equal(ids, np.tile(np.arange(5), (3, 1)))
    assert np.array_equal(w, np.full((3, 5), 0.2))


def test_bucket_matches_brute_force():
    assert check_bucket_vs_brute(O.bucket_csr)


@pytest.mark.parametrize("tile", [1, 4, 16, 128])
def test_bucket_invariants(tile):
    rng = np.random.default_rng(7)
    T, k, E = 300, 4, 32
    logits = rng.standard_normal((T, E))
    logits[:, :2] += 3.0  # skew
    ids, _ = O.topk_softmax(logits, k)
    b = O.bucket_csr(ids, E, tile)
    counts, basep, rows, inv = b["counts"], b["basep"], b["rows"], b["inv"]
    assert counts.sum() == T * k
    assert np.all(basep % tile == 0) and np.all(np.diff(basep) >= 0)
    assert basep[E] == sum(-(-c // tile) * tile for c in counts)
    live = rows[rows >= 0]
    # every token appears exactly k times
    assert np.array_equal(np.bincount(live // k, minlength=T), np.full(T, k))
    for e in range(E):
        seg = rows[basep[e]:basep[e + 1]]
        n = counts[e]
        assert np.all(seg[n:] == -1)
        assert np.all(np.diff(seg[:n]) > 0)
        assert np.all(ids.reshape(-1)[seg[:n]] == e)
    assert np.all(rows[basep[E]:] == -1)
    assert np.array_equal(rows[inv], np.arange(T * k))
    assert len(rows) == O.bucket_max_rows(T, k, E, tile)


def test_bucket_token_permutation():
    # Permuting the tokens permutes the bucket contents accordingly.
    rng = np.random.default_rng(8)
    T, k, E = 50, 3, 7
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)])
    perm = rng.permutation(T)
    a = O.bucket_csr(ids, E, 4)
    b = O.bucket_csr(ids[perm], E, 4)
    assert np.array_equal(a["counts"], b["counts"]) and np.array_equal(a["basep"], b["basep"])
    for e in range(E):
        s, n = a["basep"][e], a["counts"][e]
        ra = a["rows"][s:s + n]
        rb = b["rows"][s:s + n]
        mapped = sorted(perm[r // k] * k + r % k for r in rb)  # b's token i is a's token perm[i]
        assert list(ra) == mapped


def test_swiglu_closed_form_points():
    assert check_swiglu_points(O.swiglu_oai)


def test_sigmoid_extremes():
    s = O.sigmoid(np.array([-1000.0, -30.0, 0.0, 30.0, 1000.0]))
    assert not np.any(np.isnan(s))
    assert s[0] == 0.0 and s[2] == 0.5 and s[4] == 1.0
    assert math.isclose(s[1], math.exp(-30) / (1 + math.exp(-30)), rel_tol=1e-15)


def test_round_bf16_closed_form():
    cases = [
        (1.0, 1.0),
        (1.0 + 2.0 ** -8, 1.0),                        # halfway, ties to even (down)
        (1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -6),        # halfway, ties to even (up)
        (1.0 + 2.0 ** -8 + 2.0 ** -20, 1.0 + 2.0 ** -7),  # just above halfway
        (-(1.0 + 2.0 ** -8 + 2.0 ** -20), -(1.0 + 2.0 ** -7)),
        (3.0, 3.0),
        (2.0 ** -133, 2.0 ** -133),                    # smallest bf16 subnormal is kept
        (0.0, 0.0),
    ]
    for a, e in cases:
        assert O.round_bf16(np.array([a]))[0] == e, a
    assert math.isnan(O.round_bf16(np.array([float("nan")]))[0])
    # every float32 with zero low half is a fixed point
    rng = np.random.default_rng(9)
    bits = (rng.integers(0, 2 ** 16, size=1000, dtype=np.uint32) << 16).astype(np.uint32)
    v = bits.view(np.float32)
    v = v[np.isfinite(v)]
    assert np.array_equal(O.round_bf16(v), v.astype(np.float64))


def test_layer_matches_brute_force():
    assert check_layer_vs_brute(O.moe_layer)


def test_one_hot_routing_is_dense_ffn():
    # A router margin of 100 on one expert gives weight 1 (to float64 rounding)
    # on it; with k=1 the layer is exactly that expert's dense FFN.
    spec = spec_for(0)
    L = make_layer(spec, layer=1)
    E, D = spec.E, spec.D
    L = dict(L)
    L["w_router"] = np.zeros((E, D), np.float32)
    L["b_router"] = np.zeros(E, np.float32)
    L["b_router"][2] = 100.0
    x = L["x"][:3]
    y, ids, w, _ = O.moe_layer(L, x, 1)
    assert np.all(ids[:, 0] == 2) and np.all(w == 1.0)
    Wg = brute.dequant(L["g_qs"][2].tolist(), L["g_sc"][2].tolist())
    Wu = brute.dequant(L["u_qs"][2].tolist(), L["u_sc"][2].tolist())
    Wd = brute.dequant(L["d_qs"][2].tolist(), L["d_sc"][2].tolist())
    for t in range(3):
        xt = [float(v) for v in x[t]]
        g = brute.matvec(Wg, xt, L["bg"][2])
        u = brute.matvec(Wu, xt, L["bu"][2])
        h = [brute.swiglu(a, b) for a, b in zip(g, u)]
        o = brute.matvec(Wd, h, L["bd"][2])
        assert np.max(O.rownorm_rel_err(y[t], np.array(o), floor=1e-300)) < 1e-12
    # with k=2 the margin still puts weight ~1 on expert 2 (the other weight is e^-100)
    y2, ids2, w2, _ = O.moe_layer(L, x, 2)
    assert np.all(ids2[:, 0] == 2) and np.all(w2[:, 1] < 1e-40)
    assert np.max(O.rownorm_rel_err(y2, y, floor=1e-300)) < 1e-12


def test_identical_experts_give_dense_ffn_whatever_the_routing():
    spec = spec_for(0)
    L = dict(make_layer(spec, layer=2))
    for key in ["g_qs", "g_sc", "u_qs", "u_sc", "d_qs", "d_sc", "bg", "bu", "bd"]:
        L[key] = np.repeat(L[key][:1], spec.E, axis=0)
    y, ids, w, _ = O.moe_layer(L, L["x"], spec.k)
    assert len(set(ids.reshape(-1).tolist())) > 1  # routing really varies
    Wg = O.dequant_mxfp4(L["g_qs"][0], L["g_sc"][0])
    Wu = O.dequant_mxfp4(L["u_qs"][0], L["u_sc"][0])
    Wd = O.dequant_mxfp4(L["d_qs"][0], L["d_sc"][0])
    dense = O.expert_ffn(L["x"], Wg, L["bg"][0], Wu, L["bu"][0], Wd, L["bd"][0])
    assert np.max(O.rownorm_rel_err(y, dense, floor=1e-300)) < 1e-12


def test_bias_linearity():
    assert check_bias_linearity(O.moe_layer)


def test_gate_up_bias_enters_before_activation():
    # With zero gate/up weights, g = bg and u = bu exactly, so h = swiglu(bg, bu).
    spec = spec_for(0)
    L = dict(make_layer(spec, layer=4))
    L["g_qs"] = np.zeros_like(L["g_qs"])
    L["u_qs"] = np.zeros_like(L["u_qs"])
    L["bg"] = np.full_like(L["bg"], 0.75)
    L["bu"] = np.full_like(L["bu"], -0.25)
    y, ids, w, _ = O.moe_layer(L, L["x"], spec.k)
    h = O.swiglu_oai(np.full(spec.F, 0.75), np.full(spec.F, -0.25))
    for t in range(spec.T):
        exp = np.zeros(spec.D)
        for j in range(spec.k):
            e = ids[t, j]
            exp += w[t, j] * (O.dequant_mxfp4(L["d_qs"][e], L["d_sc"][e]) @ h + L["bd"][e])
        assert np.max(O.rownorm_rel_err(y[t], exp, floor=1e-300)) < 1e-12


def test_bf16_operand_variant_stays_close():
    # The bf16-operand reading of the prefill rail differs from the float64 layer by
    # bf16 rounding of x and h only: well inside the prefill tolerance 2e-2.
    spec = spec_for(0)
    L = make_layer(spec, layer=0)
    y64, _, _, _ = O.moe_layer(L, L["x"], spec.k)
    ybf, _, _, _ = O.moe_layer(L, L["x"], spec.k, operands="bf16")
    err = O.rownorm_rel_err(ybf, y64)
    assert np.all(err < 2e-2) and np.all(err > 0)


def test_bf16_split_operand_closed_form():
    # hi + lo reproduces x to 16 significant bits: exact for x with <= 16 bits,
    # and otherwise within 2^-16 relative.
    x = np.array([1.0 + 2.0 ** -12, -3.0 - 2.0 ** -15, 0.1, 12345.678], np.float32)
    hi = O.round_bf16(x)
    lo = O.round_bf16(x.astype(np.float64) - hi)
    assert hi[0] == 1.0 and lo[0] == 2.0 ** -12
    assert hi[1] + lo[1] == -3.0 - 2.0 ** -15
    rel = np.abs((hi + lo) - x.astype(np.float64)) / np.abs(x.astype(np.float64))
    assert np.all(rel <= 2.0 ** -16)


def test_bf16_operand_sensitivity_at_full_scale():
    """At the gpt-oss-shaped scale (E8M0 up to 135, D = 2880) |g| and |u| reach ~1e4,
    so rounding x alone to bf16 moves a few g, u across the swiglu clamp knees and
    the layer output by several percent; the split (hi + lo) operand stays far
    inside the 2e-2 prefill tolerance. Oracle against oracle, two tokens."""
    spec = spec_for(2)
    L = make_layer(spec, with_tokens=False)
    from synthetic import make_tokens
    x = make_tokens(spec, T=2, seed=3)
    cache = O.ExpertCache(L)
    y64, ids, w, _ = O.moe_layer(L, x, spec.k, cache=cache)
    ysplit, _, _, _ = O.moe_layer(L, x, spec.k, cache=cache, operands="bf16_split")
    ybf, _, _, _ = O.moe_layer(L, x, spec.k, cache=cache, operands="bf16")
    assert O.rownorm_rel_err(ysplit, y64).max() < 2e-3
    assert O.rownorm_rel_err(ybf, y64).max() > 2e-2


# ----------------------------------------------------------------------------
# E4M3 rounding and the E4M3-term operand of the block-scaled rail
# ----------------------------------------------------------------------------

def e4m3_code_values():
    """Every E4M3 code's value from the bit fields (NaN for the two NaN codes)."""
    vals = []
    for c in range(256):
        sign = -1.0 if c & 0x80 else 1.0
        e, m = (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            vals.append(float("nan"))
        elif e == 0:
            vals.append(sign * (m / 8.0) * 2.0 ** -6)
        else:
            vals.append(sign * (1 + m / 8.0) * 2.0 ** (e - 7))
    return vals


def brute_round_e4m3(v):
    """Nearest finite E4M3 value by exhaustive search; ties to the even code."""
    best, best_d, best_c = None, None, None
    for c, cv in enumerate(e4m3_code_values()):
        if cv != cv:
            continue
        if math.copysign(1.0, cv) != math.copysign(1.0, v) and cv == 0.0:
            continue  # keep the sign of zero
        d = abs(cv - v)
        if best is None or d < best_d or (d == best_d and (c & 1) == 0 and (best_c & 1) == 1):
            best, best_d, best_c = cv, d, c
    return best


def e4m3_probe_values():
    rng = np.random.default_rng(5)
    v = list(rng.normal(0, 3, 300)) + list(rng.normal(0, 200, 100)) + list(rng.normal(0, 0.01, 100))
    v += [0.0, -0.0, 448.0, 460.0, 464.0, 470.0, 1e9, -1e9, 1.0625, 1.1875, -2.5 * 2.0 ** -9,
          2.0 ** -10, 3 * 2.0 ** -10, 15 * 2.0 ** -10, 2.0 ** -6 - 2.0 ** -10, 240.0, 232.0]
    return [float(np.float32(x)) for x in v]


def check_round_e4m3(round_e4m3):
    vals = e4m3_probe_values()
    got = round_e4m3(np.array(vals))
    return all(g == brute_round_e4m3(v) and math.copysign(1, g) == math.copysign(1, brute_round_e4m3(v))
               for g, v in zip(got, vals))


def brute_split_e4m3_terms(block, nterms):
    """One block of 32 values, pure Python: per term the scale exponent from
    frexp (|max| / 2^s in [128, 256)), elements by exhaustive E4M3 search."""
    r = [float(np.float32(x)) for x in block]
    total = [0.0] * len(r)
    for _ in range(nterms):
        amax = max(abs(x) for x in r)
        if amax == 0.0:
            s = -127
        else:
            _, e = math.frexp(amax)  # amax = m * 2^e, m in [0.5, 1)
            s = max(e - 8, -127)
        for i in range(len(r)):
            t = brute_round_e4m3(r[i] / 2.0 ** s) * 2.0 ** s
            total[i] += t
            r[i] -= t
    return total


def check_split_vs_brute(split_e4m3_terms, seed=6):
    rng = np.random.default_rng(seed)
    for scale in (1.0, 1e-30, 3e4, 2.0 ** -120):
        blocks = (rng.normal(0, scale, (3, 32)) * rng.choice([1.0, 0.01, 1e-4], (3, 32))).astype(np.float32)
        blocks[2, 5:] = 0.0
        for n in (1, 2, 3):
            got = split_e4m3_terms(blocks, n)
            for b in range(3):
                if list(got[b]) != brute_split_e4m3_terms(blocks[b], n):
                    return False
    return True


def test_round_e4m3_matches_exhaustive_search():
    assert check_round_e4m3(O.round_e4m3)


def test_split_e4m3_terms_matches_brute_force():
    assert check_split_vs_brute(O.split_e4m3_terms)


def test_split_e4m3_terms_error_bound():
    # each term leaves at most 2^-4 of the block's largest residual: n terms
    # reproduce every block within 2^(-4n) of its largest magnitude
    rng = np.random.default_rng(8)
    x = (rng.normal(0, 1, (64, 64)) * np.exp(rng.normal(0, 3, (64, 1)))).astype(np.float32)
    blocks = x.astype(np.float64).reshape(64, 2, 32)
    amax = np.abs(blocks).max(axis=-1, keepdims=True)
    for n in (1, 2, 3, 4):
        err = np.abs(O.split_e4m3_terms(x, n).reshape(64, 2, 32) - blocks)
        assert np.all(err <= amax * 2.0 ** (-4 * n)), n
    assert np.array_equal(O.split_e4m3_terms(np.zeros((2, 32), np.float32), 3), np.zeros((2, 32)))


def test_e4m3_term_operands_at_full_scale():
    """The block-scaled rail's operands (x in three E4M3 terms, h in two) keep the
    gpt-oss-shaped layer well inside the 2e-2 prefill tolerance. Oracle against
    oracle, two tokens."""
    spec = spec_for(2)
    L = make_layer(spec, with_tokens=False)
    from synthetic import make_tokens
    x = make_tokens(spec, T=2, seed=3)
    cache = O.ExpertCache(L)
    y64, _, _, _ = O.moe_layer(L, x, spec.k, cache=cache)
    ye4, _, _, _ = O.moe_layer(L, x, spec.k, cache=cache, operands="e4m3_terms")
    err = O.rownorm_rel_err(ye4, y64)
    assert np.all(err < 1e-2) and np.all(err > 0)


def test_routing_margins_closed_form():
    assert check_routing_margins(O.routing_margins)


def test_rownorm_rel_err_closed_form():
    assert check_rownorm_rel_err(O.rownorm_rel_err)


def test_bucket_max_rows_hand_values_and_bound():
    assert check_bucket_max_rows(O.bucket_max_rows)


def test_decode_terms_layer_reduces_to_the_layer():
    assert check_decode_terms_layer(O.moe_layer_decode_terms)


def test_round_e2m1_matches_exhaustive_search():
    assert check_round_e2m1(O.round_e2m1)
    # every E2M1 value is a fixed point
    vals = np.array(e2m1_magnitudes() + [-m for m in e2m1_magnitudes()[1:]])
    assert np.array_equal(O.round_e2m1(vals), vals)


def test_split_e2m1_terms_matches_brute_force():
    assert check_split_e2m1_vs_brute(O.split_e2m1_terms)


def test_split_e2m1_terms_converges():
    # 13 terms hold every bit of a float32 block (each term takes >= 2 bits of the
    # residual's leading value); fewer terms stay within their own residual bound
    x = np.random.default_rng(3).standard_normal((16, 256)).astype(np.float32)
    assert np.array_equal(O.split_e2m1_terms(x, 13), x.astype(np.float64))
    for n in (2, 4, 8):
        err = np.abs(O.split_e2m1_terms(x, n) - x).reshape(16, 8, 32).max(-1)
        amax = np.abs(x).reshape(16, 8, 32).max(-1)
        assert np.all(err <= amax * 3.0 ** -n), n


def test_decode_terms_layer_in_both_formats():
    spec = spec_for(0)
    L = make_layer(spec, layer=6)
    y_ref, _, _, _ = O.moe_layer(L, L["x"], spec.k)
    for fmt, n in (("e2m1", 8), ("e4m3", 5)):
        y, _, _, _ = O.moe_layer_decode_terms(L, L["x"], spec.k, x_terms=n, h_terms=n, fmt=fmt)
        assert np.max(O.rownorm_rel_err(y, y_ref)) < 1e-5, fmt


def test_rms_renorm_closed_forms():
    # [3, 4]: mean square 12.5; a constant row becomes its sign; every nonzero
    # row ends with mean square 1; a zero row stays zero; rows are independent.
    y = O.rms_renorm(np.array([[3.0, 4.0], [-2.0, -2.0], [0.0, 0.0]]))
    assert np.allclose(y[0], [3 / math.sqrt(12.5), 4 / math.sqrt(12.5)], rtol=0, atol=1e-15)
    assert np.array_equal(y[1], [-1.0, -1.0])
    assert np.array_equal(y[2], [0.0, 0.0])
    rng = np.random.default_rng(5)
    z = rng.standard_normal((4, 2880)) * np.array([[1e-3], [1.0], [7.0], [1e4]])
    r = O.rms_renorm(z)
    assert np.allclose(np.mean(r * r, axis=1), 1.0, rtol=1e-12)
    assert np.allclose(r * np.sqrt(np.mean(z * z, axis=1, keepdims=True)), z, rtol=1e-12)


# ---------------------------------------------------------------------------
# Q8 activations and the MXFP4 x Q8 integer dot
# ---------------------------------------------------------------------------
def check_quantize_q8(fn) -> bool:
    """Closed forms of the 32-block requant: scale = block max / 127, codes
    rounded to nearest with ties to even, zero blocks zero, scaling by a power
    of two moves only the scale, and every code reconstructs within half a step."""
    v = np.zeros((2, 64), np.float32)
    v[0, :4] = [127.0, -63.5, 0.5, 1.5]  # scale 1: ties go to even codes
    v[0, 32:35] = [-254.0, 127.0, 3.0]   # scale 2
    q, d = fn(v)
    ok = q.dtype == np.int8 and d.dtype == np.float32 and q.shape == (2, 64) and d.shape == (2, 2)
    ok &= list(q[0, :4]) == [127, -64, 0, 2] and d[0, 0] == 1.0
    ok &= list(q[0, 32:35]) == [-127, 64, 2] and d[0, 1] == 2.0  # 1.5 -> 2 (tie to even)
    ok &= not q[1].any() and not d[1].any()  # all-zero blocks
    rng = np.random.default_rng(17)
    x = (rng.standard_normal((5, 2880)) * rng.uniform(1e-3, 1e3, (5, 1))).astype(np.float32)
    q1, d1 = fn(x)
    q2, d2 = fn((x * np.float32(2.0 ** -9)).astype(np.float32))
    ok &= np.array_equal(q1, q2) and np.array_equal(d2, (d1 * np.float32(2.0 ** -9)).astype(np.float32))
    blk_max = np.abs(q1.reshape(5, 90, 32)).max(axis=2)
    ok &= bool(np.all(blk_max == 127))  # the largest element of a block takes the full code
    rec = q1.reshape(5, 90, 32).astype(np.float64) * d1[..., None].astype(np.float64)
    ok &= bool(np.all(np.abs(rec - x.reshape(5, 90, 32)) <= 0.5 * d1[..., None] * (1 + 1e-5) + 1e-30))
    return bool(ok)


def check_q8_block_dots(fn) -> bool:
    """Brute force on small matrices: element by element, the stored byte
    order of a block (column j low nibble, column 16+j high) and integer sums."""
    rng = np.random.default_rng(23)
    R, C = 3, 96
    qs = rng.integers(0, 256, (R, C // 2), dtype=np.uint8)
    q = rng.integers(-127, 128, C).astype(np.int8)
    got = fn(qs, q)
    ok = got.shape == (R, C // 32)
    for r in range(R):
        for b in range(C // 32):
            s = 0
            for j in range(32):
                byte = int(qs[r, 16 * b + (j % 16)])
                code = byte & 15 if j < 16 else byte >> 4
                s += int(round(2 * O.e2m1_value(code))) * int(q[32 * b + j])
            ok &= int(got[r, b]) == s
    return bool(ok)


def check_gemv_q8(fn) -> bool:
    """The float32 result against the exact float64 sum of the block products
    (within the rounding of 90 float32 additions), and the one-block case,
    where the order leaves a single rounding: out = fl(fl(isum * factor) + bias)."""
    rng = np.random.default_rng(29)
    R, C = 5, 2880
    qs = rng.integers(0, 256, (R, C // 2), dtype=np.uint8)
    sc = rng.integers(118, 136, (R, C // 32), dtype=np.uint8)
    x = rng.standard_normal(C).astype(np.float32)
    q, d = O.quantize_q8(x)
    bias = rng.standard_normal(R).astype(np.float32)
    got = fn(qs, sc, q, d, bias)
    isum = O.mxfp4_q8_block_dots(qs, q).astype(np.float64)
    fac = d.astype(np.float64)[None, :] * np.ldexp(1.0, sc.astype(np.int64) - 128)
    exact = (isum * fac).sum(axis=1) + bias
    scale = np.abs(isum * fac).sum(axis=1) + np.abs(bias)
    ok = got.dtype == np.float32 and bool(np.all(np.abs(got - exact) <= 2e-6 * scale))
    q1 = np.zeros(C, np.int8)
    q1[32:64] = q[32:64]  # only block 1 (lane 1) is live
    d1 = d.copy()
    one = fn(qs, sc, q1, d1, bias)
    i1 = O.mxfp4_q8_block_dots(qs, q1)[:, 1].astype(np.float32)
    f1 = (d1[1] * np.ldexp(np.float32(1.0), sc[:, 1].astype(np.int64) - 128)).astype(np.float32)
    ok &= np.array_equal(one, ((i1 * f1).astype(np.float32) + bias).astype(np.float32))
    # a sign flip of all codes flips the result without the bias exactly (no order effect)
    neg = fn(qs, sc, (-q.astype(np.int16)).astype(np.int8), d, None)
    pos = fn(qs, sc, q, d, None)
    ok &= np.array_equal(neg, -pos)
    return bool(ok)


def test_quantize_q8_closed_forms():
    assert check_quantize_q8(O.quantize_q8)


def test_q8_block_dots_brute_force():
    assert check_q8_block_dots(O.mxfp4_q8_block_dots)


def test_gemv_q8_exact_sum_and_single_block():
    assert check_gemv_q8(O.mxfp4_gemv_q8)


def test_q8_operands_of_the_layer_reduce_to_requantised_inputs():
    # the q8 operand model is the layer evaluated on requantised x and h: with
    # activations already on the Q8 grid (codes times a power-of-two scale),
    # the requant of x is exact and gate/up equal the float64 projections
    spec = spec_for(0)
    L = make_layer(spec, with_tokens=False)
    rng = np.random.default_rng(31)
    codes = rng.integers(-127, 128, (1, spec.D)).astype(np.float32)
    codes[:, ::32] = 127  # every block reaches the full code
    x = (codes * np.float32(2.0 ** -5)).astype(np.float32)
    qx, dx = O.quantize_q8(x)
    assert np.array_equal(O.dequant_q8(qx, dx), x.astype(np.float64))
