"""Plain, slow, float64 oracle of the gpt-oss-style routed MoE expert chain.

TEST INFRASTRUCTURE ONLY. Nothing in the library imports this module; only
the tests, the smoke check and the benchmark's CPU-baseline leg do.

What it computes, and where each step is defined:

* MXFP4 weights: 32-element blocks of E2M1 codes sharing one E8M0 exponent
  byte ("dasLLAMA: dig the last two board reds green", section "gpt-oss: mx4
  kernels to the lab-winning shape": the 16-value E2M1 table and the E8M0
  exponent decode). A value is E2M1[q] * 2**(s - 127). Inside a block, byte i
  holds element i in its low nibble and element i + 16 in its high nibble
  (the low/high nibble split of the mx4 dot in "dasLLAMA gpt-oss arc", commit
  "dot_mx4q8_template rewritten in plain das").
* Router: logits over the E experts, the top k taken (descending logit,
  lower expert index first on equal logits), then a softmax over the k taken.
* Bucket: a CSR of the T*k (token, slot) assignments grouped by expert, each
  expert's row range padded to a tile height, with the padded prefix
  ``basep`` ("dasLLAMA gpt-oss arc", Metal fusion lane commit, third bullet:
  the prefix folded into MetalMoeBucket, bit-identical CSR).
* Expert FFN: gate and up projections with bias (the bias seeds the
  accumulator in the pages' kernels, Metal fusion lane commit, first bullet;
  here it is simply added), swiglu_oai, down projection with bias.
* Combine: the router-weighted sum over the k slots, in slot order
  ("dasLLAMA gpt-oss arc", fused MoE expert chain commit: stage 1 sums the
  experts' down rows "in slot order").

Where the pages are silent the oracle takes the plainest reading; the readings
that change arithmetic are noted beside the function that takes them.

Every function here is pinned by a test in tests/test_oracle_pins.py against
something other than itself (the printed E2M1 table, math.ldexp, brute force
in oracle/brute.py, closed forms and invariants).
"""

from __future__ import annotations

import math
from typing import Dict, Optional, Tuple

import numpy as np

SWIGLU_ALPHA = 1.702
SWIGLU_LIMIT = 7.0


# ----------------------------------------------------------------------------
# MXFP4 element and scale decoding
# ----------------------------------------------------------------------------

def e2m1_value(code: int) -> float:
    """Value of a 4-bit E2M1 code: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit.

    Exponent field 0 is subnormal (m * 0.5). Code 8 is negative zero.
    """
    code = int(code) & 0xF
    sign = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        mag = 0.5 * m
    else:
        mag = 2.0 ** (e - 1) * (1.0 + 0.5 * m)
    return sign * mag


E2M1_LUT = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)


def e8m0_value(s: int) -> float:
    """Value of an E8M0 scale byte: 2**(s - 127); byte 255 is NaN."""
    s = int(s)
    if s == 255:
        return float("nan")
    return math.ldexp(1.0, s - 127)


E8M0_LUT = np.array([e8m0_value(s) for s in range(256)], dtype=np.float64)


def dequant_mxfp4(qs: np.ndarray, sc: np.ndarray) -> np.ndarray:
    """Dequantise an MXFP4 matrix stored as planes qs [R, C/2] and sc [R, C/32] to float64 [R, C]."""
    qs = np.asarray(qs, dtype=np.uint8)
    sc = np.asarray(sc, dtype=np.uint8)
    R, half = qs.shape
    C = half * 2
    nb = C // 32
    assert sc.shape == (R, nb)
    blocks = qs.reshape(R, nb, 16)
    low = E2M1_LUT[blocks & 0x0F]          # block elements 0..15
    high = E2M1_LUT[blocks >> 4]           # block elements 16..31
    vals = np.concatenate([low, high], axis=2)  # [R, nb, 32]
    vals = vals * E8M0_LUT[sc][:, :, None]
    return vals.reshape(R, C)


# ----------------------------------------------------------------------------
# Router: logits, top-k, softmax over the selected k
# ----------------------------------------------------------------------------

def router_logits(x: np.ndarray, w_router: np.ndarray, b_router: Optional[np.ndarray]) -> np.ndarray:
    """l[t, e] = sum_i x[t, i] * Wr[e, i] + br[e], in float64 from the float32 inputs."""
    l = np.asarray(x, np.float64) @ np.asarray(w_router, np.float64).T
    if b_router is not None:
        l = l + np.asarray(b_router, np.float64)[None, :]
    return l


def topk_softmax(logits: np.ndarray, k: int) -> Tuple[np.ndarray, np.ndarray]:
    """Top-k experts per token (descending logit, lower index first on ties), then softmax over them.

    Returns ids int32 [T, k] in slot order and weights float64 [T, k].
    """
    logits = np.asarray(logits, np.float64)
    T, E = logits.shape
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-logits[t, e], e))[:k]
        ids[t] = order
        sel = logits[t, order]
        ex = np.exp(sel - sel[0])  # sel[0] is the largest
        w[t] = ex / ex.sum()
    return ids, w


# ----------------------------------------------------------------------------
# Bucket: CSR grouped by expert with a tile-padded prefix
# ----------------------------------------------------------------------------

def bucket_max_rows(T: int, k: int, E: int, tile: int) -> int:
    """Worst-case padded row count T*k + E*(tile-1), rounded up to a whole tile."""
    n = T * k + E * (tile - 1)
    return ((n + tile - 1) // tile) * tile


def bucket_csr(ids: np.ndarray, E: int, tile: int) -> Dict[str, np.ndarray]:
    """CSR of the (token, slot) assignments grouped by expert.

    counts[e]      number of assignments to expert e
    basep[e]       padded prefix: sum over e' < e of ceil(counts[e']/tile)*tile; basep[E] = mpad
    rows[p]        for p in [basep[e], basep[e] + counts[e]): the assignment index t*k + j,
                   in ascending order; -1 for pad rows and for every p >= mpad
    inv[t*k + j]   the row position p of that assignment (-1 if its id is out of range)
    """
    ids = np.asarray(ids, dtype=np.int64)
    T, k = ids.shape
    flat = ids.reshape(-1)
    counts = np.zeros(E, dtype=np.int32)
    for a in range(T * k):
        e = flat[a]
        if 0 <= e < E:
            counts[e] += 1
    basep = np.zeros(E + 1, dtype=np.int32)
    for e in range(E):
        basep[e + 1] = basep[e] + ((counts[e] + tile - 1) // tile) * tile
    rows = np.full(bucket_max_rows(T, k, E, tile), -1, dtype=np.int32)
    inv = np.full(T * k, -1, dtype=np.int32)
    fill = np.zeros(E, dtype=np.int64)
    for a in range(T * k):
        e = flat[a]
        if 0 <= e < E:
            p = basep[e] + fill[e]
            rows[p] = a
            inv[a] = p
            fill[e] += 1
    return dict(counts=counts, basep=basep, rows=rows, inv=inv)


# ----------------------------------------------------------------------------
# Activation
# ----------------------------------------------------------------------------

def sigmoid(z: np.ndarray) -> np.ndarray:
    """Logistic function evaluated without overflow: 1/(1+e^-z) for z >= 0, e^z/(1+e^z) otherwise."""
    z = np.asarray(z, np.float64)
    out = np.empty_like(z)
    pos = z >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-z[pos]))
    ez = np.exp(z[~pos])
    out[~pos] = ez / (1.0 + ez)
    return out


def swiglu_oai(g: np.ndarray, u: np.ndarray, alpha: float = SWIGLU_ALPHA,
               limit: float = SWIGLU_LIMIT) -> np.ndarray:
    """min(g, limit) * sigmoid(alpha * min(g, limit)) * (clamp(u, -limit, limit) + 1)."""
    g = np.minimum(np.asarray(g, np.float64), limit)
    u = np.clip(np.asarray(u, np.float64), -limit, limit)
    return g * sigmoid(alpha * g) * (u + 1.0)


# ----------------------------------------------------------------------------
# bfloat16 rounding (operand precision of the prefill rail's tensor-core MMAs)
# ----------------------------------------------------------------------------

def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round to the nearest bfloat16 (ties to even), returned as float64.

    The value is first taken to float32 (the operands arrive as float32 in
    this layer), then its low 16 bits are rounded away.
    """
    f = np.asarray(a, dtype=np.float32)
    bits = f.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    rounded = (bits + 0x7FFF + lsb) & 0xFFFF0000
    nan = np.isnan(f)
    out = rounded.astype(np.uint32).view(np.float32).astype(np.float64)
    out[nan] = np.nan
    return out


E4M3_MAX = 448.0


def round_e4m3(a: np.ndarray) -> np.ndarray:
    """Round to the nearest E4M3 value, ties to the even mantissa, saturating at +-448.

    E4M3 (OCP 8-bit float): sign, 4 exponent bits with bias 7, 3 mantissa bits.
    Normal values are (1 + m/8) * 2^(e-7) for e = 1..15 (e = 15, m = 7 is NaN, so
    the largest finite value is 448); subnormals are (m/8) * 2^-6. So a magnitude
    in [2^k, 2^(k+1)) (k >= -6) is rounded to a multiple of 2^(k-3), and anything
    below 2^-6 to a multiple of 2^-9.
    """
    a = np.asarray(a, np.float64)
    mag = np.abs(a)
    k = np.floor(np.log2(np.where(mag > 0, mag, 1.0)))
    quantum = 2.0 ** (np.maximum(k, -6.0) - 3.0)
    r = np.minimum(np.round(mag / quantum) * quantum, E4M3_MAX)  # np.round: half to even
    return np.copysign(r, a)


def split_e4m3_terms(v: np.ndarray, nterms: int) -> np.ndarray:
    """The operand the block-scaled prefill rail multiplies instead of v.

    A reading of the prefill operand precision for the block-scaled rail (the
    pages fix no 8-bit activation operand): along the last axis every block of
    32 values is carried as a sum of nterms E4M3 blocks. Term t takes the
    residual r of the terms before it (r = v for the first), gets the power of
    two 2^s with s = floor(log2 max|r|) - 7 (bounded below by E8M0's -127), so
    that the block's largest |r| / 2^s lies in [128, 256), and is
    2^s * round_e4m3(r / 2^s). The values are taken as float32 first (the
    layer's activations are float32). Returns the sum of the terms.
    """
    v = np.asarray(v, np.float32).astype(np.float64)
    shape = v.shape
    assert shape[-1] % 32 == 0
    r = v.reshape(shape[:-1] + (shape[-1] // 32, 32))
    total = np.zeros_like(r)
    for _ in range(nterms):
        amax = np.max(np.abs(r), axis=-1, keepdims=True)
        s = np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 7.0
        s = np.maximum(s, -127.0)
        term = round_e4m3(r / 2.0 ** s) * 2.0 ** s
        total = total + term
        r = r - term
    return total.reshape(shape)


E2M1_MAX = 6.0


def round_e2m1(a: np.ndarray) -> np.ndarray:
    """Round to the nearest E2M1 value, ties to the even code (mantissa bit 0), saturating at +-6.

    The E2M1 magnitudes are {0, 0.5, 1, 1.5, 2, 3, 4, 6} (the table of the
    pages' MXFP4 format): a multiple of 0.5 below 2, of 1 in [2, 4) and of 2 in
    [4, 6]. Codes with an even mantissa are 0, 1, 2, 4 (and 6 has an odd one),
    so a tie between two neighbours goes to 0, 1, 2 or 4.
    """
    a = np.asarray(a, np.float64)
    mag = np.abs(a)
    q = np.where(mag < 2.0, 0.5, np.where(mag < 4.0, 1.0, 2.0))
    lo = np.floor(mag / q) * q
    hi = lo + q
    frac = mag - lo
    # lo's code is even when lo is 0, 1, 2 or 4 (0.5, 1.5, 3 and 6 are odd)
    lo_even = np.isin(lo, (0.0, 1.0, 2.0, 4.0))
    up = (frac > q / 2) | ((frac == q / 2) & ~lo_even)
    r = np.minimum(np.where(up, hi, lo), E2M1_MAX)
    return np.copysign(r, a)


def split_e2m1_terms(v: np.ndarray, nterms: int) -> np.ndarray:
    """The activation operand of the block-scaled decode rail: each block of 32
    values along the last axis as a sum of nterms E2M1 blocks.

    A reading of the decode precision for that rail (the pages' decode GEMV
    multiplies float activations; an activation operand in the MXFP4 element
    format is not on the pages). Term t takes the residual r of the terms
    before it (r = v for the first), gets the power of two 2^e with the
    smallest e such that the block's largest |r| / 2^e <= 6 (bounded to
    E8M0's range [-127, 127]), and is 2^e * round_e2m1(r / 2^e). The values
    are taken as float32 first. Returns the sum of the terms.
    """
    v = np.asarray(v, np.float32).astype(np.float64)
    shape = v.shape
    assert shape[-1] % 32 == 0
    r = v.reshape(shape[:-1] + (shape[-1] // 32, 32))
    total = np.zeros_like(r)
    for _ in range(nterms):
        amax = np.max(np.abs(r), axis=-1, keepdims=True)
        e = np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 2.0
        e = np.where(amax > E2M1_MAX * 2.0 ** e, e + 1.0, e)
        e = np.clip(e, -127.0, 127.0)
        term = round_e2m1(r / 2.0 ** e) * 2.0 ** e
        total = total + term
        r = r - term
    return total.reshape(shape)


# ----------------------------------------------------------------------------
# Projections and the expert FFN
# ----------------------------------------------------------------------------

# ----------------------------------------------------------------------------
# Q8 activations and the MXFP4 x Q8 integer dot ("dasLLAMA gpt-oss arc": the
# dot_mx4q8 template takes a weight block's nibbles through a table lookup, the
# low nibble by masking with 15 and the high one by a shift of 4, and
# accumulates integer dot products of four lanes; the fused MoE expert chain
# commit requantises the activations of its first stage in blocks of 32)
# ----------------------------------------------------------------------------
# The E2M1 table doubled: every entry becomes an integer in [-12, 12], so a
# block's products with int8 activations add up exactly in integers.
E2M1_X2 = np.array([int(round(2.0 * e2m1_value(c))) for c in range(16)], dtype=np.int64)


def quantize_q8(v: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Blocks of 32 values as int8 codes and one float32 scale per block.

    Reading (the pages name a 32-block requant and the Q8 format, not its
    arithmetic): the scale is d = amax / 127 of the block's largest magnitude
    and each code q = round(v * (127 / amax)), nearest with ties to even,
    every step in float32; an all-zero block has d = 0 and q = 0. Returns
    (q int8 [..., C], d float32 [..., C/32]).
    """
    v = np.asarray(v, dtype=np.float32)
    C = v.shape[-1]
    assert C % 32 == 0
    blk = v.reshape(v.shape[:-1] + (C // 32, 32))
    amax = np.max(np.abs(blk), axis=-1)
    live = amax > 0
    safe = np.where(live, amax, np.float32(1.0)).astype(np.float32)
    inv = (np.float32(127.0) / safe).astype(np.float32)
    q = np.rint((blk * inv[..., None]).astype(np.float32))
    q = np.where(live[..., None], q, 0.0).astype(np.int8)
    d = np.where(live, (safe / np.float32(127.0)).astype(np.float32), np.float32(0.0)).astype(np.float32)
    return q.reshape(v.shape), d


def dequant_q8(q: np.ndarray, d: np.ndarray) -> np.ndarray:
    """The values that Q8 codes stand for, float64: q * d per block of 32."""
    q = np.asarray(q, np.float64)
    C = q.shape[-1]
    blk = q.reshape(q.shape[:-1] + (C // 32, 32))
    return (blk * np.asarray(d, np.float64)[..., None]).reshape(q.shape)


def mxfp4_q8_block_dots(qs: np.ndarray, q: np.ndarray) -> np.ndarray:
    """Integer dot of every 32-block of an MXFP4 matrix's rows with int8 codes:
    isum[r, b] = sum_i E2M1_X2[code of column 32b+i of row r] * q[32b+i]
    (byte j of a block: column j in the low nibble, column 16+j in the high).
    qs [R, C/2] uint8, q [C] int8; returns int64 [R, C/32]."""
    qs = np.asarray(qs, dtype=np.uint8)
    R, half = qs.shape
    nb = half // 16
    blocks = qs.reshape(R, nb, 16)
    w = np.concatenate([E2M1_X2[blocks & 0x0F], E2M1_X2[blocks >> 4]], axis=2)  # [R, nb, 32]
    return np.einsum("rbi,bi->rb", w, np.asarray(q, np.int64).reshape(nb, 32))


def q8_block_scales(sc: np.ndarray, d: np.ndarray) -> np.ndarray:
    """Per (row, block) float32 factor d_b * 2**(s - 128): the activation
    block scale times the weight block's E8M0 scale, halved for the doubled
    table (E8M0 byte 255, NaN, stays NaN)."""
    sc = np.asarray(sc, dtype=np.int64)
    w = np.where(sc == 255, np.nan, np.ldexp(1.0, sc - 128)).astype(np.float32)
    return (np.asarray(d, np.float32)[None, :] * w).astype(np.float32)


def mxfp4_gemv_q8(qs: np.ndarray, sc: np.ndarray, q: np.ndarray, d: np.ndarray,
                  bias: Optional[np.ndarray]) -> np.ndarray:
    """out[r] = sum_b isum[r, b] * d_b * 2**(s[r, b] - 128) + bias[r], float32.

    The float32 additions follow a fixed order (so that the result is a
    function of the inputs alone, and a GPU warp can reproduce it exactly):
    lane l of 32 adds the products of blocks l, l+32, l+64, ... in ascending
    order, each product float32(isum) * factor rounded to float32; the 32
    lane sums then meet in a butterfly over lane distances 16, 8, 4, 2, 1
    (each lane adds its partner's sum), and the bias is added last."""
    isum = mxfp4_q8_block_dots(qs, q).astype(np.float32)  # |isum| <= 12*127*32: exact
    fac = q8_block_scales(sc, d)
    R, nb = isum.shape
    lanes = np.zeros((R, 32), dtype=np.float32)
    for b in range(nb):
        prod = (isum[:, b] * fac[:, b]).astype(np.float32)
        lanes[:, b % 32] = (lanes[:, b % 32] + prod).astype(np.float32)
    idx = np.arange(32)
    for m in (16, 8, 4, 2, 1):
        lanes = (lanes + lanes[:, idx ^ m]).astype(np.float32)
    out = lanes[:, 0]
    if bias is not None:
        out = (out + np.asarray(bias, np.float32)).astype(np.float32)
    return out


def mxfp4_gemv(qs: np.ndarray, sc: np.ndarray, x: np.ndarray, bias: Optional[np.ndarray]) -> np.ndarray:
    """out = W x + bias for one MXFP4 matrix W [R, C] and vector(s) x [..., C]."""
    W = dequant_mxfp4(qs, sc)
    out = np.asarray(x, np.float64) @ W.T
    if bias is not None:
        out = out + np.asarray(bias, np.float64)
    return out


def expert_ffn(x_rows: np.ndarray, Wg: np.ndarray, bg, Wu: np.ndarray, bu, Wd: np.ndarray, bd,
               operands: str = "f64") -> np.ndarray:
    """One expert on a batch of token rows, with dequantised float64 weights.

    g = Wg x + bg, u = Wu x + bu, h = swiglu_oai(g, u), o = Wd h + bd.
    operands selects the precision of the projections' activation operands
    (the weights are exact in bfloat16 already):
      "f64"        float64 throughout (the layer's definition);
      "bf16"       x and h rounded to bfloat16 (bf16 tensor-core operands);
      "bf16_split" x carried as two bfloat16 parts, hi = bf16(x) and
                   lo = bf16(x - hi), so the gate/up operand is hi + lo;
                   h rounded to bfloat16;
      "e4m3_terms" the block-scaled rail's operands: x as three E4M3 terms
                   and h as two (split_e4m3_terms);
      "q8"         the q8 rail's operands: x and h (rounded to float32)
                   requantised in blocks of 32 (quantize_q8), exact products.
      "e2m1_terms" the prefill rail on prepacked planes: x as six E2M1 terms
                   and h as four (split_e2m1_terms), exact products.
    """
    x = np.asarray(x_rows, np.float64)
    if operands == "bf16":
        x = round_bf16(x)
    elif operands == "bf16_split":
        hi = round_bf16(x)
        x = hi + round_bf16(np.asarray(x, np.float64) - hi)
    elif operands == "e4m3_terms":
        x = split_e4m3_terms(x, 3)
    elif operands == "q8":
        x = dequant_q8(*quantize_q8(x))
    elif operands == "e2m1_terms":
        x = split_e2m1_terms(x, 6)
    elif operands != "f64":
        raise ValueError(operands)
    g = x @ Wg.T + (0.0 if bg is None else np.asarray(bg, np.float64))
    u = x @ Wu.T + (0.0 if bu is None else np.asarray(bu, np.float64))
    h = swiglu_oai(g, u)
    if operands in ("bf16", "bf16_split"):
        h = round_bf16(h)
    elif operands == "e4m3_terms":
        h = split_e4m3_terms(h, 2)
    elif operands == "q8":
        h = dequant_q8(*quantize_q8(h.astype(np.float32)))
    elif operands == "e2m1_terms":
        h = split_e2m1_terms(h, 4)
    return h @ Wd.T + (0.0 if bd is None else np.asarray(bd, np.float64))


class ExpertCache:
    """Dequantises each expert's three matrices on first use (float64)."""

    def __init__(self, layer: Dict[str, np.ndarray]):
        self.layer = layer
        self._cache: Dict[int, Tuple[np.ndarray, np.ndarray, np.ndarray]] = {}

    def __call__(self, e: int):
        if e not in self._cache:
            L = self.layer
            self._cache[e] = (dequant_mxfp4(L["g_qs"][e], L["g_sc"][e]),
                              dequant_mxfp4(L["u_qs"][e], L["u_sc"][e]),
                              dequant_mxfp4(L["d_qs"][e], L["d_sc"][e]))
        return self._cache[e]


def moe_layer(layer: Dict[str, np.ndarray], x: np.ndarray, k: int, token_idx=None,
              operands: str = "f64", ids: Optional[np.ndarray] = None,
              weights: Optional[np.ndarray] = None, cache: Optional[ExpertCache] = None):
    """The full layer for the tokens in ``token_idx`` (all tokens by default).

    Returns (y [n, D] float64, ids [T, k], weights [T, k], logits [T, E]).
    ``ids``/``weights`` may be given to evaluate the experts under a fixed
    routing (used when a near-tie makes the routing ambiguous).
    """
    x = np.asarray(x, np.float32)
    T = x.shape[0]
    logits = router_logits(x, layer["w_router"], layer.get("b_router"))
    if ids is None:
        ids, weights = topk_softmax(logits, k)
    if token_idx is None:
        token_idx = np.arange(T)
    cache = cache or ExpertCache(layer)
    D = layer["d_qs"].shape[1]
    y = np.zeros((len(token_idx), D), dtype=np.float64)
    for n, t in enumerate(token_idx):
        for j in range(k):  # slot order
            e = int(ids[t, j])
            Wg, Wu, Wd = cache(e)
            o = expert_ffn(x[t:t + 1], Wg, layer["bg"][e], Wu, layer["bu"][e], Wd, layer["bd"][e],
                           operands=operands)[0]
            y[n] += float(weights[t, j]) * o
    return y, ids, weights, logits


def moe_layer_decode_terms(layer: Dict[str, np.ndarray], x: np.ndarray, k: int, x_terms: int = 8,
                           h_terms: int = 8, token_idx=None, cache: Optional[ExpertCache] = None,
                           fmt: str = "e2m1"):
    """The operands of the block-scaled decode rail, evaluated in float64.

    A reading of the decode precision for that rail (the pages' decode GEMV
    multiplies float activations; a low-precision tensor-core operand is not
    on the pages): x enters gate/up as x_terms terms (fmt "e2m1":
    split_e2m1_terms, the MXFP4 element format; "e4m3": split_e4m3_terms), and
    the router weight is folded into the down operand, which is w_j * h_j
    carried as h_terms terms of the same format, so that
        y[t] = sum_j ( Wd[e_j] . split(w_j * h_j) + w_j * bd[e_j] )
    with h_j = swiglu_oai(Wg[e_j] . split(x_t) + bg, Wu[e_j] . split(x_t) + bu).
    Without the splitting this is the layer itself (the weight distributes over
    the down projection). Returns (y [n, D], ids, weights, h [n, k, F]).
    """
    x = np.asarray(x, np.float32)
    T = x.shape[0]
    logits = router_logits(x, layer["w_router"], layer.get("b_router"))
    ids, weights = topk_softmax(logits, k)
    if token_idx is None:
        token_idx = np.arange(T)
    cache = cache or ExpertCache(layer)
    D = layer["d_qs"].shape[1]
    F = layer["g_qs"].shape[1]
    y = np.zeros((len(token_idx), D), dtype=np.float64)
    hs = np.zeros((len(token_idx), k, F), dtype=np.float64)
    split = {"e2m1": split_e2m1_terms, "e4m3": split_e4m3_terms}[fmt]
    for n, t in enumerate(token_idx):
        xt = split(x[t:t + 1].astype(np.float64), x_terms)
        for j in range(k):  # slot order
            e = int(ids[t, j])
            Wg, Wu, Wd = cache(e)
            g = xt @ Wg.T + np.asarray(layer["bg"][e], np.float64)
            u = xt @ Wu.T + np.asarray(layer["bu"][e], np.float64)
            h = swiglu_oai(g, u)
            hs[n, j] = h[0]
            hw = split(float(weights[t, j]) * h, h_terms)
            y[n] += (hw @ Wd.T)[0] + float(weights[t, j]) * np.asarray(layer["bd"][e], np.float64)
    return y, ids, weights, hs


# ----------------------------------------------------------------------------
# Comparison helpers used by the tests
# ----------------------------------------------------------------------------

def rms_renorm(y: np.ndarray) -> np.ndarray:
    """Each row divided by its root mean square, in float64 (a zero row stays
    zero): the renormalisation between the layers of a stack of MoE layers,
    which keeps a deep stack's hidden state bounded. Not a step of the MoE
    layer itself (gpt-oss puts an RMSNorm, with a learned gain not modelled
    here, before each MoE block)."""
    y64 = np.asarray(y, dtype=np.float64)
    ms = np.mean(y64 * y64, axis=-1, keepdims=True)
    inv = np.where(ms > 0, 1.0 / np.sqrt(np.where(ms > 0, ms, 1.0)), 0.0)
    return y64 * inv


def rownorm_rel_err(y: np.ndarray, y_ref: np.ndarray, floor: float = 1e-3) -> np.ndarray:
    """Per row t: max_c |y - y_ref| / max(max_c |y_ref|, floor)."""
    y = np.asarray(y, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    num = np.abs(y - y_ref).max(axis=-1)
    den = np.maximum(np.abs(y_ref).max(axis=-1), floor)
    return num / den


def routing_margins(logits: np.ndarray, k: int) -> np.ndarray:
    """Smallest gap, per token, among the sorted top k+1 logits (the tie guard of the router test)."""
    s = -np.sort(-np.asarray(logits, np.float64), axis=1)
    kk = min(k + 1, s.shape[1])
    gaps = s[:, :kk - 1] - s[:, 1:kk]
    return gaps.min(axis=1) if gaps.shape[1] else np.full(s.shape[0], np.inf)
