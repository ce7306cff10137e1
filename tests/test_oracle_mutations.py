"""Negative controls for the oracle's pins: a planted mistake must turn the pin red.

Each mutation is built on the CPU from a copy of an oracle function; the
oracle module itself is never modified.
"""

import numpy as np

from oracle import moe_oracle as O
from tests.test_oracle_pins import (
    check_bias_linearity,
    check_bucket_max_rows,
    check_bucket_vs_brute,
    check_decode_terms_layer,
    check_gemv_q8,
    check_q8_block_dots,
    check_quantize_q8,
    check_dequant_vs_brute,
    check_e2m1,
    check_layer_vs_brute,
    check_round_e2m1,
    check_round_e4m3,
    check_routing_margins,
    check_rownorm_rel_err,
    check_split_e2m1_vs_brute,
    check_split_vs_brute,
    check_swiglu_points,
    check_topk_vs_brute,
)


def test_pins_pass_on_the_real_oracle():
    assert check_e2m1(O.e2m1_value)
    assert check_dequant_vs_brute(O.dequant_mxfp4)
    assert check_topk_vs_brute(O.topk_softmax)
    assert check_bucket_vs_brute(O.bucket_csr)
    assert check_swiglu_points(O.swiglu_oai)
    assert check_round_e4m3(O.round_e4m3)
    assert check_split_vs_brute(O.split_e4m3_terms)
    assert check_routing_margins(O.routing_margins)
    assert check_rownorm_rel_err(O.rownorm_rel_err)
    assert check_bucket_max_rows(O.bucket_max_rows)
    assert check_round_e2m1(O.round_e2m1)
    assert check_split_e2m1_vs_brute(O.split_e2m1_terms)
    assert check_quantize_q8(O.quantize_q8)
    assert check_q8_block_dots(O.mxfp4_q8_block_dots)
    assert check_gemv_q8(O.mxfp4_gemv_q8)


def test_e2m1_subnormal_mistake_is_caught():
    def bad(code):  # treats exponent field 0 as normal
        code &= 0xF
        sign = -1.0 if code & 8 else 1.0
        e, m = (code >> 1) & 3, code & 1
        return sign * 2.0 ** (e - 1) * (1 + 0.5 * m)
    assert not check_e2m1(bad)


def test_swapped_nibbles_are_caught():
    def bad(qs, sc):
        swapped = ((qs & 0x0F) << 4) | (qs >> 4)
        return O.dequant_mxfp4(swapped.astype(np.uint8), sc)
    assert not check_dequant_vs_brute(bad)


def test_interleaved_nibbles_are_caught():
    # Reading low/high nibbles as adjacent columns (2i, 2i+1) instead of (i, i+16).
    def bad(qs, sc):
        R, half = qs.shape
        lo = O.E2M1_LUT[qs & 0x0F]
        hi = O.E2M1_LUT[qs >> 4]
        vals = np.stack([lo, hi], axis=-1).reshape(R, half * 2)
        return vals * np.repeat(O.E8M0_LUT[sc], 32, axis=1)
    assert not check_dequant_vs_brute(bad)


def test_scale_off_by_one_is_caught():
    def bad(qs, sc):
        return O.dequant_mxfp4(qs, sc) * 2.0
    assert not check_dequant_vs_brute(bad)


def test_tie_break_mistake_is_caught():
    def bad(logits, k):
        T, E = logits.shape
        ids = np.empty((T, k), np.int32)
        w = np.empty((T, k))
        for t in range(T):
            order = sorted(range(E), key=lambda e: (-logits[t, e], -e))[:k]  # higher index first
            ids[t] = order
            ex = np.exp(logits[t, order] - logits[t, order[0]])
            w[t] = ex / ex.sum()
        return ids, w
    assert not check_topk_vs_brute(bad)


def test_softmax_over_all_experts_is_caught():
    def bad(logits, k):
        ids, _ = O.topk_softmax(logits, k)
        ex = np.exp(logits - logits.max(axis=1, keepdims=True))
        full = ex / ex.sum(axis=1, keepdims=True)
        return ids, np.take_along_axis(full, ids.astype(np.int64), axis=1)
    assert not check_topk_vs_brute(bad)


def test_unpadded_prefix_is_caught():
    def bad(ids, E, tile):
        out = O.bucket_csr(ids, E, 1)  # forgets the tile padding
        mr = O.bucket_max_rows(ids.shape[0], ids.shape[1], E, tile)
        rows = np.full(mr, -1, np.int32)
        rows[:len(out["rows"])] = out["rows"][:mr]
        out["rows"] = rows
        return out
    assert not check_bucket_vs_brute(bad)


def test_descending_bucket_order_is_caught():
    def bad(ids, E, tile):
        out = O.bucket_csr(ids, E, tile)
        rows = out["rows"].copy()
        for e in range(E):
            s, n = out["basep"][e], out["counts"][e]
            rows[s:s + n] = rows[s:s + n][::-1]
        out["rows"] = rows
        return out
    assert not check_bucket_vs_brute(bad)


def test_swiglu_missing_plus_one_is_caught():
    def bad(g, u):
        g = np.minimum(g, 7.0)
        return g * O.sigmoid(1.702 * g) * np.clip(u, -7, 7)
    assert not check_swiglu_points(bad)


def test_swiglu_two_sided_gate_clamp_is_caught():
    def bad(g, u):
        g = np.clip(g, -7.0, 7.0)
        return g * O.sigmoid(1.702 * g) * (np.clip(u, -7, 7) + 1)
    assert not check_swiglu_points(bad)


def test_dropped_down_bias_is_caught():
    def bad(layer, x, k, **kw):
        L = dict(layer)
        L["bd"] = np.zeros_like(layer["bd"])
        return O.moe_layer(L, x, k, **kw)
    assert not check_bias_linearity(bad)
    assert not check_layer_vs_brute(bad)


def test_transposed_down_projection_is_caught():
    # Uses the down matrix as if stored [F, D] (square shapes make it type-check).
    def bad(layer, x, k, **kw):
        L = dict(layer)
        E = layer["d_qs"].shape[0]
        full = np.stack([O.dequant_mxfp4(layer["d_qs"][e], layer["d_sc"][e]).T for e in range(E)])

        class Cache(O.ExpertCache):
            def __call__(self, e):
                g, u, _ = super().__call__(e)
                return g, u, full[e]
        return O.moe_layer(L, x, k, cache=Cache(L), **kw)
    assert not check_layer_vs_brute(bad)


def test_unweighted_combine_is_caught():
    def bad(layer, x, k, **kw):
        y, ids, w, logits = O.moe_layer(layer, x, k, **kw)
        y2, _, _, _ = O.moe_layer(layer, x, k, ids=ids, weights=np.ones_like(w))
        return y2, ids, w, logits
    assert not check_layer_vs_brute(bad)


def test_e4m3_truncation_is_caught():
    def bad(a):  # rounds toward zero instead of to nearest
        a = np.asarray(a, np.float64)
        mag = np.abs(a)
        k = np.floor(np.log2(np.where(mag > 0, mag, 1.0)))
        q = 2.0 ** (np.maximum(k, -6.0) - 3.0)
        return np.copysign(np.minimum(np.floor(mag / q) * q, O.E4M3_MAX), a)
    assert not check_round_e4m3(bad)


def test_e4m3_ties_away_from_zero_are_caught():
    def bad(a):
        a = np.asarray(a, np.float64)
        mag = np.abs(a)
        k = np.floor(np.log2(np.where(mag > 0, mag, 1.0)))
        q = 2.0 ** (np.maximum(k, -6.0) - 3.0)
        return np.copysign(np.minimum(np.floor(mag / q + 0.5) * q, O.E4M3_MAX), a)
    assert not check_round_e4m3(bad)


def test_e4m3_term_scale_off_by_one_is_caught():
    # scale exponent floor(log2 max) - 8: the largest values saturate at 448
    def bad(v, nterms):
        v = np.asarray(v, np.float32).astype(np.float64)
        shape = v.shape
        r = v.reshape(shape[:-1] + (shape[-1] // 32, 32))
        total = np.zeros_like(r)
        for _ in range(nterms):
            amax = np.max(np.abs(r), axis=-1, keepdims=True)
            s = np.maximum(np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 8.0, -127.0)
            term = O.round_e4m3(r / 2.0 ** s) * 2.0 ** s
            total, r = total + term, r - term
        return total.reshape(shape)
    assert not check_split_vs_brute(bad)


def test_e4m3_terms_without_residual_are_caught():
    # every term re-encodes v instead of the residual of the terms before it
    def bad(v, nterms):
        one = O.split_e4m3_terms(v, 1)
        return one * nterms
    assert not check_split_vs_brute(bad)


def test_margin_of_the_boundary_gap_only_is_caught():
    # only the k-th / (k+1)-th gap, not the gaps between the selected slots
    def bad(logits, k):
        s = -np.sort(-np.asarray(logits, np.float64), axis=1)
        if k >= s.shape[1]:
            return np.full(s.shape[0], np.inf)
        return s[:, k - 1] - s[:, k]
    assert not check_routing_margins(bad)


def test_margin_without_the_boundary_gap_is_caught():
    # gaps among the k selected only (the k / k+1 boundary forgotten)
    def bad(logits, k):
        s = -np.sort(-np.asarray(logits, np.float64), axis=1)
        gaps = s[:, :k - 1] - s[:, 1:k]
        return gaps.min(axis=1) if gaps.shape[1] else np.full(s.shape[0], np.inf)
    assert not check_routing_margins(bad)


def test_margin_over_the_wrong_axis_is_caught():
    def bad(logits, k):
        s = -np.sort(-np.asarray(logits, np.float64), axis=0)  # sorts across tokens
        kk = min(k + 1, s.shape[1])
        gaps = s[:, :kk - 1] - s[:, 1:kk]
        return np.abs(gaps).min(axis=1) if gaps.shape[1] else np.full(s.shape[0], np.inf)
    assert not check_routing_margins(bad)


def test_margin_of_the_smallest_logits_is_caught():
    def bad(logits, k):
        s = np.sort(np.asarray(logits, np.float64), axis=1)  # ascending: the bottom k+1
        kk = min(k + 1, s.shape[1])
        gaps = s[:, 1:kk] - s[:, :kk - 1]
        return gaps.min(axis=1) if gaps.shape[1] else np.full(s.shape[0], np.inf)
    assert not check_routing_margins(bad)


def test_error_relative_to_the_result_is_caught():
    def bad(y, y_ref, floor=1e-3):
        num = np.abs(np.asarray(y) - np.asarray(y_ref)).max(axis=-1)
        return num / np.maximum(np.abs(np.asarray(y)).max(axis=-1), floor)
    assert not check_rownorm_rel_err(bad)


def test_error_with_one_scale_for_all_rows_is_caught():
    def bad(y, y_ref, floor=1e-3):
        num = np.abs(np.asarray(y) - np.asarray(y_ref)).max(axis=-1)
        return num / max(np.abs(np.asarray(y_ref)).max(), floor)
    assert not check_rownorm_rel_err(bad)


def test_mean_error_is_caught():
    def bad(y, y_ref, floor=1e-3):
        num = np.abs(np.asarray(y) - np.asarray(y_ref)).mean(axis=-1)
        return num / np.maximum(np.abs(np.asarray(y_ref)).max(axis=-1), floor)
    assert not check_rownorm_rel_err(bad)


def test_error_with_a_fixed_floor_is_caught():
    def bad(y, y_ref, floor=1e-3):
        return O.rownorm_rel_err(y, y_ref, floor=1e-3)
    assert not check_rownorm_rel_err(bad)


def test_max_rows_without_the_round_up_is_caught():
    def bad(T, k, E, tile):
        return T * k + E * (tile - 1)
    assert not check_bucket_max_rows(bad)


def test_max_rows_with_a_full_tile_per_expert_is_caught():
    def bad(T, k, E, tile):
        n = T * k + E * tile
        return -(-n // tile) * tile
    assert not check_bucket_max_rows(bad)


def test_max_rows_without_the_expert_padding_is_caught():
    def bad(T, k, E, tile):
        return -(-(T * k) // tile) * tile
    assert not check_bucket_max_rows(bad)


def test_decode_terms_with_the_weight_applied_twice_are_caught():
    def bad(layer, x, k, x_terms=8, h_terms=8):
        y, ids, w, h = O.moe_layer_decode_terms(layer, x, k, x_terms, h_terms)
        # the combine multiplies by w again although the operand already carries it
        y2 = np.zeros_like(y)
        for t in range(x.shape[0]):
            for j in range(k):
                e = int(ids[t, j])
                Wd = O.dequant_mxfp4(layer["d_qs"][e], layer["d_sc"][e])
                hw = O.split_e2m1_terms(w[t, j] * h[t:t + 1, j], h_terms)
                y2[t] += w[t, j] * ((hw @ Wd.T)[0] + layer["bd"][e])
        return y2, ids, w, h
    assert not check_decode_terms_layer(bad)


def test_decode_terms_without_the_gate_bias_are_caught():
    def bad(layer, x, k, x_terms=8, h_terms=8):
        L = dict(layer)
        L["bg"] = np.zeros_like(layer["bg"])
        return O.moe_layer_decode_terms(L, x, k, x_terms, h_terms)
    assert not check_decode_terms_layer(bad)


def test_e2m1_ties_away_from_zero_are_caught():
    def bad(a):
        a = np.asarray(a, np.float64)
        mag = np.abs(a)
        q = np.where(mag < 2.0, 0.5, np.where(mag < 4.0, 1.0, 2.0))
        return np.copysign(np.minimum(np.floor(mag / q + 0.5) * q, 6.0), a)
    assert not check_round_e2m1(bad)


def test_e2m1_without_saturation_is_caught():
    def bad(a):
        a = np.asarray(a, np.float64)
        mag = np.abs(a)
        q = np.where(mag < 2.0, 0.5, np.where(mag < 4.0, 1.0, 2.0))
        lo = np.floor(mag / q) * q
        frac = mag - lo
        even = np.isin(lo, (0.0, 1.0, 2.0, 4.0))
        up = (frac > q / 2) | ((frac == q / 2) & ~even)
        return np.copysign(np.where(up, lo + q, lo), a)  # 7.0 stays 8.0
    assert not check_round_e2m1(bad)


def test_e2m1_term_scale_one_step_too_small_is_caught():
    # 2^e with max|r| / 2^e in (6, 12]: the largest values saturate at 6
    def bad(v, nterms):
        v = np.asarray(v, np.float32).astype(np.float64)
        shape = v.shape
        r = v.reshape(shape[:-1] + (shape[-1] // 32, 32))
        total = np.zeros_like(r)
        for _ in range(nterms):
            amax = np.max(np.abs(r), axis=-1, keepdims=True)
            e = np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 2.0
            e = np.clip(e - (amax <= 6.0 * 2.0 ** e), -127.0, 127.0)
            term = O.round_e2m1(r / 2.0 ** e) * 2.0 ** e
            total, r = total + term, r - term
        return total.reshape(shape)
    assert not check_split_e2m1_vs_brute(bad)


def test_e2m1_terms_without_residual_are_caught():
    def bad(v, nterms):
        return O.split_e2m1_terms(v, 1) * nterms
    assert not check_split_e2m1_vs_brute(bad)


def test_q8_truncating_codes_are_caught():
    def bad(v):
        v = np.asarray(v, np.float32)
        q, d = O.quantize_q8(v)
        blk = v.reshape(v.shape[:-1] + (-1, 32))
        amax = np.abs(blk).max(-1)
        inv = np.float32(127) / np.where(amax > 0, amax, 1).astype(np.float32)
        qt = np.trunc(blk * inv[..., None]).astype(np.int8).reshape(v.shape)
        return qt, d
    assert not check_quantize_q8(bad)


def test_q8_ties_away_from_zero_are_caught():
    def bad(v):
        v = np.asarray(v, np.float32)
        _, d = O.quantize_q8(v)
        blk = v.reshape(v.shape[:-1] + (-1, 32))
        amax = np.abs(blk).max(-1)
        inv = np.float32(127) / np.where(amax > 0, amax, 1).astype(np.float32)
        t = (blk * inv[..., None]).astype(np.float32)
        qa = (np.sign(t) * np.floor(np.abs(t) + 0.5)).astype(np.int8).reshape(v.shape)
        return qa, d
    assert not check_quantize_q8(bad)


def test_q8_scale_of_255_is_caught():
    def bad(v):
        v = np.asarray(v, np.float32)
        blk = v.reshape(v.shape[:-1] + (-1, 32))
        amax = np.abs(blk).max(-1)
        safe = np.where(amax > 0, amax, 1).astype(np.float32)
        q = np.rint(blk * (np.float32(255) / safe)[..., None] / 2).astype(np.int8).reshape(v.shape)
        return q, np.where(amax > 0, safe / np.float32(127), 0).astype(np.float32)
    assert not check_quantize_q8(bad)


def test_q8_dot_with_swapped_nibbles_is_caught():
    def bad(qs, q):
        return O.mxfp4_q8_block_dots((((qs & 0x0F) << 4) | (qs >> 4)).astype(np.uint8), q)
    assert not check_q8_block_dots(bad)


def test_q8_dot_with_the_plain_table_is_caught():
    def bad(qs, q):  # the E2M1 table not doubled: the integer sums come out halved
        return O.mxfp4_q8_block_dots(qs, q) // 2
    assert not check_q8_block_dots(bad)


def test_q8_gemv_with_the_undoubled_scale_is_caught():
    def bad(qs, sc, q, d, bias):  # 2**(s-127): the doubled table not compensated
        return O.mxfp4_gemv_q8(qs, (sc.astype(np.int64) + 1).clip(0, 254).astype(np.uint8), q, d, bias)
    assert not check_gemv_q8(bad)


def test_q8_gemv_without_the_bias_is_caught():
    def bad(qs, sc, q, d, bias):
        return O.mxfp4_gemv_q8(qs, sc, q, d, None)
    assert not check_gemv_q8(bad)
