"""Host-side checks of the C ABI: exports, size queries, argument rejection.

Nothing here launches a kernel; every call either is a pure host query or is
rejected on the host before the library touches the device.
"""

import os
import numpy as np
import pytest

from oracle import moe_oracle as O

FAKE = 1 << 20  # a non-null, 256-byte aligned pointer value that is never dereferenced


def test_library_exports_every_declared_symbol(moe):
    names = moe._lib.declared_functions()
    assert len(names) == 31
    assert set(names) <= set(moe._lib._SIGS), "every declared function has a binding"
    for n in names:
        assert hasattr(moe._lib._lib, n), n


@pytest.mark.parametrize("T,k,E,tile", [(0, 2, 4, 4), (1, 4, 32, 128), (8, 2, 4, 128), (512, 4, 32, 128),
                                        (4096, 4, 32, 128), (13, 3, 5, 16), (40, 4, 6, 1)])
def test_bucket_max_rows_matches_oracle(moe, T, k, E, tile):
    assert moe.moe_bucket_max_rows(T, k, E, tile) == O.bucket_max_rows(T, k, E, tile)


def test_bucket_max_rows_rejects(moe):
    assert moe.moe_bucket_max_rows(-1, 2, 4, 4) == 0
    assert moe.moe_bucket_max_rows(1, 0, 4, 4) == 0
    assert moe.moe_bucket_max_rows(1, 2, 4, 0) == 0


def test_workspace_bytes(moe):
    gemv = moe.moe_ffn_workspace_bytes(1, 2880, 2880, 32, 4, moe.MOE_RAIL_GEMV)
    mm = moe.moe_ffn_workspace_bytes(512, 2880, 2880, 32, 4, moe.MOE_RAIL_GROUPED_MM)
    assert gemv >= 4 * 2880 * 4 and gemv % 256 == 0
    mr = O.bucket_max_rows(512, 4, 32, 128)
    assert mm >= mr * 2880 * 2 * 2
    assert moe.moe_ffn_workspace_bytes(1, 2880, 2880, 32, 4, moe.MOE_RAIL_AUTO) == gemv
    assert moe.moe_ffn_workspace_bytes(512, 2880, 2880, 32, 4, moe.MOE_RAIL_AUTO) == mm
    assert moe.moe_ffn_workspace_bytes(1, 2880, 2880, 4, 8, moe.MOE_RAIL_AUTO) == 0  # k > E
    assert moe.moe_ffn_workspace_bytes(1, 2880, 2880, 32, 4, 7) == 0  # unknown rail
    mx = moe.moe_ffn_workspace_bytes(512, 2880, 2880, 32, 4, moe.MOE_RAIL_GROUPED_MX)
    # three E4M3 terms of x and two of h, plus one scale word per 4 blocks of each term
    assert mx >= mr * 2880 * 5 + 5 * 23 * mr * 4 and mx % 256 == 0


def test_route_topk_rejects_bad_arguments(moe):
    E, EINVAL = moe.MOE_EINVAL, moe.MOE_EINVAL
    args = dict(x=FAKE, T=4, D=64, w_router=FAKE, b_router=None, E=8, k=2, logits=FAKE, ids=FAKE,
                weights=FAKE)
    bad = [dict(x=None), dict(T=-1), dict(D=6), dict(k=0), dict(k=9), dict(E=300, k=2),
           dict(logits=None), dict(x=FAKE + 4)]
    for b in bad:
        a = dict(args, **b)
        assert moe.moe_route_topk(*a.values(), stream=0) == EINVAL, b


def test_t_zero_is_a_host_side_noop(moe):
    # T = 0 returns before touching the device, even with null buffers.
    assert moe.moe_route_topk(None, 0, 64, None, None, 8, 2, None, None, None, stream=0) == moe.MOE_OK
    assert moe.moe_mxfp4_gemv(None, None, 4, 64, 64, None, 0, None, 0, None, None, stream=0) == moe.MOE_OK
    assert moe.moe_swiglu_oai(None, None, None, 0, moe.MOE_DTYPE_F32, stream=0) == moe.MOE_OK


def test_bucket_rejects_bad_arguments(moe):
    EINVAL = moe.MOE_EINVAL
    assert moe.moe_bucket(FAKE, 4, 2, 8, 0, FAKE, FAKE, FAKE, FAKE, stream=0) == EINVAL
    assert moe.moe_bucket(FAKE, 4, 0, 8, 4, FAKE, FAKE, FAKE, FAKE, stream=0) == EINVAL
    assert moe.moe_bucket(FAKE, 4, 2, 0, 4, FAKE, FAKE, FAKE, FAKE, stream=0) == EINVAL
    assert moe.moe_bucket(None, 4, 2, 8, 4, FAKE, FAKE, FAKE, FAKE, stream=0) == EINVAL
    assert moe.moe_bucket(FAKE, 4, 2, 8, 4, FAKE, None, FAKE, FAKE, stream=0) == EINVAL


def test_gemv_rejects_bad_arguments(moe):
    EINVAL = moe.MOE_EINVAL
    ok = [FAKE, FAKE, 4, 64, 64, FAKE, 2, FAKE, 64, None, FAKE]
    for i, v in [(4, 48), (4, 0), (3, 0), (8, 6), (0, None), (7, FAKE + 8)]:
        a = list(ok)
        a[i] = v
        assert moe.moe_mxfp4_gemv(*a, stream=0) == EINVAL, (i, v)
    a = list(ok)
    a[4] = 8192
    assert moe.moe_mxfp4_gemv(*a, stream=0) == moe.MOE_EUNSUPPORTED


def test_swiglu_rejects_bad_dtype(moe):
    assert moe.moe_swiglu_oai(FAKE, FAKE, FAKE, 10, 5, stream=0) == moe.MOE_EINVAL
    assert moe.moe_swiglu_oai(None, FAKE, FAKE, 10, 0, stream=0) == moe.MOE_EINVAL


def test_rms_renorm_rejects_bad_arguments(moe):
    assert moe.moe_rms_renorm(None, 0, 64, None, stream=0) == moe.MOE_OK
    assert moe.moe_rms_renorm(FAKE, -1, 64, FAKE, stream=0) == moe.MOE_EINVAL
    assert moe.moe_rms_renorm(FAKE, 2, 0, FAKE, stream=0) == moe.MOE_EINVAL
    assert moe.moe_rms_renorm(None, 2, 64, FAKE, stream=0) == moe.MOE_EINVAL


def test_grouped_mm_rejects_bad_arguments(moe):
    EINVAL, EUNS = moe.MOE_EINVAL, moe.MOE_EUNSUPPORTED
    base = dict(w_qs=FAKE, w_sc=FAKE, bias=None, w2_qs=None, w2_sc=None, bias2=None, E=4, R=64, C=64,
                a=FAKE, a_lo=None, counts=FAKE, basep=FAKE, rows=FAKE, max_rows=512, k=2, weights=None,
                epilogue=moe.MOE_EPI_STORE_BF16, alpha=1.702, limit=7.0, out=FAKE, out_ld=64)
    call = lambda **kw: moe.moe_mxfp4_grouped_mm(*dict(base, **kw).values(), stream=0)  # noqa: E731
    assert call(epilogue=9) == EINVAL
    assert call(max_rows=100) == EINVAL
    assert call(out_ld=32) == EINVAL
    assert call(C=96) == EUNS            # C not a multiple of 64
    assert call(R=60) == EUNS            # R not a multiple of 8
    assert call(C=8192) == EUNS
    assert call(epilogue=moe.MOE_EPI_SWIGLU_BF16) == EINVAL          # second matrix missing
    assert call(epilogue=moe.MOE_EPI_SCATTER_WEIGHTED) == EINVAL     # weights missing
    assert call(a=FAKE + 8) == EINVAL
    assert call(a_lo=FAKE + 8) == EINVAL


def test_ffn_layer_rejects_bad_arguments(moe):
    EINVAL = moe.MOE_EINVAL
    need = moe.moe_ffn_workspace_bytes(4, 64, 64, 4, 2, moe.MOE_RAIL_GEMV)
    base = [FAKE, 4, 64, 64, 4, 2] + [FAKE] * 11 + [moe.MOE_RAIL_GEMV, FAKE, need, FAKE]
    base[7] = None  # b_router may be NULL

    def call(**kw):
        a = list(base)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return moe.moe_ffn_layer(*a, stream=0)

    assert call(a2=48) == EINVAL                     # D not a multiple of 64
    assert call(a5=5) == EINVAL                      # k > E
    assert call(a17=moe.MOE_RAIL_GEMV, a1=9) == EINVAL  # GEMV rail beyond its token limit
    assert call(a19=need - 1) == EINVAL              # workspace too small
    assert call(a18=FAKE + 16) == EINVAL             # workspace misaligned
    assert call(a0=None) == EINVAL
    assert call(a17=5) == EINVAL                     # unknown rail


def test_status_reader_rejects_null(moe):
    import ctypes
    assert moe._lib._lib.moe_get_status(None, ctypes.POINTER(ctypes.c_int)()) == moe.MOE_EINVAL


def test_valid_call_without_a_gpu_reports_a_cuda_error(moe):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc, _ = moe.moe_get_status(stream=0)
    assert rc in (moe.MOE_ECUDA, moe.MOE_EUNSUPPORTED)


def test_hostio_rejects_missing_arguments(moe):
    """moe_ffn_layer_hostio checks its argument block on the host before enqueueing anything."""
    assert moe.moe_ffn_layer_hostio(None, 0, 0, 0) == moe.MOE_EINVAL
    args = moe.MoeFfnArgs(1, 64, 64, 4, 2, moe.MOE_RAIL_GEMV)
    assert moe.moe_ffn_layer_hostio(args, 0, 0, 0) == moe.MOE_EINVAL  # no host or staging buffers
    args.T = 0
    assert moe.moe_ffn_layer_hostio(args, 0, 0, 0) == moe.MOE_OK      # nothing to do


def test_packed_sizes(moe):
    # qs_p: E * R * ceil(C/128) * 64 bytes; sf_p: one 512-byte atom per 128-row tile and 128-column chunk
    assert moe.moe_mxfp4_packed_qs_bytes(32, 2880, 2880) == 32 * 2880 * 23 * 64  # rows padded to 128-column chunks
    assert moe.moe_mxfp4_packed_sf_bytes(32, 2880, 2880) == 32 * 23 * 23 * 512
    assert moe.moe_mxfp4_packed_qs_bytes(3, 192, 320) == 3 * 192 * 3 * 64
    assert moe.moe_mxfp4_packed_sf_bytes(3, 192, 320) == 3 * 2 * 3 * 512
    assert moe.moe_mxfp4_packed_qs_bytes(3, 100, 320) == 0
    assert moe.moe_mxfp4_packed_sf_bytes(3, 192, 48) == 0
    assert moe.moe_ffn_packed_workspace_bytes(1, 2880, 2880, 32, 4, moe.MOE_RAIL_AUTO) > 0
    assert moe.moe_ffn_packed_workspace_bytes(1, 2880, 2880, 32, 4, moe.MOE_RAIL_DECODE_MX) % 256 == 0
    # beyond decode sizes the packed layer runs the prefill rail on the same planes
    assert moe.moe_ffn_packed_workspace_bytes(9, 2880, 2880, 32, 4, moe.MOE_RAIL_AUTO) == \
        moe.moe_ffn_packed_workspace_bytes(9, 2880, 2880, 32, 4, moe.MOE_RAIL_GROUPED_MX4) > 0
    assert moe.moe_ffn_packed_workspace_bytes(9, 2880, 2880, 32, 4, moe.MOE_RAIL_DECODE_MX) == 0


def test_packed_layer_rejects_on_the_host(moe):
    L = moe.make_packed_layer(2880, 2880, 32, 4, FAKE, None, FAKE, FAKE, None, FAKE, FAKE, None, FAKE, FAKE, None)
    n = moe.moe_ffn_packed_workspace_bytes(1, 2880, 2880, 32, 4, moe.MOE_RAIL_AUTO)
    assert moe.moe_ffn_layer_packed(None, FAKE, 1, 0, FAKE, n, FAKE, stream=0) == moe.MOE_EINVAL
    assert moe.moe_ffn_layer_packed(L, FAKE, 1, 0, FAKE, n - 256, FAKE, stream=0) == moe.MOE_EINVAL
    assert moe.moe_ffn_layer_packed(L, FAKE + 8, 1, 0, FAKE, n, FAKE, stream=0) == moe.MOE_EINVAL
    L.g_qs = FAKE + 16  # prepacked planes must be 32-byte aligned for the copy engine
    assert moe.moe_ffn_layer_packed(L, FAKE, 1, 0, FAKE, n, FAKE, stream=0) == moe.MOE_EINVAL
    L.g_qs = FAKE
    L.D = 2880 + 32
    assert moe.moe_ffn_layer_packed(L, FAKE, 1, 0, FAKE, n, FAKE, stream=0) == moe.MOE_EINVAL
    L.D = 2880
    assert moe.moe_ffn_layer_packed(L, FAKE, 0, 0, FAKE, n, FAKE, stream=0) == moe.MOE_OK


def test_binding_constants_match_the_header(moe):
    import re

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    text = open(os.path.join(root, "include", "moe_mxfp4.h")).read()
    checked = 0
    for name, raw in re.findall(r"^#define (MOE_[A-Z0-9_]+)\s+([^/\n]+)", text, re.M):
        v = raw.strip().strip("()").replace("u", "")
        if re.fullmatch(r"-?(0x[0-9a-fA-F]+|\d+)", v):
            val = int(v, 0)
        elif re.fullmatch(r"\d+\s*\*\s*\d+", v):
            a, b = (int(t) for t in v.split("*"))
            val = a * b
        else:
            continue
        if hasattr(moe, name):
            assert getattr(moe, name) == val, name
            checked += 1
    assert checked >= 20


def test_q8_entry_points_reject_bad_arguments(moe):
    EINVAL = moe.MOE_EINVAL
    assert moe.moe_quantize_q8(None, 0, 64, None, None, stream=0) == moe.MOE_OK
    assert moe.moe_quantize_q8(FAKE, 2, 48, FAKE, FAKE, stream=0) == EINVAL  # C not a multiple of 32
    assert moe.moe_quantize_q8(None, 2, 64, FAKE, FAKE, stream=0) == EINVAL
    assert moe.moe_mxfp4_gemv_q8(FAKE, FAKE, 2, 8, 64, FAKE, 0, 1, FAKE, FAKE, None, FAKE, stream=0) == moe.MOE_OK
    assert moe.moe_mxfp4_gemv_q8(FAKE, FAKE, 2, 8, 64, FAKE, 1, 0, FAKE, FAKE, None, FAKE, stream=0) == EINVAL
    assert moe.moe_mxfp4_gemv_q8(FAKE, FAKE, 2, 8, 8192, FAKE, 1, 1, FAKE, FAKE, None, FAKE,
                                 stream=0) == moe.MOE_EUNSUPPORTED
    assert moe.moe_ffn_workspace_bytes(1, 2880, 2880, 32, 4, moe.MOE_RAIL_GEMV_Q8) > 0
    assert moe.moe_ffn_workspace_bytes(9, 2880, 2880, 32, 4, moe.MOE_RAIL_GEMV_Q8) == 0
