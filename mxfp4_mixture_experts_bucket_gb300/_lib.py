"""ctypes binding of libmoe_mxfp4.so: the C ABI of include/moe_mxfp4.h, same names.

Argument marshalling only. Tensors are passed as raw pointers (torch tensors
by ``data_ptr()``), streams default to torch's current CUDA stream. Every
kernel runs inside the library; if the library is missing this module raises
at import time instead of falling back to anything else.
"""

from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
# MOE_MXFP4_CHECKED=1 loads the checked build (libmoe_mxfp4_checked.so: device-side bounds checks)
LIB_PATH = os.path.join(HERE, "libmoe_mxfp4_checked.so" if os.environ.get("MOE_MXFP4_CHECKED") == "1"
                        else "libmoe_mxfp4.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "moe_mxfp4.h")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'` "
        "or `python -m mxfp4_mixture_experts_bucket_gb300.build`")

_lib = ctypes.CDLL(LIB_PATH)

# ---- constants mirrored from the header ----
MOE_OK = 0
MOE_EINVAL = -1
MOE_ECUDA = -2
MOE_EUNSUPPORTED = -3
MOE_ESCRATCH = -4
MOE_DECODE_SCRATCH_BYTES = 512 * 1024
MOE_STATUS_BAD_EXPERT_ID = 0x1
MOE_STATUS_WAIT_TIMEOUT = 0x2
MOE_STATUS_OUT_OF_BOUNDS = 0x4
MOE_DTYPE_F32 = 0
MOE_DTYPE_BF16 = 1
MOE_EPI_STORE_BF16 = 0
MOE_EPI_SWIGLU_BF16 = 1
MOE_EPI_SCATTER_WEIGHTED = 2
MOE_RAIL_AUTO = 0
MOE_RAIL_GEMV = 1
MOE_RAIL_GROUPED_MM = 2
MOE_RAIL_GROUPED_MX = 3
MOE_RAIL_DECODE_MX = 4
MOE_RAIL_GEMV_Q8 = 5
MOE_RAIL_GROUPED_MX4 = 6
MOE_STAGE_PROLOGUE = 1
MOE_STAGE_GATEUP = 2
MOE_STAGE_DOWN = 4
MOE_GEMV_MAX_T = 8
MOE_AUTO_GEMV_MAX_T = 8
MOE_AUTO_MX_MAX_T = 320
MOE_AUTO_DECODE_MX_MAX_T = 2
MOE_MM_TILE = 128

P = ctypes.c_void_p
I = ctypes.c_int
I64 = ctypes.c_int64
F = ctypes.c_float
SZ = ctypes.c_size_t

_SIGS = {
    "moe_bucket_max_rows": (SZ, [I, I, I, I]),
    "moe_ffn_workspace_bytes": (SZ, [I, I, I, I, I, I]),
    "moe_route_topk": (I, [P, I, I, P, P, I, I, P, P, P, P]),
    "moe_bucket": (I, [P, I, I, I, I, P, P, P, P, P]),
    "moe_mxfp4_gemv": (I, [P, P, I, I, I, P, I, P, I64, P, P, P]),
    "moe_swiglu_oai": (I, [P, P, P, I64, I, F, F, P]),
    "moe_rms_renorm": (I, [P, I, I, P, P]),
    "moe_ffn_layer_gu": (I, [P, I, I, I, I, I, P, P, P, P, P, P, P, P, I, P, SZ, P, P, P, P]),
    "moe_mxfp4_prepack_gu": (I, [P, P, I, I, I, P, P, P, P, P]),
    "moe_quantize_q8": (I, [P, I64, I, P, P, P]),
    "moe_mxfp4_gemv_q8": (I, [P, P, I, I, I, P, I, I, P, P, P, P, P]),
    "moe_selftest_wait_timeout": (I, [P, P]),
    "moe_gather_rows_bf16": (I, [P, I, I, I, P, P, I, I, P, P, P, P]),
    "moe_mxfp4_grouped_mm": (I, [P, P, P, P, P, P, I, I, I, P, P, P, P, P, I, I, P, I, F, F, P, I64, P]),
    "moe_expert_gateup_swiglu": (I, [P, P, P, P, P, P, I, I, I, I, I, P, P, F, F, P, P]),
    "moe_expert_down_combine": (I, [P, P, P, I, I, I, I, I, P, P, P, P, P]),
    "moe_ffn_layer": (I, [P, I, I, I, I, I, P, P, P, P, P, P, P, P, P, P, P, I, P, SZ, P, P, P, P]),
    "moe_ffn_layer_hostio": (I, [P, P, P, P]),
    "moe_ffn_layer_decode_static": (I, [P, I, I, I, I, I, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P]),
    "moe_mxfp4_packed_qs_bytes": (SZ, [I, I, I]),
    "moe_mxfp4_packed_sf_bytes": (SZ, [I, I, I]),
    "moe_mxfp4_prepack": (I, [P, P, I, I, I, P, P, P]),
    "moe_ffn_packed_workspace_bytes": (SZ, [I, I, I, I, I, I]),
    "moe_ffn_layer_packed": (I, [P, P, I, I, P, SZ, P, P, P, P, P]),
    "moe_ffn_layer_packed_hostio": (I, [P, I, I, P, SZ, P, P, P]),
    "moe_ffn_layer_packed_stage": (I, [P, P, I, P, SZ, I, P, P, P, P, P]),
    "moe_checked_build": (I, []),
    "moe_get_status": (I, [P, ctypes.POINTER(ctypes.c_int)]),
    "moe_get_timeout_site": (I, [P, ctypes.POINTER(ctypes.c_int)]),
    "moe_last_cuda_error": (I, []),
    "moe_kernel_launches": (ctypes.c_uint64, []),
}

for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


def declared_functions():
    """Names of the functions include/moe_mxfp4.h declares."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


class MoeError(RuntimeError):
    pass


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    if hasattr(t, "ctypes"):  # numpy array (host memory): only for host-side argument checks
        return t.ctypes.data
    raise TypeError(f"cannot pass {type(t)} as a pointer")


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream
    return s


def check(rc: int, what: str = "call"):
    if rc != MOE_OK:
        extra = f" (cudaError {moe_last_cuda_error()})" if rc == MOE_ECUDA else ""
        raise MoeError(f"{what} returned {rc}{extra}")
    return rc


# ---- thin wrappers, same names and argument order as the C ABI ----

def moe_bucket_max_rows(T, k, E, tile):
    return _lib.moe_bucket_max_rows(T, k, E, tile)


def moe_ffn_workspace_bytes(T, D, F, E, k, rail=MOE_RAIL_AUTO):
    return _lib.moe_ffn_workspace_bytes(T, D, F, E, k, rail)


def moe_route_topk(x, T, D, w_router, b_router, E, k, logits, ids, weights, stream=None):
    return _lib.moe_route_topk(_ptr(x), T, D, _ptr(w_router), _ptr(b_router), E, k, _ptr(logits),
                               _ptr(ids), _ptr(weights), _stream(stream))


def moe_bucket(ids, T, k, E, tile, counts, basep, rows, inv, stream=None):
    return _lib.moe_bucket(_ptr(ids), T, k, E, tile, _ptr(counts), _ptr(basep), _ptr(rows), _ptr(inv),
                           _stream(stream))


def moe_mxfp4_gemv(w_qs, w_sc, E, R, C, experts, n, x, x_stride, bias, out, stream=None):
    return _lib.moe_mxfp4_gemv(_ptr(w_qs), _ptr(w_sc), E, R, C, _ptr(experts), n, _ptr(x), x_stride,
                               _ptr(bias), _ptr(out), _stream(stream))


def moe_selftest_wait_timeout(src, stream=None):
    return _lib.moe_selftest_wait_timeout(_ptr(src), _stream(stream))


def moe_quantize_q8(x, rows, C, q, d, stream=None):
    return _lib.moe_quantize_q8(_ptr(x), rows, C, _ptr(q), _ptr(d), _stream(stream))


def moe_mxfp4_gemv_q8(w_qs, w_sc, E, R, C, experts, n, act_div, q, d, bias, out, stream=None):
    return _lib.moe_mxfp4_gemv_q8(_ptr(w_qs), _ptr(w_sc), E, R, C, _ptr(experts), n, act_div, _ptr(q), _ptr(d),
                                  _ptr(bias), _ptr(out), _stream(stream))


def moe_ffn_layer_gu(x, T, D, F, E, k, w_router, b_router, gu_qs, gu_sc, gu_b, d_qs, d_sc, bd, rail,
                     workspace, workspace_bytes, y, ids_out=None, weights_out=None, stream=None):
    return _lib.moe_ffn_layer_gu(_ptr(x), T, D, F, E, k, _ptr(w_router), _ptr(b_router), _ptr(gu_qs), _ptr(gu_sc),
                                 _ptr(gu_b), _ptr(d_qs), _ptr(d_sc), _ptr(bd), rail, _ptr(workspace),
                                 workspace_bytes, _ptr(y), _ptr(ids_out), _ptr(weights_out), _stream(stream))


def moe_mxfp4_prepack_gu(gu_qs, gu_sc, E, F, D, g_qs_p, g_sf_p, u_qs_p, u_sf_p, stream=None):
    return _lib.moe_mxfp4_prepack_gu(_ptr(gu_qs), _ptr(gu_sc), E, F, D, _ptr(g_qs_p), _ptr(g_sf_p), _ptr(u_qs_p),
                                     _ptr(u_sf_p), _stream(stream))


def moe_rms_renorm(x, T, D, y, stream=None):
    return _lib.moe_rms_renorm(_ptr(x), T, D, _ptr(y), _stream(stream))


def moe_swiglu_oai(g, u, h, n, h_dtype, alpha=1.702, limit=7.0, stream=None):
    return _lib.moe_swiglu_oai(_ptr(g), _ptr(u), _ptr(h), n, h_dtype, alpha, limit, _stream(stream))


def moe_gather_rows_bf16(x, T, D, k, rows, basep, E, max_rows, xg, xg_lo=None, y_zero=None, stream=None):
    return _lib.moe_gather_rows_bf16(_ptr(x), T, D, k, _ptr(rows), _ptr(basep), E, max_rows, _ptr(xg),
                                     _ptr(xg_lo), _ptr(y_zero), _stream(stream))


def moe_mxfp4_grouped_mm(w_qs, w_sc, bias, w2_qs, w2_sc, bias2, E, R, C, a, a_lo, counts, basep, rows,
                         max_rows, k, weights, epilogue, alpha, limit, out, out_ld, stream=None):
    return _lib.moe_mxfp4_grouped_mm(_ptr(w_qs), _ptr(w_sc), _ptr(bias), _ptr(w2_qs), _ptr(w2_sc),
                                     _ptr(bias2), E, R, C, _ptr(a), _ptr(a_lo), _ptr(counts), _ptr(basep),
                                     _ptr(rows), max_rows, k, _ptr(weights), epilogue, alpha, limit,
                                     _ptr(out), out_ld, _stream(stream))


def moe_expert_gateup_swiglu(g_qs, g_sc, bg, u_qs, u_sc, bu, E, F, D, T, k, x, ids, alpha, limit, h,
                             stream=None):
    return _lib.moe_expert_gateup_swiglu(_ptr(g_qs), _ptr(g_sc), _ptr(bg), _ptr(u_qs), _ptr(u_sc),
                                         _ptr(bu), E, F, D, T, k, _ptr(x), _ptr(ids), alpha, limit,
                                         _ptr(h), _stream(stream))


def moe_expert_down_combine(d_qs, d_sc, bd, E, D, F, T, k, h, ids, weights, y, stream=None):
    return _lib.moe_expert_down_combine(_ptr(d_qs), _ptr(d_sc), _ptr(bd), E, D, F, T, k, _ptr(h),
                                        _ptr(ids), _ptr(weights), _ptr(y), _stream(stream))


def moe_ffn_layer(x, T, D, F, E, k, w_router, b_router, g_qs, g_sc, bg, u_qs, u_sc, bu, d_qs, d_sc,
                  bd, rail, workspace, workspace_bytes, y, ids_out=None, weights_out=None,
                  stream=None):
    return _lib.moe_ffn_layer(_ptr(x), T, D, F, E, k, _ptr(w_router), _ptr(b_router), _ptr(g_qs),
                              _ptr(g_sc), _ptr(bg), _ptr(u_qs), _ptr(u_sc), _ptr(bu), _ptr(d_qs),
                              _ptr(d_sc), _ptr(bd), rail, _ptr(workspace), workspace_bytes, _ptr(y),
                              _ptr(ids_out), _ptr(weights_out), _stream(stream))


class MoeFfnArgs(ctypes.Structure):
    """moe_ffn_args_t of the header: the fixed arguments of moe_ffn_layer_hostio."""
    _fields_ = [("T", I), ("D", I), ("F", I), ("E", I), ("k", I), ("rail", I),
                ("w_router", P), ("b_router", P), ("g_qs", P), ("g_sc", P), ("bg", P),
                ("u_qs", P), ("u_sc", P), ("bu", P), ("d_qs", P), ("d_sc", P), ("bd", P),
                ("workspace", P), ("workspace_bytes", SZ), ("x_dev", P), ("y_dev", P)]


def make_ffn_args(T, D, F, E, k, rail, w_router, b_router, g_qs, g_sc, bg, u_qs, u_sc, bu, d_qs, d_sc,
                  bd, workspace, workspace_bytes, x_dev, y_dev) -> MoeFfnArgs:
    return MoeFfnArgs(T, D, F, E, k, rail, _ptr(w_router), _ptr(b_router), _ptr(g_qs), _ptr(g_sc),
                      _ptr(bg), _ptr(u_qs), _ptr(u_sc), _ptr(bu), _ptr(d_qs), _ptr(d_sc), _ptr(bd),
                      _ptr(workspace), workspace_bytes, _ptr(x_dev), _ptr(y_dev))


def moe_ffn_layer_hostio(args, x_host, y_host, stream=None):
    return _lib.moe_ffn_layer_hostio(None if args is None else ctypes.byref(args), _ptr(x_host),
                                     _ptr(y_host), _stream(stream))


def byref_args(args):
    """A reference to an argument struct that can be passed again without rebuilding it
    (keep `args` alive as long as the reference is used)."""
    return ctypes.byref(args)


def moe_ffn_layer_hostio_ref(args_ref, x_host_ptr, y_host_ptr, stream_handle):
    """moe_ffn_layer_hostio with everything already converted: args_ref from byref_args,
    host addresses and the stream handle as ints (the per-step path of MoeLayer.forward_host)."""
    return _lib.moe_ffn_layer_hostio(args_ref, x_host_ptr, y_host_ptr, stream_handle)


def moe_ffn_layer_decode_static(x, T, D, F, E, k, w_router, b_router, g_qs, g_sc, bg, u_qs, u_sc, bu,
                                d_qs, d_sc, bd, y, ids_out=None, weights_out=None, stream=None):
    return _lib.moe_ffn_layer_decode_static(_ptr(x), T, D, F, E, k, _ptr(w_router), _ptr(b_router),
                                            _ptr(g_qs), _ptr(g_sc), _ptr(bg), _ptr(u_qs), _ptr(u_sc),
                                            _ptr(bu), _ptr(d_qs), _ptr(d_sc), _ptr(bd), _ptr(y),
                                            _ptr(ids_out), _ptr(weights_out), _stream(stream))


def moe_mxfp4_packed_qs_bytes(E, R, C):
    return _lib.moe_mxfp4_packed_qs_bytes(E, R, C)


def moe_mxfp4_packed_sf_bytes(E, R, C):
    return _lib.moe_mxfp4_packed_sf_bytes(E, R, C)


def moe_mxfp4_prepack(qs, sc, E, R, C, qs_p, sf_p, stream=None):
    return _lib.moe_mxfp4_prepack(_ptr(qs), _ptr(sc), E, R, C, _ptr(qs_p), _ptr(sf_p), _stream(stream))


class MoePackedLayer(ctypes.Structure):
    """moe_packed_layer_t of the header: one layer's weights with prepacked expert planes."""
    _fields_ = [("D", I), ("F", I), ("E", I), ("k", I), ("w_router", P), ("b_router", P),
                ("g_qs", P), ("g_sf", P), ("bg", P), ("u_qs", P), ("u_sf", P), ("bu", P),
                ("d_qs", P), ("d_sf", P), ("bd", P)]


def make_packed_layer(D, F, E, k, w_router, b_router, g_qs, g_sf, bg, u_qs, u_sf, bu, d_qs, d_sf,
                      bd) -> MoePackedLayer:
    return MoePackedLayer(D, F, E, k, _ptr(w_router), _ptr(b_router), _ptr(g_qs), _ptr(g_sf), _ptr(bg),
                          _ptr(u_qs), _ptr(u_sf), _ptr(bu), _ptr(d_qs), _ptr(d_sf), _ptr(bd))


def moe_ffn_packed_workspace_bytes(T, D, F, E, k, rail=MOE_RAIL_AUTO):
    return _lib.moe_ffn_packed_workspace_bytes(T, D, F, E, k, rail)


def moe_ffn_layer_packed(layer, x, T, rail, workspace, workspace_bytes, y, ids_out=None, weights_out=None,
                         h_out=None, stream=None):
    return _lib.moe_ffn_layer_packed(None if layer is None else ctypes.byref(layer), _ptr(x), T, rail,
                                     _ptr(workspace), workspace_bytes, _ptr(y), _ptr(ids_out),
                                     _ptr(weights_out), _ptr(h_out), _stream(stream))


def moe_ffn_layer_packed_stage(layer, x, T, workspace, workspace_bytes, stages, y=None, ids_out=None,
                               weights_out=None, h_out=None, stream=None):
    return _lib.moe_ffn_layer_packed_stage(None if layer is None else ctypes.byref(layer), _ptr(x), T,
                                           _ptr(workspace), workspace_bytes, stages, _ptr(y), _ptr(ids_out),
                                           _ptr(weights_out), _ptr(h_out), _stream(stream))


def moe_ffn_layer_packed_hostio(layer, T, rail, workspace, workspace_bytes, x_host, y_host, stream=None):
    return _lib.moe_ffn_layer_packed_hostio(None if layer is None else ctypes.byref(layer), T, rail,
                                            _ptr(workspace), workspace_bytes, _ptr(x_host), _ptr(y_host),
                                            _stream(stream))


def moe_checked_build():
    return _lib.moe_checked_build()


def moe_get_status(stream=None):
    v = ctypes.c_int(0)
    rc = _lib.moe_get_status(_stream(stream), ctypes.byref(v))
    return rc, v.value


def moe_get_timeout_site(stream=None):
    v = ctypes.c_int(0)
    rc = _lib.moe_get_timeout_site(_stream(stream), ctypes.byref(v))
    return rc, v.value


def moe_last_cuda_error():
    return _lib.moe_last_cuda_error()


def moe_kernel_launches():
    return _lib.moe_kernel_launches()
