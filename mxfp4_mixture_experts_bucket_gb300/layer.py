"""A routed MXFP4 MoE layer object: device weights + workspace around moe_ffn_layer.

Marshalling only: every step of the layer runs in libmoe_mxfp4.so. PyTorch
provides device memory and the stream.
"""

from __future__ import annotations

from typing import Dict, Optional

import torch

from . import _lib

_WEIGHT_KEYS = ("w_router", "b_router", "g_qs", "g_sc", "u_qs", "u_sc", "d_qs", "d_sc",
                "bg", "bu", "bd", "gu_qs", "gu_sc", "gu_b")


class MoeLayer:
    """Holds one layer's weights on a CUDA device and runs it through the C ABI.

    weights: dict with w_router [E, D] f32, b_router [E] f32 (optional),
    g_qs/u_qs [E, F, D/2] u8, g_sc/u_sc [E, F, D/32] u8, d_qs [E, D, F/2] u8,
    d_sc [E, D, F/32] u8, bg/bu [E, F] f32, bd [E, D] f32 (biases optional).
    Gate and up may instead come as gpt-oss stores them, one interleaved plane
    per expert: gu_qs [E, 2F, D/2], gu_sc [E, 2F, D/32], gu_b [E, 2F] (gate row
    f = row 2f, up row f = row 2f+1); the layer then runs moe_ffn_layer_gu.
    Host (numpy or torch CPU) arrays are copied to `device` once.
    """

    def __init__(self, weights: Dict[str, object], k: int, device="cuda", packed: bool = False,
                 keep_canonical: bool = True):
        self.device = torch.device(device)
        self.w: Dict[str, Optional[torch.Tensor]] = {}
        for key in _WEIGHT_KEYS:
            v = weights.get(key)
            if v is None:
                self.w[key] = None
                continue
            t = v if isinstance(v, torch.Tensor) else torch.from_numpy(v)
            self.w[key] = t.to(self.device).contiguous()
        self.E, self.D = self.w["w_router"].shape
        self.interleaved = self.w["gu_qs"] is not None
        if self.interleaved and self.w["g_qs"] is not None:
            raise ValueError("give gate/up either as g_*/u_* planes or as one interleaved gu_* plane")
        self.F = self.w["gu_qs"].shape[1] // 2 if self.interleaved else self.w["g_qs"].shape[1]
        self.k = k
        self._ws: Dict[int, torch.Tensor] = {}
        self._io: Dict[tuple, tuple] = {}
        self.packed = None
        if packed:
            self._prepack()
            if not keep_canonical:
                for key in ("g_qs", "g_sc", "u_qs", "u_sc", "d_qs", "d_sc", "gu_qs", "gu_sc"):
                    self.w[key] = None

    def _prepack(self):
        """Prepacked copies of the three expert stacks (moe_mxfp4_prepack) and the layer struct."""
        pk: Dict[str, torch.Tensor] = {}
        for m, (R, C) in (("g", (self.F, self.D)), ("u", (self.F, self.D)), ("d", (self.D, self.F))):
            nq = _lib.moe_mxfp4_packed_qs_bytes(self.E, R, C)
            ns = _lib.moe_mxfp4_packed_sf_bytes(self.E, R, C)
            if nq == 0 or ns == 0:
                raise _lib.MoeError(f"shape ({self.E}, {R}, {C}) cannot be prepacked")
            pk[m + "_qs"] = torch.empty(nq, dtype=torch.uint8, device=self.device)
            pk[m + "_sf"] = torch.empty(ns, dtype=torch.uint8, device=self.device)
            if m == "d" or not self.interleaved:
                _lib.check(_lib.moe_mxfp4_prepack(self.w[m + "_qs"], self.w[m + "_sc"], self.E, R, C, pk[m + "_qs"],
                                                  pk[m + "_sf"]), "moe_mxfp4_prepack")
        if self.interleaved:
            _lib.check(_lib.moe_mxfp4_prepack_gu(self.w["gu_qs"], self.w["gu_sc"], self.E, self.F, self.D,
                                                 pk["g_qs"], pk["g_sf"], pk["u_qs"], pk["u_sf"]),
                       "moe_mxfp4_prepack_gu")
        self.packed = pk
        w = self.w
        bg, bu = w["bg"], w["bu"]
        if self.interleaved and w["gu_b"] is not None:  # the packed layer struct takes separate bias rows
            gb = w["gu_b"].view(self.E, self.F, 2)
            self._bias_split = (gb[:, :, 0].contiguous(), gb[:, :, 1].contiguous())
            bg, bu = self._bias_split
        self.packed_struct = _lib.make_packed_layer(self.D, self.F, self.E, self.k, w["w_router"], w["b_router"],
                                                    pk["g_qs"], pk["g_sf"], bg, pk["u_qs"], pk["u_sf"],
                                                    bu, pk["d_qs"], pk["d_sf"], w["bd"])

    def _use_packed(self, T: int, rail: int) -> bool:
        # MOE_RAIL_AUTO with both sets of planes takes the rail measured fastest on
        # GB300 at each T: the CUDA-core GEMV rail (canonical) at T = 1, the
        # prepacked planes beyond (the library's choice there: the block-scaled
        # decode rail for T <= MOE_AUTO_DECODE_MX_MAX_T, the kind::mxf4 grouped
        # rail after it). Without the canonical planes the prepacked planes serve
        # every T.
        if self.packed is None:
            return False
        if rail in (_lib.MOE_RAIL_DECODE_MX, _lib.MOE_RAIL_GROUPED_MX4):
            return True
        if rail != _lib.MOE_RAIL_AUTO:
            return False
        return (self.w["g_qs"] is None and self.w["gu_qs"] is None) or T >= 2

    def workspace(self, T: int, rail: int) -> torch.Tensor:
        if self._use_packed(T, rail):
            n = _lib.moe_ffn_packed_workspace_bytes(T, self.D, self.F, self.E, self.k, rail)
        else:
            n = _lib.moe_ffn_workspace_bytes(T, self.D, self.F, self.E, self.k, rail)
        if n == 0 and T > 0:
            raise _lib.MoeError("invalid shape for the layer's workspace")
        key = (n, rail, self._use_packed(T, rail))
        buf = self._ws.get(key)
        if buf is None:
            buf = torch.empty(max(n, 256), dtype=torch.uint8, device=self.device)
            self._ws[key] = buf
        return buf

    def forward(self, x: torch.Tensor, rail: int = _lib.MOE_RAIL_AUTO, out: Optional[torch.Tensor] = None,
                ids_out: Optional[torch.Tensor] = None, weights_out: Optional[torch.Tensor] = None,
                stream=None, h_out: Optional[torch.Tensor] = None) -> torch.Tensor:
        T = x.shape[0]
        if out is None:
            out = torch.empty((T, self.D), dtype=torch.float32, device=self.device)
        ws = self.workspace(T, rail)
        if self._use_packed(T, rail):
            rc = _lib.moe_ffn_layer_packed(self.packed_struct, x, T, rail, ws, ws.numel(), out, ids_out,
                                           weights_out, h_out, stream)
            _lib.check(rc, "moe_ffn_layer_packed")
            return out
        w = self.w
        if self.interleaved:
            rc = _lib.moe_ffn_layer_gu(x, T, self.D, self.F, self.E, self.k, w["w_router"], w["b_router"],
                                       w["gu_qs"], w["gu_sc"], w["gu_b"], w["d_qs"], w["d_sc"], w["bd"], rail, ws,
                                       ws.numel(), out, ids_out, weights_out, stream)
            _lib.check(rc, "moe_ffn_layer_gu")
            return out
        rc = _lib.moe_ffn_layer(x, T, self.D, self.F, self.E, self.k, w["w_router"], w["b_router"],
                                w["g_qs"], w["g_sc"], w["bg"], w["u_qs"], w["u_sc"], w["bu"],
                                w["d_qs"], w["d_sc"], w["bd"], rail, ws, ws.numel(), out, ids_out,
                                weights_out, stream)
        _lib.check(rc, "moe_ffn_layer")
        return out

    def forward_host(self, x_host: torch.Tensor, y_host: Optional[torch.Tensor] = None,
                     rail: int = _lib.MOE_RAIL_AUTO, stream=None) -> torch.Tensor:
        """The layer for tokens in host memory, one C call per step (moe_ffn_layer_hostio).

        x_host: [T, D] float32 CPU tensor, ideally pinned; y_host (allocated pinned
        if None): [T, D] float32 CPU tensor. The copies and the layer are only
        enqueued on the stream: synchronise it before reading y_host.
        """
        if x_host.dim() != 2 or x_host.shape[1] != self.D:
            raise ValueError(f"x_host must be [T, {self.D}]")
        T = x_host.shape[0]
        if x_host.is_cuda or x_host.dtype is not torch.float32 or not x_host.is_contiguous():
            raise ValueError("x_host must be a contiguous float32 CPU tensor")
        if y_host is None:
            y_host = torch.empty((T, self.D), dtype=torch.float32, pin_memory=True)
        elif (y_host.is_cuda or y_host.dtype is not torch.float32 or not y_host.is_contiguous()
              or y_host.shape != x_host.shape):
            raise ValueError(f"y_host must be a contiguous float32 CPU tensor of shape [{T}, {self.D}]")
        sp = _lib._stream(stream)
        io = self._io.get((T, rail))
        if io is not None:  # staging buffers and the C arguments of this (T, rail) exist already
            rc = _lib.moe_ffn_layer_hostio_ref(io[2], x_host.data_ptr(), y_host.data_ptr(), sp)
            if rc:
                _lib.check(rc, "moe_ffn_layer_hostio")
            return y_host
        if self._use_packed(T, rail):
            ws = self.workspace(T, rail)
            rc = _lib.moe_ffn_layer_packed_hostio(self.packed_struct, T, rail, ws, ws.numel(), x_host, y_host,
                                                  sp)
            _lib.check(rc, "moe_ffn_layer_packed_hostio")
            return y_host
        if self.interleaved:
            raise NotImplementedError("host I/O runs on separate gate/up planes or the prepacked rail")
        # staging buffers and the fixed arguments, once per (T, rail)
        xd = torch.empty((T, self.D), dtype=torch.float32, device=self.device)
        yd = torch.empty((T, self.D), dtype=torch.float32, device=self.device)
        ws = self.workspace(T, rail)
        w = self.w
        args = _lib.make_ffn_args(T, self.D, self.F, self.E, self.k, rail, w["w_router"], w["b_router"],
                                  w["g_qs"], w["g_sc"], w["bg"], w["u_qs"], w["u_sc"], w["bu"],
                                  w["d_qs"], w["d_sc"], w["bd"], ws, ws.numel(), xd, yd)
        io = (xd, yd, _lib.byref_args(args), args)
        self._io[(T, rail)] = io
        rc = _lib.moe_ffn_layer_hostio_ref(io[2], x_host.data_ptr(), y_host.data_ptr(), sp)
        _lib.check(rc, "moe_ffn_layer_hostio")
        return y_host

    __call__ = forward
