"""Seeded synthetic workloads for the gpt-oss-shaped MXFP4 MoE layer.

Storage layout (the library's own, fixed here so both sides agree on it):

* An MXFP4 matrix W[R, C] is two planes.
  - ``qs``: uint8 [R, C/2]. Block b of row r covers columns 32b..32b+31 and
    occupies bytes 16b..16b+15 of the row. Byte i of the block holds column
    32b+i in its low nibble and column 32b+16+i in its high nibble.
  - ``sc``: uint8 [R, C/32], one E8M0 exponent byte per block.
* Expert matrices are stacked: gate and up are [E, F, D] (qs [E, F, D/2]),
  down is [E, D, F] (qs [E, D, F/2]).
* Biases are float32: bg, bu [E, F]; bd [E, D]. Router: w_router [E, D]
  float32, b_router [E] float32.

Value distributions follow the workload descriptions of the gpt-oss-20b
shaped MoE layer (E=32 experts, top-4, dim = nfe = 2880): activations
N(0, 1), router N(0, 0.1), nibbles uniform over the 16 codes (so bytes are
uniform), exponent bytes uniform in a closed range, biases N(0, 0.02).
Nothing here computes any part of the layer.
"""

from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Dict, Optional

import numpy as np


@dataclass(frozen=True)
class LayerSpec:
    name: str
    E: int
    k: int
    D: int
    F: int
    T: int
    s_lo: int  # inclusive lower bound of the E8M0 exponent byte
    s_hi: int  # inclusive upper bound
    router: str = "normal"  # "normal" | "equal_norm" | "skew"
    seed: int = 1000
    layers: int = 1


# The five workloads (tiny oracle case, decode, prefill, 24-layer stack, skew).
CONFIGS: Dict[int, LayerSpec] = {
    0: LayerSpec("tiny", E=4, k=2, D=64, F=64, T=8, s_lo=120, s_hi=130, seed=1000),
    1: LayerSpec("decode_T1", E=32, k=4, D=2880, F=2880, T=1, s_lo=110, s_hi=135, seed=1001),
    2: LayerSpec("prefill_T512", E=32, k=4, D=2880, F=2880, T=512, s_lo=110, s_hi=135,
                 router="equal_norm", seed=1002),
    3: LayerSpec("stack24", E=32, k=4, D=2880, F=2880, T=1, s_lo=110, s_hi=135, seed=1003,
                 layers=24),
    4: LayerSpec("skew_T4096", E=32, k=4, D=2880, F=2880, T=4096, s_lo=110, s_hi=135,
                 router="skew", seed=1004),
}


def spec_for(cfg: int, **overrides) -> LayerSpec:
    spec = CONFIGS[cfg]
    return replace(spec, **overrides) if overrides else spec


def _mx_planes(rng: np.random.Generator, E: int, R: int, C: int, s_lo: int, s_hi: int):
    qs = rng.integers(0, 256, size=(E, R, C // 2), dtype=np.uint8)
    sc = rng.integers(s_lo, s_hi + 1, size=(E, R, C // 32), dtype=np.uint8)
    return qs, sc


def _router(rng: np.random.Generator, spec: LayerSpec):
    E, D = spec.E, spec.D
    wr = (rng.standard_normal((E, D), dtype=np.float32) * np.float32(0.1)).astype(np.float32)
    br = np.zeros((E,), dtype=np.float32)
    if spec.router == "equal_norm":
        # Every row rescaled to the same norm 0.1*sqrt(D): near-uniform load.
        norms = np.sqrt((wr.astype(np.float64) ** 2).sum(axis=1, keepdims=True))
        wr = (wr.astype(np.float64) / norms * (0.1 * np.sqrt(D))).astype(np.float32)
    elif spec.router == "skew":
        # Row norm 1 (logit sigma ~ 1 for N(0,1) tokens); +4 on two hot experts,
        # -2 on the last four so that several experts stay (nearly) empty.
        norms = np.sqrt((wr.astype(np.float64) ** 2).sum(axis=1, keepdims=True))
        wr = (wr.astype(np.float64) / norms).astype(np.float32)
        br[0] = 4.0
        br[1] = 4.0
        br[E - 4:] = -2.0
    elif spec.router != "normal":
        raise ValueError(spec.router)
    return wr, br


def make_tokens(spec: LayerSpec, T: Optional[int] = None, seed: Optional[int] = None) -> np.ndarray:
    """Fresh N(0,1) float32 activations [T, D]."""
    rng = np.random.default_rng(spec.seed + 7919 if seed is None else seed)
    T = spec.T if T is None else T
    return rng.standard_normal((T, spec.D), dtype=np.float32)


def make_layer(spec: LayerSpec, layer: int = 0, with_tokens: bool = True) -> Dict[str, np.ndarray]:
    """One layer's weights (and tokens) as host numpy arrays, seeded by spec.seed and layer."""
    rng = np.random.default_rng([spec.seed, layer])
    E, D, F = spec.E, spec.D, spec.F
    wr, br = _router(rng, spec)
    g_qs, g_sc = _mx_planes(rng, E, F, D, spec.s_lo, spec.s_hi)
    u_qs, u_sc = _mx_planes(rng, E, F, D, spec.s_lo, spec.s_hi)
    d_qs, d_sc = _mx_planes(rng, E, D, F, spec.s_lo, spec.s_hi)
    bg = (rng.standard_normal((E, F), dtype=np.float32) * np.float32(0.02)).astype(np.float32)
    bu = (rng.standard_normal((E, F), dtype=np.float32) * np.float32(0.02)).astype(np.float32)
    bd = (rng.standard_normal((E, D), dtype=np.float32) * np.float32(0.02)).astype(np.float32)
    out = dict(w_router=wr, b_router=br, g_qs=g_qs, g_sc=g_sc, u_qs=u_qs, u_sc=u_sc,
               d_qs=d_qs, d_sc=d_sc, bg=bg, bu=bu, bd=bd)
    if with_tokens:
        out["x"] = make_tokens(spec)
    return out


def make_layer_torch(spec: LayerSpec, layer: int, device, with_tokens: bool = False):
    """The same recipe drawn with torch's generator directly on `device`.

    Used where a host draw would be too large (multi-layer stacks of several
    GB). Values differ from :func:`make_layer` (another generator) but follow
    the same distributions; callers that need the oracle copy the touched
    experts back to the host.
    """
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(spec.seed * 1000 + layer)
    E, D, F = spec.E, spec.D, spec.F

    def planes(R, C):
        qs = torch.randint(0, 256, (E, R, C // 2), generator=g, device=device, dtype=torch.uint8)
        sc = torch.randint(spec.s_lo, spec.s_hi + 1, (E, R, C // 32), generator=g, device=device,
                           dtype=torch.uint8)
        return qs, sc

    wr = torch.randn((E, D), generator=g, device=device, dtype=torch.float32) * 0.1
    br = torch.zeros((E,), device=device, dtype=torch.float32)
    if spec.router == "equal_norm":
        wr = wr / wr.double().norm(dim=1, keepdim=True).float() * float(0.1 * np.sqrt(D))
    elif spec.router == "skew":
        wr = wr / wr.double().norm(dim=1, keepdim=True).float()
        br[0] = 4.0
        br[1] = 4.0
        br[E - 4:] = -2.0
    g_qs, g_sc = planes(F, D)
    u_qs, u_sc = planes(F, D)
    d_qs, d_sc = planes(D, F)
    bg = torch.randn((E, F), generator=g, device=device) * 0.02
    bu = torch.randn((E, F), generator=g, device=device) * 0.02
    bd = torch.randn((E, D), generator=g, device=device) * 0.02
    out = dict(w_router=wr.contiguous(), b_router=br, g_qs=g_qs, g_sc=g_sc, u_qs=u_qs, u_sc=u_sc,
               d_qs=d_qs, d_sc=d_sc, bg=bg, bu=bu, bd=bd)
    if with_tokens:
        out["x"] = torch.randn((spec.T, D), generator=g, device=device, dtype=torch.float32)
    return out


def interleave_gate_up(layer: Dict[str, object]) -> Dict[str, object]:
    """The same layer with gate and up stored as gpt-oss stores them: one plane
    per expert of 2F rows, gate row f at row 2f and up row f at row 2f+1
    (gu_qs [E, 2F, D/2], gu_sc [E, 2F, D/32], gu_b [E, 2F]). A storage layout
    only: numpy arrays stay numpy, torch tensors stay on their device."""
    out = {k: v for k, v in layer.items() if k not in ("g_qs", "g_sc", "u_qs", "u_sc", "bg", "bu")}

    def inter(a, b):
        if isinstance(a, np.ndarray):
            E, F = a.shape[:2]
            return np.stack([a, b], axis=2).reshape((E, 2 * F) + a.shape[2:])
        import torch
        E, F = a.shape[:2]
        return torch.stack([a, b], dim=2).reshape((E, 2 * F) + tuple(a.shape[2:])).contiguous()

    out["gu_qs"] = inter(layer["g_qs"], layer["u_qs"])
    out["gu_sc"] = inter(layer["g_sc"], layer["u_sc"])
    if layer.get("bg") is not None and layer.get("bu") is not None:
        out["gu_b"] = inter(layer["bg"], layer["bu"])
    return out
