"""Shared helpers for the GPU parity tests (CUDA path vs the CPU oracle)."""

import numpy as np
import torch

from oracle import moe_oracle as O

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None

DECODE_TOL = 1e-4   # fp32 decode rail, row-normwise
PREFILL_TOL = 2e-2  # bf16-MMA prefill rail vs the float64 layer, row-normwise (1e-3 floor)
PREFILL_BF16_TOL = 5e-3  # prefill rail vs the oracle evaluated with the same bf16 operands
PREFILL_MX_TOL = 1e-3    # block-scaled rail vs the oracle evaluated with the same E4M3-term operands


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a)) if not isinstance(a, torch.Tensor) else a
    if dtype is not None:
        t = t.to(dtype)
    return t.to(DEV)


def empty(shape, dtype):
    return torch.empty(shape, dtype=dtype, device=DEV)


def status(moe):
    rc, st = moe.moe_get_status()
    assert rc == 0, rc
    if st & moe.MOE_STATUS_WAIT_TIMEOUT:
        _, site = moe.moe_get_timeout_site()
        print(f"timeout site 0x{site:08x}: kernel {site >> 24} role {(site >> 20) & 15} "
              f"stage {(site >> 12) & 255} seq {site & 4095}")
    return st


def bf16_bits_to_f64(t: torch.Tensor) -> np.ndarray:
    """A torch uint16/int16/bfloat16 tensor holding bf16 bit patterns -> float64 values."""
    u = t.view(torch.int16).cpu().numpy().view(np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def routing_check(logits_gpu, ids_gpu, w_gpu, logits_ref, k):
    """Routing parity (bit-exact ids where the oracle has a clear margin).

    Tokens whose top-(k+1) logits are closer than 1e-4 * max|l| may legitimately
    differ between fp32 and fp64 logits; for those the GPU's ids must equal the
    oracle's top-k evaluated on the GPU's own logits. Weights are checked
    against the softmax of the float64 logits over the GPU's ids.
    """
    lg = np.asarray(logits_gpu, np.float64)
    ids = np.asarray(ids_gpu)
    scale = max(np.abs(logits_ref).max(), 1e-30)
    assert np.max(np.abs(lg - logits_ref)) <= 1e-5 * scale + 1e-6
    ids_ref, _ = O.topk_softmax(logits_ref, k)
    margin = O.routing_margins(logits_ref, k)
    clear = margin > 1e-4 * scale
    assert np.array_equal(ids[clear], ids_ref[clear])
    if (~clear).any():
        ids_own, _ = O.topk_softmax(lg[~clear], k)
        assert np.array_equal(ids[~clear], ids_own)
    sel = np.take_along_axis(logits_ref, ids.astype(np.int64), axis=1)
    ex = np.exp(sel - sel[:, :1])
    w_ref = ex / ex.sum(axis=1, keepdims=True)
    assert np.max(np.abs(np.asarray(w_gpu, np.float64) - w_ref)) <= 1e-5
    return int((~clear).sum())
