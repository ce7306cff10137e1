"""Child process of tests/test_gpu_checked.py: runs the layer through every rail
on the checked build (MOE_MXFP4_CHECKED=1 in its environment, so the binding
loads libmoe_mxfp4_checked.so) and checks the results and the status word.
Not collected by pytest (no test_ prefix); exits non-zero on a mismatch."""

import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import mxfp4_mixture_experts_bucket_gb300 as moe  # noqa: E402
from oracle import moe_oracle as O  # noqa: E402
from synthetic import make_layer, make_tokens, spec_for  # noqa: E402


def reference(L, x_np, k, ids, token_idx, cache):
    """The float64 layer under the GPU's routing (weights: softmax of the float64
    logits over those ids), so that a near-tie cannot fail the comparison."""
    lg = O.router_logits(x_np, L["w_router"], L.get("b_router"))
    sel = np.take_along_axis(lg, ids.astype(np.int64), axis=1)
    w = np.exp(sel - sel.max(axis=1, keepdims=True))
    w /= w.sum(axis=1, keepdims=True)
    y, _, _, _ = O.moe_layer(L, x_np, k, token_idx=token_idx, ids=ids, weights=w, cache=cache)
    return y, lg


def main():
    assert os.environ.get("MOE_MXFP4_CHECKED") == "1"
    assert moe.moe_checked_build() == 1, "the checked library was not loaded"
    dev = torch.device("cuda:0")
    # (config, T, sampled tokens or None for all): a tiny layer and the gpt-oss-shaped one
    cases = [(0, 8, None), (0, 1, None), (1, 1, None), (1, 24, [0, 23])]
    for cfg, T, toks in cases:
        spec = spec_for(cfg)
        L = make_layer(spec)
        cache = O.ExpertCache(L)
        x_np = make_tokens(spec, T=T, seed=700 + 10 * cfg + T)
        token_idx = np.arange(T) if toks is None else np.asarray(toks)
        x = torch.from_numpy(x_np).to(dev)
        canon = moe.MoeLayer(L, k=spec.k, device=dev)
        packed = moe.MoeLayer(L, k=spec.k, device=dev, packed=True, keep_canonical=False)
        rails = [(canon, moe.MOE_RAIL_GROUPED_MM, 2e-2), (canon, moe.MOE_RAIL_GROUPED_MX, 2e-2),
                 (packed, moe.MOE_RAIL_GROUPED_MX4, 2e-2)]
        if T <= 8:
            rails += [(canon, moe.MOE_RAIL_GEMV, 1e-4), (packed, moe.MOE_RAIL_DECODE_MX, 1e-4)]
        for layer, rail, tol in rails:
            ids = torch.empty((T, spec.k), dtype=torch.int32, device=dev)
            y = layer(x, rail=rail, ids_out=ids)
            torch.cuda.synchronize()
            rc, st = moe.moe_get_status()
            assert rc == 0 and st == 0, f"config {cfg} T={T} rail {rail}: status {st:#x}"
            ids_np = ids.cpu().numpy()
            y_ref, lg = reference(L, x_np, spec.k, ids_np, token_idx, cache)
            err = O.rownorm_rel_err(y.cpu().numpy()[token_idx], y_ref).max()
            assert err <= tol, f"config {cfg} T={T} rail {rail}: error {err:.3e} > {tol}"
            ids_ref, _ = O.topk_softmax(lg, spec.k)
            clear = O.routing_margins(lg, spec.k) > 1e-4 * max(np.abs(lg).max(), 1e-30)
            assert np.array_equal(ids_np[clear], ids_ref[clear]), f"config {cfg} T={T} rail {rail}: routing"
        del canon, packed
        torch.cuda.empty_cache()
    print("checked build ok")


if __name__ == "__main__":
    main()
