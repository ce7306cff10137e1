"""The allocation-free decode entry point (moe_ffn_layer_decode_static).

It exists for callers that cannot allocate device memory where they run the
layer (allocation-free serving loops, plugins handed only a stream and
tensors); its scratch is a static device array inside the library.
This file is collected last so that a failure here leaves every other test
already run.
"""

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from synthetic import make_layer, make_tokens, spec_for
from tests.gpu_helpers import DECODE_TOL, dev, empty, status

FAKE = 1 << 20


def _call(moe, layer, x, y, ids, w):
    W = layer.w
    return moe.moe_ffn_layer_decode_static(x, x.shape[0], layer.D, layer.F, layer.E, layer.k, W["w_router"],
                                           W["b_router"], W["g_qs"], W["g_sc"], W["bg"], W["u_qs"], W["u_sc"],
                                           W["bu"], W["d_qs"], W["d_sc"], W["bd"], y, ids, w)


@pytest.mark.gpu
def test_static_scratch_matches_workspace_entry_point_on_consecutive_calls(moe):
    spec = spec_for(1)
    layer = moe.MoeLayer(make_layer(spec, with_tokens=False), k=spec.k)
    # two calls in a row; the second (larger) one reuses what the first left in the scratch
    for call, T in enumerate((1, 8)):
        x = dev(make_tokens(spec, T=T, seed=900 + call))
        ids_ref = empty((T, spec.k), torch.int32)
        w_ref = empty((T, spec.k), torch.float32)
        y_ref = layer(x, rail=moe.MOE_RAIL_GEMV, ids_out=ids_ref, weights_out=w_ref)
        y = torch.full((T, spec.D), float("nan"), device="cuda")
        ids = empty((T, spec.k), torch.int32)
        w = empty((T, spec.k), torch.float32)
        assert _call(moe, layer, x, y, ids, w) == moe.MOE_OK
        torch.cuda.synchronize()
        assert status(moe) == 0
        assert torch.equal(ids, ids_ref) and torch.equal(w, w_ref)
        err = O.rownorm_rel_err(y.cpu().numpy(), y_ref.cpu().numpy()).max()
        assert err <= DECODE_TOL, err


def test_static_scratch_rejects_shapes_beyond_its_size(moe):
    # T = 8, k = 8, F = 4096 needs 8*8*4096*4 B of h alone (1 MiB) > the 512 KiB array:
    # rejected on the host before anything is enqueued.
    rc = moe.moe_ffn_layer_decode_static(FAKE, 8, 64, 4096, 8, 8, *([FAKE] * 11), FAKE, None, None, stream=0)
    assert rc == moe.MOE_ESCRATCH
    assert moe.moe_ffn_workspace_bytes(8, 64, 4096, 8, 8, moe.MOE_RAIL_GEMV) > moe.MOE_DECODE_SCRATCH_BYTES
    # beyond the GEMV rail's token limit
    rc = moe.moe_ffn_layer_decode_static(FAKE, 9, 64, 64, 4, 2, *([FAKE] * 11), FAKE, None, None, stream=0)
    assert rc == moe.MOE_EINVAL
    # the gpt-oss width with eight tokens of eight experts: h alone is 8*8*2880*4 B > 512 KiB
    assert moe.moe_ffn_workspace_bytes(8, 2880, 2880, 32, 8, moe.MOE_RAIL_GEMV) > moe.MOE_DECODE_SCRATCH_BYTES
    rc = moe.moe_ffn_layer_decode_static(FAKE, 8, 2880, 2880, 32, 8, *([FAKE] * 11), FAKE, None, None, stream=0)
    assert rc == moe.MOE_ESCRATCH


def test_static_scratch_zero_tokens_is_a_no_op(moe):
    n0 = moe.moe_kernel_launches()
    rc = moe.moe_ffn_layer_decode_static(FAKE, 0, 2880, 2880, 32, 4, *([FAKE] * 11), FAKE, None, None, stream=0)
    assert rc == moe.MOE_OK
    assert moe.moe_kernel_launches() == n0
