"""GPU parity: sage_splitk_combine against the oracle's LSE combine."""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close, f32, np_

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("S", [1, 5, 40])
def test_combine_random_partials(sage, D, S):
    g = torch.Generator().manual_seed(D * 100 + S)
    R = 37
    o = torch.randn((R, S, D), generator=g)
    lse = torch.randn((R, S), generator=g) * 3
    if S > 1:
        lse[::3, 0] = -float("inf")        # empty segments are skipped
    lse[5, :] = -float("inf")              # a row with no keys at all
    o[5] = 0
    oc, lc = o.cuda(), lse.cuda()
    out, lout = sage.sage_splitk_combine(oc, lc, out_dtype=torch.float16, return_lse=True)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.splitk_combine(o.numpy(), lse.numpy())
    assert_close(f32(out), o_ref)
    assert_close(np_(lout), l_ref, "lse", rel=1e-6, abs_=1e-5)
    assert np.all(f32(out)[5] == 0) and np.isneginf(np_(lout)[5])


def test_combine_bf16_batched_shape(sage):
    # attention-sized outputs (|o| ~ 0.05) keep bf16 output rounding inside tolerance
    o = torch.randn((2, 3, 4, 128), generator=torch.Generator().manual_seed(1)) * 0.05
    lse = torch.randn((2, 3, 4), generator=torch.Generator().manual_seed(2))
    out = sage.sage_splitk_combine(o.cuda(), lse.cuda(), out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    o_ref, _ = oracle.splitk_combine(o.numpy(), lse.numpy())
    assert out.shape == (2, 3, 128)
    assert_close(f32(out), o_ref)
