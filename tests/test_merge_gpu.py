"""LSE merge kernel against the float64 oracle."""
import numpy as np
import pytest
import torch

import exact_attention_sm_gb300 as ea
from exact_attention_sm_gb300 import inputs
from oracle import attention as orc
from tests.gpu_util import to_np

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("S", [1, 3, 24, 64, 200])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("empty", [0.0, 0.3])
def test_merge_matches_oracle(S, d, empty):
    o_p, l_p = inputs.merge_inputs(300, S, d, seed=S * 1000 + d, empty_frac=empty)
    o_ref, l_ref = orc.merge_states_batched(o_p.numpy(), l_p.numpy())
    o32, l32 = ea.attn_merge_states(o_p.cuda(), l_p.cuda(), out_dtype=torch.float32)
    ob, lb = ea.attn_merge_states(o_p.cuda(), l_p.cuda(), out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    got, lse = to_np(o32), to_np(l32)
    assert np.isfinite(got).all()
    assert np.abs(got - o_ref).max() < 1e-5
    fin = np.isfinite(l_ref)
    assert (np.isneginf(lse) == ~fin).all()
    assert np.abs(lse[fin] - l_ref[fin]).max() < 1e-5
    # bf16 output: within half a bf16 ulp of the fp32 result plus fp32 rounding
    gb = to_np(ob)
    assert (np.abs(gb - o_ref) <= np.abs(o_ref) * 2.0 ** -8 + 1e-5).all()
    if empty > 0:
        assert (got[0] == 0).all() and np.isneginf(lse[0])


def test_merge_is_deterministic():
    o_p, l_p = inputs.merge_inputs(512, 37, 128, seed=1, empty_frac=0.1)
    o_p, l_p = o_p.cuda(), l_p.cuda()
    outs = [ea.attn_merge_states(o_p, l_p, out_dtype=torch.float32) for _ in range(3)]
    torch.cuda.synchronize()
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])


@pytest.mark.parametrize("S", [5, 24, 100])
def test_empty_states_are_not_read_by_value(S):
    """An empty state (LSE = -inf) may hold anything in O, NaN included: it
    gets weight 0 and its O never reaches the sum."""
    o_p, l_p = inputs.merge_inputs(64, S, 128, seed=S, empty_frac=0.4)
    o_ref, l_ref = orc.merge_states_batched(o_p.numpy(), l_p.numpy())
    o_bad = o_p.clone()
    o_bad[torch.isneginf(l_p)] = float("nan")
    o32, l32 = ea.attn_merge_states(o_bad.cuda(), l_p.cuda(), out_dtype=torch.float32)
    torch.cuda.synchronize()
    got = to_np(o32)
    assert np.isfinite(got).all()
    assert np.abs(got - o_ref).max() < 1e-5
