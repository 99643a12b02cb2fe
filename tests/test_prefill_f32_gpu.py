"""fp32 prefill (CUDA cores) against the float64 oracle."""
import math

import pytest
import torch

import exact_attention_sm_gb300 as ea
from exact_attention_sm_gb300 import inputs
from oracle import attention as orc
from tests.gpu_util import check_lse, check_o, to_np

pytestmark = pytest.mark.gpu


def run_case(B, Hq, Hkv, Lq, Lk, d, causal, seed=0):
    q, k, v = inputs.prefill_inputs(B, Hq, Hkv, Lq, Lk, d, "f32", seed)
    scale = 1.0 / math.sqrt(d)
    o, lse = ea.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    torch.cuda.synchronize()
    o_ref, lse_ref = orc.prefill(q.numpy(), k.numpy(), v.numpy(), scale, causal)
    check_o(to_np(o), o_ref, "f32")
    check_lse(to_np(lse), lse_ref, "f32")


@pytest.mark.parametrize("causal", [False, True])
def test_single_head_L256_d64(causal):
    """B=1, H=1, L=256, d=64, fp32 N(0,1) from seed 0, scale 1/8."""
    run_case(1, 1, 1, 256, 256, 64, causal)


@pytest.mark.parametrize("L", [1, 17, 63, 65, 200, 257])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_lengths(L, causal):
    run_case(2, 4, 2, L, L, 64, causal, seed=L)


def test_rectangular_and_d128():
    run_case(1, 8, 2, 37, 301, 128, False, seed=5)
    run_case(1, 2, 1, 130, 130, 128, True, seed=6)
