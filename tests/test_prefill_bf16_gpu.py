"""bf16 prefill (TMA + tcgen05 + TMEM kernel) against the float64 oracle."""
import math

import numpy as np
import pytest
import torch

import exact_attention_sm_gb300 as ea
from exact_attention_sm_gb300 import inputs
from oracle import attention as orc
from tests.gpu_util import check_lse, check_o, to_np

pytestmark = pytest.mark.gpu


def full_case(B, Hq, Hkv, Lq, Lk, d, causal, seed=0):
    q, k, v = inputs.prefill_inputs(B, Hq, Hkv, Lq, Lk, d, "bf16", seed)
    scale = 1.0 / math.sqrt(d)
    o, lse = ea.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == "ATTN_OK"
    o_ref, lse_ref = orc.prefill(q.float().numpy(), k.float().numpy(), v.float().numpy(), scale, causal)
    check_o(to_np(o), o_ref, "bf16")
    check_lse(to_np(lse), lse_ref, "bf16")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("L", [1, 17, 128, 129, 300, 640])
def test_small_shapes(d, causal, L):
    full_case(2, 4, 2, L, L, d, causal, seed=L + d)


@pytest.mark.parametrize("d", [64, 128])
def test_rectangular_non_causal(d):
    full_case(1, 4, 1, 200, 777, d, False, seed=1)
    full_case(1, 2, 2, 513, 64, d, False, seed=2)


def sampled_case(B, Hq, Hkv, L, d, causal):
    """Sampled rows against the oracle.  O and LSE start as NaN, so a work
    item that no CTA took would leave non-finite rows behind."""
    q, k, v = inputs.prefill_inputs(B, Hq, Hkv, L, L, d, "bf16", seed=0)
    scale = 1.0 / math.sqrt(d)
    o = torch.full((B, Hq, L, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, Hq, L), float("nan"), dtype=torch.float32, device="cuda")
    ea.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale, out=o, lse=lse)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == "ATTN_OK"
    rows = inputs.sample_rows(B, Hq, L)
    o_ref, lse_ref = orc.prefill_rows(q.float().numpy(), k.float().numpy(), v.float().numpy(),
                                      scale, causal, rows)
    idx = torch.tensor(rows)
    got_o = o[idx[:, 0], idx[:, 1], idx[:, 2]]
    got_l = lse[idx[:, 0], idx[:, 1], idx[:, 2]]
    check_o(to_np(got_o), o_ref, "bf16")
    check_lse(to_np(got_l), lse_ref, "bf16")
    # properties that hold for every row
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    return o, lse


def test_gpt2_medium_shape_B64_H16_L1024_d64_causal():
    sampled_case(64, 16, 16, 1024, 64, True)


def test_long_causal_rows_dealt_in_reversed_odd_rounds():
    """17 pair positions x 32 heads = 544 items on the persistent grid: the
    smallest d = 128 causal rows dealt from the per-CTA item list, with odd
    rounds in reverse CTA order."""
    sampled_case(1, 32, 8, 4352, 128, True)


def test_llama3_8b_shape_L8192_gqa_causal():
    sampled_case(1, 32, 8, 8192, 128, True)


def test_llama3_8b_shape_L32768_gqa_causal():
    sampled_case(1, 32, 8, 32768, 128, True)


def test_prefill_is_deterministic():
    q, k, v = (t.cuda() for t in inputs.prefill_inputs(2, 8, 2, 1000, 1000, 128, "bf16", seed=4))
    outs = [ea.attn_fwd(q, k, v, causal=True) for _ in range(3)]
    torch.cuda.synchronize()
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])


def test_lse_optional():
    q, k, v = (t.cuda() for t in inputs.prefill_inputs(1, 2, 2, 256, 256, 64, "bf16", seed=5))
    o1, _ = ea.attn_fwd(q, k, v, causal=True, want_lse=False)
    o2, _ = ea.attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_row_max_is_exact(d, causal):
    """Scores of about 200 (natural-log units) where key j matches query row
    i (j = i mod d) and 0 elsewhere: the matching columns fall in every
    32-column chunk of a 128-key tile as i runs.  Softmax is only safe if the
    tile's row max is the true maximum: a maximum that missed one chunk
    would leave exp2 arguments near +290, which overflow to inf and turn O
    into NaN.  Covers the maximum taken from the S load (unmasked tiles), the
    masked-tile maximum (diagonal and tail tiles) and rescales by 2^-290."""
    B, H, L = 1, 2, 300
    a = 40.0  # q and k entries, exact in bf16: score a * a * scale
    q = torch.zeros(B, H, L, d)
    k = torch.zeros(B, H, L, d)
    idx = torch.arange(L)
    q[:, :, idx, idx % d] = a
    k[:, :, idx, idx % d] = a
    v = torch.randn(B, H, L, d, generator=torch.Generator().manual_seed(12))
    q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
    scale = 1.0 / math.sqrt(d)
    o, lse = ea.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == "ATTN_OK"
    o_ref, lse_ref = orc.prefill(q.float().numpy(), k.float().numpy(), v.float().numpy(), scale,
                                 causal)
    check_o(to_np(o), o_ref, "bf16")
    check_lse(to_np(lse), lse_ref, "bf16")
