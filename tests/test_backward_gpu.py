"""Backward pass (dQ, dK, dV) on the GPU against the float64 oracle.

Tolerance for bf16 gradients, from the arithmetic: the kernels round P and dS
to bf16 (relative 2^-9 each) before the tensor-core products, take D from the
bf16 O, and rebuild P from the forward's fp32 LSE (itself within 1e-2 of the
exact value in the worst row, far less typically).  Each gradient element is
a sum of such products, so its error is a small fraction of the gradient's
own scale: max |err| <= 2e-2 * max |ref| and sum |err| <= 1e-2 * sum |ref|
per tensor.
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_sm_gb300 as ea
from exact_attention_sm_gb300 import inputs
from oracle import attention as orc
from tests.gpu_util import to_np

pytestmark = pytest.mark.gpu

MAX_REL, SUM_REL = 2e-2, 1e-2


def check_grad(got, want, name):
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    assert got.shape == want.shape, name
    assert np.isfinite(got).all(), f"{name}: non-finite"
    err = np.abs(got - want)
    scale = max(np.abs(want).max(), 1e-3)  # an all-zero gradient (one key) has no scale of its own
    total = max(np.abs(want).sum(), 1e-3 * want.size)
    # The measured margins, printed beside the bounds (pytest -s or -rP shows them).
    print(f"{name}: max|err|/scale {err.max() / scale:.2e} (bound {MAX_REL:.0e}), "
          f"sum|err|/sum|ref| {err.sum() / total:.2e} (bound {SUM_REL:.0e})")
    assert err.max() <= MAX_REL * scale, f"{name}: max {err.max():.3e} vs scale {scale:.3e}"
    assert err.sum() <= SUM_REL * total, f"{name}: sum-rel {err.sum() / total:.3e}"


def run(B, Hq, Hkv, Lq, Lk, d, causal, seed=0):
    q, k, v = inputs.prefill_inputs(B, Hq, Hkv, Lq, Lk, d, "bf16", seed=seed)
    g = torch.Generator().manual_seed(seed + 1)
    do = torch.randn(B, Hq, Lq, d, generator=g).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(d)
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = ea.attn_fwd(qc, kc, vc, causal=causal, scale=scale)
    dq, dk, dv = ea.attn_bwd(qc, kc, vc, o, lse, doc, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == "ATTN_OK"
    rq, rk, rv = orc.backward(q.float().numpy(), k.float().numpy(), v.float().numpy(),
                              do.float().numpy(), scale, causal)
    check_grad(to_np(dq), rq, "dQ")
    check_grad(to_np(dk), rk, "dK")
    check_grad(to_np(dv), rv, "dV")
    return (qc, kc, vc, o, lse, doc), (dq, dk, dv)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_gqa(d, causal):
    """Three Q/K tiles with a ragged tail, two query heads per KV head."""
    run(2, 4, 2, 300, 300, d, causal, seed=1)


@pytest.mark.parametrize("d", [64, 128])
def test_exact_tile_and_single_row(d):
    run(1, 2, 2, 128, 128, d, True, seed=2)
    run(1, 2, 1, 1, 1, d, True, seed=3)


@pytest.mark.parametrize("d", [64, 128])
def test_cross_lengths_non_causal(d):
    run(2, 2, 1, 200, 333, d, False, seed=4)


def test_longer_sequence_mha():
    run(1, 4, 1, 1024, 1024, 128, True, seed=5)


def test_deterministic():
    args, (dq, dk, dv) = run(1, 4, 2, 257, 257, 64, True, seed=6)
    for _ in range(2):
        dq2, dk2, dv2 = ea.attn_bwd(*args, causal=True)
        torch.cuda.synchronize()
        assert torch.equal(dq, dq2) and torch.equal(dk, dk2) and torch.equal(dv, dv2)


@pytest.mark.parametrize("d", [64, 128])
def test_more_items_than_ctas_ragged(d):
    """288 K/V tiles and 288 Q tiles (2 x 16 heads x 9 tiles, the last 76 rows
    long): more work items than persistent CTAs, so CTAs take several items,
    some of them ragged, through the item ring and the staged stores."""
    run(2, 16, 16, 1100, 1100, d, True, seed=8)


@pytest.mark.parametrize("d", [64, 128])
def test_workspace_reused_across_calls(d):
    """One workspace for several calls: the work counters in it are reset by
    every call (the persistent CTAs claim all items again), results equal."""
    args, (dq, dk, dv) = run(2, 4, 2, 300, 300, d, True, seed=7)
    B, Hq, Lq = args[0].shape[0], args[0].shape[1], args[0].shape[2]
    ws = torch.empty(ea.lib().attn_bwd_workspace_bytes(B, Hq, Lq), dtype=torch.uint8, device="cuda")
    for _ in range(3):
        dq2, dk2, dv2 = ea.attn_bwd(*args, causal=True, scale=1.0 / math.sqrt(d), workspace=ws)
        torch.cuda.synchronize()
        assert ea.attn_get_device_status() == "ATTN_OK"
        assert torch.equal(dq, dq2) and torch.equal(dk, dk2) and torch.equal(dv, dv2)


def run_sampled_groups(B, Hq, Hkv, L, d, groups, seed):
    """Full-size causal backward on the GPU; the oracle checks the sampled
    (batch, KV head) groups: dQ of every query head of the group, and the
    group's dK, dV (summed over its query heads, as the GQA rule says)."""
    q, k, v = inputs.prefill_inputs(B, Hq, Hkv, L, L, d, "bf16", seed=seed)
    g = torch.Generator().manual_seed(seed + 1)
    do = torch.randn(B, Hq, L, d, generator=g).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(d)
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = ea.attn_fwd(qc, kc, vc, causal=True, scale=scale)
    dq, dk, dv = ea.attn_bwd(qc, kc, vc, o, lse, doc, causal=True, scale=scale)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == "ATTN_OK"
    per = Hq // Hkv
    f = lambda t: t.float().numpy()
    for b, kh in groups:
        rk = np.zeros((L, d))
        rv = np.zeros((L, d))
        for h in range(kh * per, (kh + 1) * per):
            gq, gk, gv, _ = orc.attention_backward(f(q[b, h]), f(k[b, kh]), f(v[b, kh]), f(do[b, h]),
                                                   scale, True)
            check_grad(to_np(dq[b, h]), gq, f"dQ[{b},{h}]")
            rk += gk
            rv += gv
        check_grad(to_np(dk[b, kh]), rk, f"dK[{b},{kh}]")
        check_grad(to_np(dv[b, kh]), rv, f"dV[{b},{kh}]")


def test_gpt2_medium_shape_sampled_heads():
    """The benchmarked GPT-2-medium shape (B 64, H 16, L 1024, d 64, causal):
    three (batch, head) pairs from randperm(B * H, seed 3)."""
    B, H = 64, 16
    pick = torch.randperm(B * H, generator=torch.Generator().manual_seed(3))[:3].tolist()
    run_sampled_groups(B, H, H, 1024, 64, [(i // H, i % H) for i in pick], seed=0)


def test_llama3_8k_shape_sampled_group():
    """The benchmarked Llama-3-8B shape (Hq 32, Hkv 8, L 8192, d 128, causal):
    one KV head from randperm(Hkv, seed 3) with its four query heads."""
    kh = int(torch.randperm(8, generator=torch.Generator().manual_seed(3))[0])
    run_sampled_groups(1, 32, 8, 8192, 128, [(0, kh)], seed=0)
