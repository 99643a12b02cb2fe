"""Paged GQA decode at head dim 64 (split-KV + LSE merge) against the float64
oracle: the same kernel as d = 128 with half the dims per lane and twice the
ring stages."""
import math

import pytest
import torch

import exact_attention_sm_gb300 as ea
from exact_attention_sm_gb300 import inputs
from oracle import attention as orc
from tests.gpu_util import check_lse, check_o, to_np

pytestmark = pytest.mark.gpu


def run_decode64(lens, Hq=16, Hkv=4, num_splits=0, seed=0, extra_cols=0, poison=False):
    q, kp, vp, table, sl = inputs.decode_inputs(lens, Hq, Hkv, 64, seed=seed, perm_seed=seed + 1,
                                                extra_table_cols=extra_cols)
    if poison:  # slots of each request's last page past its length hold NaN
        for b, n in enumerate(lens):
            if n % 16:
                last = int(table[b, -(-n // 16) - 1])
                kp[last, n % 16:] = float("nan")
                vp[last, n % 16:] = float("nan")
    scale = 1.0 / math.sqrt(64)
    o, lse = ea.attn_decode_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), sl.cuda(),
                                  seq_lens_host=lens, num_splits=num_splits, scale=scale)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == "ATTN_OK"
    o_ref, lse_ref = orc.decode_paged(q.float().numpy(), kp.float().numpy(), vp.float().numpy(),
                                      table.numpy(), lens, scale)
    check_o(to_np(o), o_ref, "bf16")
    check_lse(to_np(lse), lse_ref, "bf16")
    return o, lse


@pytest.mark.parametrize("splits", [0, 1, 2, 7])
def test_d64_partial_pages_and_splits(splits):
    """Lengths 1, 17, 1000, 4096 (partial last pages), forced and planned splits."""
    run_decode64([1, 17, 1000, 4096], num_splits=splits, extra_cols=3, poison=True)


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 4), (12, 4), (32, 8)])
def test_d64_group_sizes(hq, hkv):
    """Group sizes 1, 3, 4 (one CTA per KV head) and padded groups."""
    run_decode64([33, 700, 16, 129], Hq=hq, Hkv=hkv, seed=4)


def test_d64_empty_request():
    o, lse = run_decode64([0, 50, 0])
    assert (o[0] == 0).all() and torch.isneginf(lse[0]).all()


def test_d64_long_context_split_kv():
    """B = 4 long contexts (uniform in [4096, 65536], seed 2): the planner splits."""
    lens = inputs.decode_lengths_uniform(4, 4096, 65536, seed=2)
    run_decode64(lens, Hq=32, Hkv=8)
    _, smax = ea.attn_decode_plan(lens, 8, 16, 0)
    assert smax > 1


def test_d64_split_kv_is_deterministic():
    lens = [3000, 777, 1]
    q, kp, vp, table, sl = inputs.decode_inputs(lens, 16, 4, 64, seed=9, perm_seed=10)
    args = (q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), sl.cuda())
    a = ea.attn_decode_paged(*args, seq_lens_host=lens, num_splits=5)
    b = ea.attn_decode_paged(*args, seq_lens_host=lens, num_splits=5)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
