"""Paged GQA decode (split-KV + LSE merge) against the float64 oracle."""
import math

import numpy as np
import pytest
import torch

import exact_attention_sm_gb300 as ea
from exact_attention_sm_gb300 import inputs
from oracle import attention as orc
from tests.gpu_util import check_lse, check_o, to_np

pytestmark = pytest.mark.gpu


def run_decode(lens, Hq=32, Hkv=8, num_splits=0, seed=0, extra_cols=0):
    q, kp, vp, table, sl = inputs.decode_inputs(lens, Hq, Hkv, 128, seed=seed, perm_seed=seed + 1,
                                                extra_table_cols=extra_cols)
    scale = 1.0 / math.sqrt(128)
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
def test_handbook_lengths(splits):
    """Context lengths 1, 17, 1000, 4096 (partial pages), Hq 32, Hkv 8, d 128."""
    run_decode([1, 17, 1000, 4096], num_splits=splits, extra_cols=3)


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (64, 8), (12, 4)])
def test_group_sizes(hq, hkv):
    run_decode([33, 700, 16, 129], Hq=hq, Hkv=hkv, num_splits=0, seed=4)


def test_empty_request():
    o, lse = run_decode([0, 50, 0], num_splits=0)
    assert (o[0] == 0).all() and torch.isneginf(lse[0]).all()


def test_batched_decode_B256_ctx1024():
    """B=256 requests x 1024 tokens, Hq 32, Hkv 8, d 128, 16-token shuffled pages."""
    run_decode([1024] * 256, num_splits=0)


def test_long_context_split_kv_B4():
    """B=4, lengths uniform in [4096, 131072] from seed 2, planner's split count."""
    lens = inputs.decode_lengths_uniform(4, 4096, 131072, seed=2)
    o, lse = run_decode(lens, num_splits=0)
    chunk, smax = ea.attn_decode_plan(lens, 8, 16, 0)
    assert smax > 1


def test_split_kv_is_deterministic():
    lens = [70000, 5000, 123457, 4096]
    q, kp, vp, table, sl = inputs.decode_inputs(lens, 32, 8, 128, seed=9)
    args = [t.cuda() for t in (q, kp, vp, table, sl)]
    outs = [ea.attn_decode_paged(*args, seq_lens_host=lens) for _ in range(3)]
    torch.cuda.synchronize()
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])


def test_block_table_indexing_bit_exact():
    """One dominant key per (request, KV head) whose V row encodes its physical
    page and slot as small integers; the output must reproduce them exactly."""
    lens = [1, 17, 40, 300, 1000]
    Hq, Hkv, d, P = 16, 4, 128, 16
    q, kp, vp, table, sl = inputs.decode_inputs(lens, Hq, Hkv, d, seed=3)
    kp = torch.zeros_like(kp)
    num_pages = kp.shape[0]
    pages = torch.arange(num_pages).view(-1, 1, 1)
    slots = torch.arange(P).view(1, -1, 1)
    heads = torch.arange(Hkv).view(1, 1, -1)
    vp = torch.zeros_like(vp)
    vp[..., 0] = (pages % 256).expand(-1, P, Hkv).to(vp.dtype)
    vp[..., 1] = (pages // 256).expand(-1, P, Hkv).to(vp.dtype)
    vp[..., 2] = slots.expand(num_pages, -1, Hkv).to(vp.dtype)
    vp[..., 3] = heads.expand(num_pages, P, -1).to(vp.dtype)
    q = torch.zeros_like(q)
    q[..., 0] = 1.0
    targets = {}
    for b, n in enumerate(lens):
        for kh in range(Hkv):
            t = (b * 7 + kh * 13) % n
            page = int(table[b, t // P])
            kp[page, t % P, kh, 0] = 128.0   # score 128 against 0 for every other key
            targets[(b, kh)] = (page, t % P)
    o, _ = ea.attn_decode_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), sl.cuda(),
                                seq_lens_host=lens, scale=1.0)
    o = o.float().cpu()
    for (b, kh), (page, slot) in targets.items():
        for h in range(kh * (Hq // Hkv), (kh + 1) * (Hq // Hkv)):
            got = o[b, h, :4].tolist()
            assert got == [page % 256, page // 256, slot, kh], (b, h, got, page, slot)


def test_bad_table_entry_is_reported_not_dereferenced():
    lens = [40, 40]
    q, kp, vp, table, sl = inputs.decode_inputs(lens, 8, 2, 128, seed=1)
    table[1, 1] = kp.shape[0] + 5
    ea.attn_decode_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), sl.cuda(), seq_lens_host=lens,
                         num_splits=1)
    assert ea.attn_get_device_status() == "ATTN_ERR_BAD_INDEX"
    assert ea.attn_get_device_status() == "ATTN_OK"   # read clears it
