"""Cascade (shared-prefix) decode against the float64 oracle."""
import math

import numpy as np
import pytest
import torch

import exact_attention_sm_gb300 as ea
from exact_attention_sm_gb300 import inputs
from oracle import attention as orc
from tests.gpu_util import check_lse, check_o, to_np

pytestmark = pytest.mark.gpu


def run_cascade(prefix_len, suffix_lens, Hq=32, Hkv=8, num_splits=0, seed=0, d=128):
    q, pk, pv, kp, vp, table, sl = inputs.cascade_inputs(prefix_len, suffix_lens, Hq, Hkv, d,
                                                         seed=seed)
    scale = 1.0 / math.sqrt(d)
    o, lse = ea.attn_decode_cascade(q.cuda(), pk.cuda(), pv.cuda(), kp.cuda(), vp.cuda(),
                                    table.cuda(), sl.cuda(), seq_lens_host=suffix_lens,
                                    num_splits=num_splits, scale=scale)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == "ATTN_OK"
    f = lambda t: t.float().numpy()
    o_ref, lse_ref = orc.decode_cascade(f(q), f(pk), f(pv), f(kp), f(vp), table.numpy(),
                                        suffix_lens, scale)
    check_o(to_np(o), o_ref, "bf16")
    check_lse(to_np(lse), lse_ref, "bf16")
    return o, lse


@pytest.mark.parametrize("splits", [0, 1])
@pytest.mark.parametrize("prefix_len", [1, 100, 128, 300, 1000])
def test_small_prefixes_and_ragged_suffixes(prefix_len, splits):
    """Prefixes below, at and past one 128-key tile (ragged chunks), suffixes
    of 0 (prefix only), 1, 17 and 200 tokens; one suffix state per row, and
    the planned splits (several per row for these short batches)."""
    run_cascade(prefix_len, [0, 1, 17, 200], num_splits=splits, seed=prefix_len)


@pytest.mark.parametrize("splits", [1, 3])
def test_forced_suffix_splits(splits):
    run_cascade(512, [5, 700, 64], num_splits=splits, seed=5)


@pytest.mark.parametrize("splits", [0, 1])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (12, 4), (64, 8)])
def test_group_sizes(hq, hkv, splits):
    run_cascade(256, [33, 0, 129], Hq=hq, Hkv=hkv, num_splits=splits, seed=7)


def test_lecture_demo_shape_B64_prefix4096_suffix256():
    """[Lecture 4] 4.4 demo 4: prefix 4096 shared by 64 requests, 256 unique
    tokens each (Hq 32, Hkv 8, d 128), checked in full."""
    run_cascade(4096, [256] * 64, seed=0)


def test_equals_plain_decode_over_whole_sequence():
    """The same requests through attn_decode_paged over prefix + suffix pages
    agree with the cascade within bf16 rounding (both are the same function)."""
    P, lens, Hq, Hkv = 320, [40, 0, 97], 16, 4
    q, pk, pv, kp, vp, table, sl = inputs.cascade_inputs(P, lens, Hq, Hkv, 128, seed=3)
    o_c, lse_c = ea.attn_decode_cascade(q.cuda(), pk.cuda(), pv.cuda(), kp.cuda(), vp.cuda(),
                                        table.cuda(), sl.cuda(), seq_lens_host=lens)
    # Whole sequences in a fresh paged cache: prefix tokens then suffix tokens.
    full = [P + n for n in lens]
    pages = [-(-n // 16) for n in full]
    kp2 = torch.zeros(sum(pages), 16, Hkv, 128, dtype=torch.bfloat16)
    vp2 = torch.zeros_like(kp2)
    tab2 = torch.full((len(lens), max(pages)), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(lens):
        kk = torch.cat([pk.permute(1, 0, 2), orc_gather(kp, table[b], n)], dim=0)
        vv = torch.cat([pv.permute(1, 0, 2), orc_gather(vp, table[b], n)], dim=0)
        for i in range(pages[b]):
            tab2[b, i] = off
            seg = slice(i * 16, min((i + 1) * 16, full[b]))
            kp2[off, : seg.stop - seg.start] = kk[seg]
            vp2[off, : seg.stop - seg.start] = vv[seg]
            off += 1
    o_p, lse_p = ea.attn_decode_paged(q.cuda(), kp2.cuda(), vp2.cuda(), tab2.cuda(),
                                      torch.tensor(full, dtype=torch.int32).cuda(),
                                      seq_lens_host=full)
    torch.cuda.synchronize()
    assert (o_c.float() - o_p.float()).abs().max().item() < 2e-2
    assert (lse_c - lse_p).abs().max().item() < 1e-2


def orc_gather(pages, table_row, n):
    """Logical-order rows of a paged tensor (torch, for building test inputs)."""
    t = torch.arange(n)
    return pages[table_row[t // 16].long(), t % 16]


@pytest.mark.parametrize("splits", [0, 1])
def test_cascade_is_deterministic(splits):
    q, pk, pv, kp, vp, table, sl = inputs.cascade_inputs(2048, [300, 5, 0, 1200], 32, 8, 128,
                                                         seed=9)
    args = [t.cuda() for t in (q, pk, pv, kp, vp, table, sl)]
    outs = [ea.attn_decode_cascade(*args, seq_lens_host=[300, 5, 0, 1200], num_splits=splits)
            for _ in range(3)]
    torch.cuda.synchronize()
    for o, lse in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(lse, outs[0][1])


@pytest.mark.parametrize("splits", [0, 1])
def test_graph_replay_with_new_queries(splits):
    """The cascade captured once in a CUDA graph (its side stream forks from
    the capturing stream and joins back before the merge pass) and replayed
    with new query values in the same buffer: every replay matches the oracle."""
    P, lens, Hq, Hkv = 1000, [256] * 20 + [3, 0, 77], 32, 8
    q, pk, pv, kp, vp, table, sl = inputs.cascade_inputs(P, lens, Hq, Hkv, 128, seed=11)
    scale = 1.0 / math.sqrt(128)
    qc = q.cuda()
    dev = [t.cuda() for t in (pk, pv, kp, vp, table, sl)]
    o = torch.empty_like(qc)
    lse = torch.empty(len(lens), Hq, dtype=torch.float32, device="cuda")
    pc, _, ss = ea.attn_cascade_plan(len(lens), Hq, Hkv, P, lens, 16, splits)
    ws = torch.empty(ea.attn_cascade_workspace_bytes(len(lens), Hq, 128, pc, ss), dtype=torch.uint8,
                     device="cuda")

    def call():
        ea.attn_decode_cascade(qc, *dev, seq_lens_host=lens, num_splits=splits, scale=scale, out=o,
                               lse=lse, workspace=ws)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    f = lambda t: t.float().numpy()
    for rep in range(3):
        qn = torch.randn(q.shape, generator=torch.Generator().manual_seed(100 + rep)).to(q.dtype)
        qc.copy_(qn)
        g.replay()
        torch.cuda.synchronize()
        assert ea.attn_get_device_status() == "ATTN_OK"
        o_ref, lse_ref = orc.decode_cascade(f(qn), f(pk), f(pv), f(kp), f(vp), table.numpy(), lens,
                                            scale)
        check_o(to_np(o), o_ref, "bf16")
        check_lse(to_np(lse), lse_ref, "bf16")


@pytest.mark.parametrize("splits", [0, 1])
@pytest.mark.parametrize("prefix_len,lens,Hq,Hkv", [(1, [0, 1, 17, 200], 32, 8),
                                                    (300, [5, 700, 64], 32, 8),
                                                    (1000, [33, 0, 129], 12, 4),
                                                    (4096, [256] * 16, 32, 8)])
def test_head_dim_64(prefix_len, lens, Hq, Hkv, splits):
    """d = 64: the prefix pass on the d = 64 prefill kernel, the suffixes on
    the d = 64 decode, the merge with two dims per lane."""
    run_cascade(prefix_len, lens, Hq=Hq, Hkv=Hkv, num_splits=splits, seed=prefix_len + 1, d=64)
