"""Load-balanced fixed-grid decode (Lecture 4 section 5.6) against the oracle."""
import math

import numpy as np
import pytest
import torch

import exact_attention_sm_gb300 as ea
from exact_attention_sm_gb300 import inputs
from oracle import attention as orc
from tests.gpu_util import check_lse, check_o, to_np

pytestmark = pytest.mark.gpu


def make(lens, Hq, Hkv, seed=0, extra_cols=0):
    q, kp, vp, table, sl = inputs.decode_inputs(lens, Hq, Hkv, 128, seed=seed,
                                                extra_table_cols=extra_cols)
    return q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), sl.cuda(), (q, kp, vp, table, sl)


def oracle(host, lens):
    q, kp, vp, table, _ = host
    return orc.decode_paged(q.float().numpy(), kp.float().numpy(), vp.float().numpy(),
                            table.numpy(), lens, 1 / math.sqrt(128))


def run(lens, Hq, Hkv, num_ctas=0, seed=0):
    q, kp, vp, table, sl, host = make(lens, Hq, Hkv, seed)
    ws = torch.empty(ea.lib().attn_decode_sched_workspace_bytes(len(lens), Hq, Hkv, 128, num_ctas),
                     dtype=torch.uint8, device="cuda")
    ea.attn_decode_schedule(lens, Hq, Hkv, ws, num_ctas=num_ctas)
    o, lse = ea.attn_decode_paged_balanced(q, kp, vp, table, sl, ws, num_ctas=num_ctas)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == "ATTN_OK"
    o_ref, lse_ref = oracle(host, lens)
    check_o(to_np(o), o_ref, "bf16")
    check_lse(to_np(lse), lse_ref, "bf16")
    return (q, kp, vp, table, sl, ws), (o, lse)


@pytest.mark.parametrize("num_ctas", [0, 7, 64])
def test_long_tail_lengths(num_ctas):
    """A long-tailed batch with empty and one-token requests; 7 CTAs put many
    segments (of several requests) through each CTA's ring."""
    run([58125, 1, 0, 300, 4096, 17, 9000, 128], 32, 8, num_ctas, seed=1)


def test_config5_lengths():
    run(inputs.decode_lengths_uniform(4, 4096, 131072, seed=2), 32, 8, seed=2)


@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (6, 3), (8, 8), (16, 1)])
def test_head_groups(Hq, Hkv):
    """Groups of 1 to 16 query heads per KV head (several CTA head groups,
    padded groups)."""
    run([700, 33, 1500], Hq, Hkv, 12, seed=3)


def test_deterministic():
    args, (o, lse) = run([3000, 5000, 10], 32, 8, 20, seed=4)
    q, kp, vp, table, sl, ws = args
    for _ in range(2):
        o2, lse2 = ea.attn_decode_paged_balanced(q, kp, vp, table, sl, ws, num_ctas=20)
        torch.cuda.synchronize()
        assert torch.equal(o, o2) and torch.equal(lse, lse2)


def test_one_graph_replays_new_plans():
    """Capture the fixed-grid call once; for each new step, write new lengths
    into the same device tensor and a new plan into the same workspace, and
    replay the graph: the results follow the new lengths."""
    B, Hq, Hkv = 4, 32, 8
    steps = [[4000, 100, 0, 2500], [300, 8000, 16, 1], [7999, 7999, 7999, 7999]]
    longest = max(max(s) for s in steps)
    pages_needed = sum(-(-longest // 16) for _ in range(B))
    q, kp, vp, table, sl, host = make([longest] * B, Hq, Hkv, seed=5)
    assert kp.shape[0] == pages_needed
    ws = torch.empty(ea.lib().attn_decode_sched_workspace_bytes(B, Hq, Hkv, 128, 0),
                     dtype=torch.uint8, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
    ea.attn_decode_schedule(steps[0], Hq, Hkv, ws)
    sl.copy_(torch.tensor(steps[0], dtype=torch.int32))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        ea.attn_decode_paged_balanced(q, kp, vp, table, sl, ws, out=o, lse=lse)
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ea.attn_decode_paged_balanced(q, kp, vp, table, sl, ws, out=o, lse=lse)
    for lens in steps:
        sl.copy_(torch.tensor(lens, dtype=torch.int32))
        ea.attn_decode_schedule(lens, Hq, Hkv, ws)
        g.replay()
        torch.cuda.synchronize()
        assert ea.attn_get_device_status() == "ATTN_OK"
        o_ref, lse_ref = oracle(host, lens)
        check_o(to_np(o), o_ref, "bf16")
        check_lse(to_np(lse), lse_ref, "bf16")


def test_damaged_plan_is_reported_not_followed():
    """Random integers in place of a plan: every entry is checked on the
    device, the bad ones are reported and skipped; nothing faults."""
    q, kp, vp, table, sl, _ = make([500, 60], 8, 2, seed=6)
    nbytes = ea.lib().attn_decode_sched_workspace_bytes(2, 8, 2, 128, 9)
    ws = torch.randint(-1 << 20, 1 << 20, (nbytes // 4,), dtype=torch.int32,
                       generator=torch.Generator().manual_seed(7)).cuda().view(torch.uint8)
    ea.attn_decode_paged_balanced(q, kp, vp, table, sl, ws, num_ctas=9)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == "ATTN_ERR_BAD_INDEX"
